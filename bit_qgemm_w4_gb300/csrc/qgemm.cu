// The stack engine of the verify GEMM (selected with spec_set_gemm_engine;
// the default split engine is in qgemm_split.cu): low-bit weights times the
// T drafted positions' activations, on the sm_103a tensor cores.
//
// What it computes ("Karpathy's Trick for Faster Local LLMs Finally Has Proper
// Tooling", section "How Uzu optimizes bytes and tokens per pass": 4-bit
// asymmetric Medium tier, 8-bit symmetric Large tier, one scale per group,
// optional random Hadamard rotation of the activations):
//   y[t][n] = sum_k x'[t][k] * (code[n][k] - zero[g][n]) * scale[g][n]   (int4)
//   y[t][n] = sum_k x'[t][k] *  code[n][k]              * scale         (int8)
// x' = x, or its block rotation (1/sqrt(B)) H_B (s .* x) per block of B k.
//
// One persistent launch runs one GEMM or a whole stack of them (a verify
// pass: every projection of every layer, in order).  The pass "streams every
// weight ... once" ("Why batch-one decoding is memory-bound"), so the design
// keeps the weight stream running across GEMM boundaries:
//  * every GEMM's (128-row tile, k-stage) units are divided evenly over the
//    grid (one CTA per SM); each CTA walks its share of GEMM 0, then of GEMM
//    1, and so on;
//  * a weight-producer warp issues, per stage, one TMA copy of the 128 rows'
//    128-byte code lines plus the stage's scale and zero rows into a ring of
//    shared-memory slots, and keeps the stream further ahead with L2
//    prefetches of the boxes it will load next;
//  * an activation-producer warp loads each stage's activation boxes
//    (128-byte swizzle, the MMA's B operand) into a second ring; before the
//    first load of a GEMM that depends on its predecessors it waits until
//    those have written every output tile (device-side counters); when the
//    MMA reads the activations in another form (fp16 for int4, or rotated)
//    every CTA first writes its share of that form into a scratch copy (the
//    rotation with the warp-shuffle fast Walsh-Hadamard transform) and the
//    loads read the copy once all shares are in;
//  * eight worker warps (two per TMEM lane quadrant, one weight row per
//    thread) dequantise each stage straight into a TMEM ring that is the
//    MMA's A operand: for int4 the group scale is folded in, (code - zero) *
//    scale rounded once to fp16 (11 significant bits), so one fp32
//    accumulator serves a whole tile and nothing is read back per stage;
//    int8 codes with one scale per output channel enter exactly (bf16) and
//    the scale multiplies the fp32 sums;
//  * MMA warps (one per 64-k group for int4) issue the K16 MMAs
//    (tcgen05.mma kind::f16, M = 128 weight rows, N = T padded to 16), all
//    adding into one fp32 accumulator of the tile (the tensor pipe applies
//    the MMAs one at a time, so their order does not matter); the
//    accumulator is double buffered between a CTA's tile segments, and the
//    workers zero it after reading it;
//  * at the end of a segment the workers write a whole tile directly, or add
//    a tile shared with other CTAs into an fp32 slot with red.global.add,
//    the last contributor to arrive finishing it.
// Every wait is bounded; a timeout records an error, raises a grid-wide
// abort flag, drains the CTA's in-flight copies and MMAs and frees its
// tensor memory before returning.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>
#include <cstring>

#include "fwht.cuh"
#include "internal.hpp"
#include "ptx.cuh"

namespace sv {
namespace {

constexpr int kTmemCols = 512;

// flags of a stage's control record (bits above the GEMM index)
constexpr uint32_t kStageSegEnd = 1u << 16;   // the CTA's segment of the tile ends here
constexpr uint32_t kStageWhole = 1u << 17;    // ... and it covered the whole tile
constexpr uint32_t kStageLast = 1u << 18;     // the CTA's last stage of the launch
constexpr uint32_t kStageFrom0 = 1u << 19;    // (at a segment end) the segment began at the tile's first k
constexpr uint32_t kStageFinStart = 1u << 20; // first stage of a segment that finishes a split tile
constexpr int kStageConvShift = 21;           // (activation records) the GEMM's xconv mode, 2 bits

template <int QUANT, int TPAD>
struct Cfg {
  static constexpr int kSub = QUANT == kW4 ? 4 : 2;             // 64-k groups per stage
  static constexpr int kStageKK = kGroupK * kSub;               // k per stage (128 code bytes per row)
  static constexpr int kWorkersPerQ = kGemmWorkers / 4;         // workers per TMEM lane quadrant
  static constexpr int kGpw = kSub / kWorkersPerQ;              // 64-k groups a worker dequantises
  static constexpr int kCols = TPAD / kWorkersPerQ;             // accumulator columns a worker reads
  // MMA warps: one per group for int4 up to T = 32 (a thread issues one
  // tcgen05.mma every ~50-75 cycles), else two; each owns an accumulator
  static constexpr int kMmaW = (QUANT == kW4 && TPAD <= 32) ? 4 : 2;
  static constexpr int kGpm = kSub / kMmaW;                     // groups per MMA warp
  // weight slot: codes [128 rows][128 B] (128-byte swizzle) | scales [<=kSub][128] fp16 | zeros [<=kSub][64]
  static constexpr int kScaleOff = kTileM * 128;
  static constexpr int kZeroOff = kScaleOff + kSub * kTileM * 2;
  static constexpr int kWSlot = (kZeroOff + (QUANT == kW4 ? kSub * 64 : 0) + 1023) / 1024 * 1024;
  // the stage's control record (written by the weight producer): the GEMM
  // index with the kStage* flags, then the tile
  static constexpr int kCtlOff = kWSlot - 16;
  static_assert(kCtlOff >= kZeroOff + (QUANT == kW4 ? kSub * 64 : 0), "control record inside the slot padding");
  // activation slot: kSub boxes [TPAD][64] 16-bit (128-byte rows, 128-byte swizzle)
  static constexpr int kXBox = TPAD * 128;
  static constexpr int kXSlot = kSub * kXBox;
  static constexpr int kXSlots = kXSlot > 16384 ? 2 : 4;
  static constexpr int kCtrl = 1024;
  static constexpr int kSmemBudget = 225 * 1024;
  // the split-tile sum a CTA finishes, fetched early into shared memory
  // ([128 rows][TPAD] fp32) where a worker reads at most 16 columns
  static constexpr int kPreBytes = TPAD / 2 <= 16 ? kTileM * TPAD * 4 : 0;
  static constexpr int kWSlotsFit = (kSmemBudget - 1024 - kCtrl - kXSlots * kXSlot - kPreBytes) / kWSlot;
  static constexpr int kWSlots = kWSlotsFit > 12 ? 12 : kWSlotsFit;
  static constexpr int kSmemBytes = 1024 + kXSlots * kXSlot + kWSlots * kWSlot + kPreBytes + kCtrl;
  // TMEM: two accumulators of TPAD columns (a CTA's consecutive tile
  // segments alternate between them; every MMA warp adds into the current
  // one), then from column 128 a ring of A slots (one stage each, 32 columns
  // per group)
  static constexpr int kDCols = TPAD;
  static constexpr int kACols = 32 * kSub;
  static constexpr int kA0 = 128;
  static constexpr int kNAFit = (kTmemCols - kA0) / kACols;
  static constexpr int kNA = kNAFit > 4 ? 4 : kNAFit;
  // warps: weight producer, activation producer, the TMEM owner, a spare
  // warp, the MMA warps, then the workers (any eight consecutive warps cover
  // each TMEM lane quadrant twice).  Four warps, one per scheduler, convert
  // activation slots in shared memory where a GEMM asks for it: the MMA
  // warps, and with two MMA warps also warps 2 and 3.
  static constexpr int kWProd = 0, kXProd = 1, kAlloc = 2, kMma0 = 4;
  static constexpr int kConvW = 4;
  static constexpr int kConv0 = kMmaW == 4 ? kMma0 : 2;          // first converting warp
  static constexpr int kWorker0 = kMma0 + kMmaW;
  static constexpr int kThreads = 32 * (kWorker0 + kGemmWorkers);
  // one CTA per SM: the register file split evenly over its threads (a
  // launch reserves registers for whole groups of four warps)
  static constexpr int kRegThreads = (kThreads + 127) / 128 * 128;
  static constexpr int kMaxRegs = (65536 / kRegThreads) / 8 * 8 > 232 ? 232 : (65536 / kRegThreads) / 8 * 8;
  static_assert(kXBox % 1024 == 0, "activation boxes must keep the 1024-byte swizzle period");
  static_assert(kWSlots >= 4, "weight ring too shallow");
  static_assert(kNA >= 2 && 2 * kDCols <= kA0 && kA0 + kNA * kACols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kCols % 8 == 0, "epilogue columns in multiples of 8");
  static constexpr int kDM = 4;                                 // ring of per-stage "MMAs done" barriers
  static_assert(kNA <= kDM && kXSlots <= kDM, "a slot is reused within the done ring");
  static_assert((2 * kWSlots + 3 * kXSlots + kNA + kDM + 4 + kGemmWorkers) * 8 + 8 <= kCtrl, "barrier block");
};

struct Params {
  const GemmEntry* entries;   // stack: device array; null: the entry passed by value
  int n_entries;
  int gate;                   // stack launch: count finished tiles, honour wait_prev
  int prep_flags;             // kAnyPrep: some entry prepares its activations with every CTA
                              // (the rotation counters are in use); kAnyConv: some entry
                              // converts its activation slots in shared memory
  int slot_ctas;              // CTAs per key in the split-tile slot arrays
  float* partials;            // [kSplitKeys][slot_ctas][128][TPAD] fp32, kept zeroed
  int* split_cnt;             // [kSplitKeys][slot_ctas][kGemmWorkers], kept zeroed
  int* done;                  // [n_entries] finished (tile, worker) parts
  int* rot_done;              // [n_entries] CTAs whose rotation share is written
  int* exit_cnt;
  int* err;
  int* abort_all;
  unsigned long long wait_ns;
  int skip_unit;              // test hook: CTA 0 never loads the weights of this unit (-1: none)
  int pf_dist;                // L2 prefetch lead (units) while the ring has room
  int pf_max;                 // lead allowed while the ring is full
};

// Abort state shared by a CTA's waits.
struct Ctl {
  volatile int* abort_cta;
  int* abort_all;
  int* err;
  unsigned long long limit;
  __device__ __forceinline__ bool aborted() const {
    if (*abort_cta) return true;
    if (*reinterpret_cast<volatile int*>(abort_all)) {
      *abort_cta = 1;
      return true;
    }
    return false;
  }
  __device__ __forceinline__ void raise() const {
    *abort_cta = 1;
    atomicCAS(err, 0, kDevErrTimeout);
    atomicExch(abort_all, 1);
  }
};

// Wait for a barrier phase; false on abort or when the limit passes.  A
// phase that is not complete at the first probe is waited for with the
// suspending form of try_wait: the thread sleeps in hardware until the phase
// completes or kSuspendNs passes, so it neither takes issue slots from the
// warps doing the work nor oversleeps the flip; the abort flags and the clock
// are looked at on every eighth probe.
constexpr uint32_t kSuspendNs = 10000;

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
    if ((i & 7u) == 0) {
      if (c.aborted()) return false;
      if (globaltimer() - t0 > c.limit) {
        c.raise();
        return false;
      }
    }
  }
}

// The same for a whole warp: every lane waits, and the outcome is uniform.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Ctl& c) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, c));
}

// Wait until a device counter reaches `target` (acquire); false on abort or
// when the limit passes.
__device__ __forceinline__ bool wait_count(const int* p, int target, const Ctl& c) {
  if (ld_acquire_gpu(p) >= target) return true;
  const unsigned long long t0 = globaltimer();
  unsigned ns = 16;
  while (true) {
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
    if (ld_acquire_gpu(p) >= target) return true;
    if (c.aborted()) return false;
    if (globaltimer() - t0 > c.limit) {
      c.raise();
      return false;
    }
  }
}

// Drain wait: ignores the abort flags, gives up after kDrainLimitNs.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, 100000u))
    if (globaltimer() - t0 > kDrainLimitNs) return;
}

// A GEMM of U units is spread over Ge = min(G, U) CTAs, CTA c < Ge owning
// units [c*U/Ge, (c+1)*U/Ge) (never empty); CTAs c >= Ge own none.  So the
// CTAs that share a tile are consecutive and each holds part of it.
__device__ __forceinline__ int spread(int total, int G) { return total < G ? total : G; }

// floor(a * b / d) for 0 <= a, b, d < 2^31; 32-bit arithmetic when the
// product fits (a 64-bit division is a long instruction sequence).
__device__ __forceinline__ int muldiv(int a, int b, int d) {
  const unsigned long long prod = (unsigned long long)a * (unsigned)b;
  if (prod <= 0xFFFFFFFFull) return (int)((uint32_t)prod / (uint32_t)d);
  return (int)(prod / (unsigned)d);
}

__device__ __forceinline__ int unit_begin(int c, int total, int G) {
  const int Ge = spread(total, G);
  return c >= Ge ? total : muldiv(c, total, Ge);
}

__device__ __forceinline__ int cta_of_unit(int u, int total, int G) {
  const int Ge = spread(total, G);
  int c = muldiv(u, Ge, total);
  while (c + 1 < Ge && unit_begin(c + 1, total, G) <= u) ++c;
  while (c > 0 && unit_begin(c, total, G) > u) --c;
  return c;
}

// Position in a ring of N slots with the parity of the current lap.
template <int N>
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == N) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Walks a CTA's units across the entries of a launch: for each entry the CTA
// owns units [c*U/G, (c+1)*U/G) of its U = tiles * ks (tile-major).
struct Walk {
  const GemmEntry* E;
  int nE, G, c;
  int e = 0, u = 0, ub = 0, ue = 0, tile = 0, kst = 0, ks = 1;
  __device__ __forceinline__ Walk(const GemmEntry* E_, int nE_, int G_, int c_)
      : E(E_), nE(nE_), G(G_), c(c_) {
    enter(0);
  }
  __device__ __forceinline__ void enter(int e0) {
    for (e = e0; e < nE; ++e) {
      const int U = E[e].units;
      ub = unit_begin(c, U, G);
      ue = unit_begin(c + 1, U, G);
      if (ub < ue) {
        u = ub;
        ks = E[e].ks;
        tile = u / ks;
        kst = u - tile * ks;
        return;
      }
    }
  }
  __device__ __forceinline__ bool valid() const { return e < nE; }
  __device__ __forceinline__ void next() {
    if (++u == ue) {
      enter(e + 1);
      return;
    }
    if (++kst == ks) {
      kst = 0;
      ++tile;
    }
  }
};

// The last GEMM of the launch in which CTA c owns a stage, or -1.
__device__ __forceinline__ int last_entry_of(const GemmEntry* E, int nE, int G, int c) {
  int e = nE - 1;
  while (e >= 0 && unit_begin(c + 1, E[e].units, G) <= unit_begin(c, E[e].units, G)) --e;
  return e;
}


// int4: the 64 codes of group j of a row's 128-byte stage line.  The line was
// written by TMA with the 128-byte swizzle: 16-byte chunk c of row m sits at
// chunk position c ^ (m & 7).
__device__ __forceinline__ void load_w4(uint32_t row_addr, uint32_t m, int j, uint32_t (&words)[8]) {
  const uint32_t sw = m & 7u;
  const uint4 c0 = lds128(row_addr + (((2u * j) ^ sw) << 4));
  const uint4 c1 = lds128(row_addr + (((2u * j + 1u) ^ sw) << 4));
  words[0] = c0.x; words[1] = c0.y; words[2] = c0.z; words[3] = c0.w;
  words[4] = c1.x; words[5] = c1.y; words[6] = c1.z; words[7] = c1.w;
}

// int4 weights of one 64-k group as fp16 pairs with the group scale folded
// in: a[i] holds k = 2i (low half) and 2i+1 (high half).  Code layout: nibble
// p (0..7, from the least significant end) of each little-endian 32-bit word
// holds k = 8w + 2*(p % 4) + p / 4, so the pairs (k0, k1), (k2, k3), (k4, k5),
// (k6, k7) sit at bits 0, 4, 8 and 12 of both 16-bit halves.  Merged under
// the fp16 exponent of 1024 (10 fraction bits), a nibble at bits 0-3 gives
// 1024 + c and one at bits 4-7 gives 1024 + 16 c, both exact, so the pairs
// (k2, k3) and (k6, k7) need no shift: they carry a factor 16, which the
// activations of those k (k % 8 in {2, 3, 6, 7}) take off.  Subtracting
// 1024 + z (or 1024 + 16 z) is exact; the product with the scale is rounded
// once to fp16.
__device__ __forceinline__ void dequant_w4_f16(const uint32_t (&q)[8], uint32_t z, uint32_t s2,
                                               uint32_t (&a)[32]) {
  const uint32_t zl = (0x6400u | z) * 0x00010001u;           // (1024 + z) x2
  const uint32_t zh = (0x6400u | (z << 4)) * 0x00010001u;    // (1024 + 16 z) x2
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q8 = q[w] >> 8;
    a[4 * w + 0] = mul_f16x2(sub_f16x2(lop3_and_or(q[w], 0x000F000Fu, 0x64006400u), zl), s2);
    a[4 * w + 1] = mul_f16x2(sub_f16x2(lop3_and_or(q[w], 0x00F000F0u, 0x64006400u), zh), s2);
    a[4 * w + 2] = mul_f16x2(sub_f16x2(lop3_and_or(q8, 0x000F000Fu, 0x64006400u), zl), s2);
    a[4 * w + 3] = mul_f16x2(sub_f16x2(lop3_and_or(q8, 0x00F000F0u, 0x64006400u), zh), s2);
  }
}

// int8: the 64 codes of group j (128-byte swizzle as above) as exact bf16.
// A biased byte b = code + 128 becomes the fp32 2^23 + b, minus 2^23 + 128
// gives the code exactly, and |code| <= 127 fits bf16's 8-bit significand.
__device__ __forceinline__ void dequant_w8(uint32_t row_addr, uint32_t m, int j, uint32_t (&a)[32]) {
  const uint32_t sw = m & 7u;
  const uint64_t bias = pack_f32x2(0x4B000080u, 0x4B000080u);  // (2^23 + 128) x 2
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = lds128(row_addr + (((uint32_t)(4 * j + c) ^ sw) << 4));
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t u = words[w] ^ 0x80808080u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t f = sub_f32x2(pack_f32x2(__byte_perm(u, 0x4B000000u, 0x7540u | (2 * h)),
                                                __byte_perm(u, 0x4B000000u, 0x7540u | (2 * h + 1))),
                                     bias);
        a[8 * c + 2 * w + h] =
            pack_bf16x2(__uint_as_float((uint32_t)f), __uint_as_float((uint32_t)(f >> 32)));
      }
    }
  }
}

// int8 with a group scale: code * scale rounded once to fp16.  A biased byte
// b = code + 128 under the fp16 exponent of 1024 is 1024 + b; minus 1152
// gives the code exactly.
__device__ __forceinline__ void dequant_w8_f16(uint32_t row_addr, uint32_t m, int j, uint32_t s2,
                                               uint32_t (&a)[32]) {
  const uint32_t sw = m & 7u;
  const uint32_t bias = 0x64806480u;                             // (1024 + 128) x2
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = lds128(row_addr + (((uint32_t)(4 * j + c) ^ sw) << 4));
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t u = words[w] ^ 0x80808080u;
      a[8 * c + 2 * w] = mul_f16x2(sub_f16x2(__byte_perm(u, 0x6464u, 0x5140u), bias), s2);
      a[8 * c + 2 * w + 1] = mul_f16x2(sub_f16x2(__byte_perm(u, 0x6464u, 0x5342u), bias), s2);
    }
  }
}

// One 16-byte chunk (8 consecutive k of one activation row, starting at a
// multiple of 8) from bf16 to the fp16 operand; with `nib` the elements
// k % 8 in {2, 3, 6, 7} (words 1 and 3) are divided by 16.
__device__ __forceinline__ uint4 chunk_bf16_to_f16(uint4 v, bool nib) {
  const float d = nib ? 0.0625f : 1.f;
  auto cv = [](uint32_t w, float f) {
    return pack_f16x2(__uint_as_float(w << 16) * f, __uint_as_float(w & 0xFFFF0000u) * f);
  };
  return make_uint4(cv(v.x, 1.f), cv(v.y, d), cv(v.z, 1.f), cv(v.w, d));
}

// The fields of a GEMM the workers' epilogue needs, held in registers while
// the walk stays in that GEMM (stores to the output could alias the entry as
// far as the compiler knows, so reading them from the entry each time would
// reload them after every store).
struct EpiEntry {
  void* y;
  const uint16_t* chscale;
  int e, N, T, y_f32, pair, per_channel;
  // a CTA's range holds at most two tiles that other CTAs share (its first
  // and its last); their first and last contributors, found once per GEMM
  int tile_a, first_a, last_a, tile_b, first_b, last_b;
};

// End of a worker's segment of a tile: v holds its rows m, accumulator
// columns c0.. of the CTA's share of the tile.  A whole tile is written out.
// A tile split over several CTAs is finished by its first contributor (the
// CTA holding its first k, whose share is the last segment of its range and
// so, in time, usually the last to complete): every other contributor adds
// its part into the tile's fp32 slot and counts itself in with a release;
// the finisher adds the slot's sum (already in shared memory at `pre_row`
// when the others had counted in by the time its segment started, else
// waited for and read here) to its own part.  False when that wait gives up
// (abort or time limit).
template <int QUANT, int TPAD>
__device__ __forceinline__ bool finish_segment(const EpiEntry& en, int tile, bool whole, bool from0,
                                            float (&v)[Cfg<QUANT, TPAD>::kCols], const float* pre_row,
                                            const Params& p, int m, int c0, int wk, int lane,
                                            const Ctl& ctl) {
  constexpr int kCols = Cfg<QUANT, TPAD>::kCols;
  const int row = tile * kTileM + m;
  if (en.per_channel) {
    const float osc = row < en.N ? __half2float(__ushort_as_half(en.chscale[row])) : 1.f;
#pragma unroll
    for (int c = 0; c < kCols; ++c) v[c] *= osc;
  }
  bool finished = whole;
  if (!whole) {
    // the tile's fp32 slot and counters are keyed by the entry and the
    // tile's first contributor (unique among the split tiles in flight)
    const bool a = tile == en.tile_a;
    const int c_first = a ? en.first_a : en.first_b;
    const int c_last = a ? en.last_a : en.last_b;
    const size_t key = (size_t)(en.e % kSplitKeys) * p.slot_ctas + c_first;
    float* slot = p.partials + (key * kTileM + m) * TPAD + c0;
    int* cnt = p.split_cnt + key * kGemmWorkers + wk;
    if (!from0) {
#pragma unroll
      for (int c = 0; c < kCols; c += 4) red_add_f32x4(slot + c, v[c], v[c + 1], v[c + 2], v[c + 3]);
      __syncwarp();
      if (lane == 0) red_release_gpu_add(cnt, 1);
    } else {
      float pre[kCols];
      if (pre_row) {
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const float4 s4 = *reinterpret_cast<const float4*>(pre_row + c);
          pre[c] = s4.x;
          pre[c + 1] = s4.y;
          pre[c + 2] = s4.z;
          pre[c + 3] = s4.w;
        }
      } else {
        int ready = 1;
        if (lane == 0) ready = wait_count(cnt, c_last - c_first, ctl) ? 1 : 0;
        ready = __shfl_sync(0xffffffffu, ready, 0);
        __syncwarp();   // orders lane 0's acquire before the other lanes' reads
        if (!ready) return false;
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const float4 s4 = ldcg_f32x4(slot + c);
          pre[c] = s4.x;
          pre[c + 1] = s4.y;
          pre[c + 2] = s4.z;
          pre[c + 3] = s4.w;
        }
      }
#pragma unroll
      for (int c = 0; c < kCols; ++c) v[c] += pre[c];
#pragma unroll
      for (int c = 0; c < kCols; c += 4)
        __stcg(reinterpret_cast<float4*>(slot + c), make_float4(0.f, 0.f, 0.f, 0.f));
      if (lane == 0) __stcg(cnt, 0);
      finished = true;
    }
  }
  if (finished) {
    if (row < en.N) {
      // a rotated bf16 GEMM's columns come in (rounded, remainder) pairs per token
      const int pair = en.pair;
      const int N = en.N, T = en.T;
      if (en.y_f32) {
        float* y = reinterpret_cast<float*>(en.y) + row;
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          if (pair && (c & 1)) continue;
          const int t = (c0 + c) >> pair;
          const float out = pair ? v[c] + v[c + 1 < kCols ? c + 1 : c] : v[c];
          if (t < T) y[(size_t)t * N] = out;
        }
      } else {
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(en.y) + row;
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          if (pair && (c & 1)) continue;
          const int t = (c0 + c) >> pair;
          const float out = pair ? v[c] + v[c + 1 < kCols ? c + 1 : c] : v[c];
          if (t < T) y[(size_t)t * N] = __float2bfloat16_rn(out);
        }
      }
    }
    if (p.gate) {
      __syncwarp();
      if (lane == 0) red_release_gpu_add(&p.done[en.e], 1);
    }
  }
  return true;
}

// One converting warp's part of a landed activation slot (warp `cw` of
// kConvW): for a GEMM that converts in shared memory, rewrite its share of
// the bf16 slot in place as the fp16 operand (a 16-byte chunk holds 8
// consecutive k at any swizzle position, so every chunk stays where it is);
// then count the warp in on the slot's xconv barrier.
template <class C>
__device__ __forceinline__ void convert_share(int mode, uint8_t* slot, uint64_t* conv, int cw, int lane) {
  if (mode) {
    constexpr int kChunks = C::kSub * C::kXBox / 16;
    const bool nib = mode == 2;
    uint4* c = reinterpret_cast<uint4*>(slot);
#pragma unroll 4
    for (int i = cw * 32 + lane; i < kChunks; i += C::kConvW * 32) c[i] = chunk_bf16_to_f16(c[i], nib);
    fence_proxy_async_smem();   // the MMA reads the slot through the async proxy
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(conv);
}

template <int QUANT, int TPAD>
__global__ void __maxnreg__((Cfg<QUANT, TPAD>::kMaxRegs))
    qgemm_kernel(const __grid_constant__ GemmEntry e0, const Params p) {
  using C = Cfg<QUANT, TPAD>;
  constexpr int SW = C::kWSlots, SX = C::kXSlots, NA = C::kNA, SUB = C::kSub;
  constexpr int kCols = C::kCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* xreg = smem;
  uint8_t* wreg = smem + SX * C::kXSlot;
  float* pre_s = reinterpret_cast<float*>(wreg + SW * C::kWSlot);
  uint8_t* ctrl = wreg + SW * C::kWSlot + C::kPreBytes;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* wempty = wfull + SW;
  uint64_t* xfull = wempty + SW;
  uint64_t* afull = xfull + SX;
  // mdone[u % kDM]: every MMA warp has committed stage u (its A slot and
  // activation slot may be reused once its MMAs complete)
  uint64_t* mdone = afull + NA;
  uint64_t* sfull = mdone + C::kDM;
  uint64_t* sempty = sfull + 2;
  // xconv[s]: the activation slot holds the MMA's operand form (after the
  // converters, for GEMMs that convert in shared memory)
  uint64_t* xconv = sempty + 2;
  // xrec[s]: the control record of the stage in activation slot s (written
  // by the activation producer before the slot's copies)
  uint2* xrec = reinterpret_cast<uint2*>(xconv + SX);
  // prebar[w]: worker w's part of an early-fetched split-tile sum has landed
  uint64_t* prebar = reinterpret_cast<uint64_t*>(xrec + SX);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(prebar + kGemmWorkers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const GemmEntry* E = p.entries ? p.entries : &e0;
  const int nE = p.entries ? p.n_entries : 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], kGemmWorkers);
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xconv[s], C::kConvW);
    }
    for (int s = 0; s < NA; ++s) mbar_init(&afull[s], kGemmWorkers);
    for (int s = 0; s < C::kDM; ++s) mbar_init(&mdone[s], C::kMmaW);   // one commit per MMA warp
    for (int s = 0; s < kGemmWorkers; ++s) mbar_init(&prebar[s], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], C::kMmaW);
      mbar_init(&sempty[s], kGemmWorkers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kAlloc) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::kWProd && lane == 0) {
    prefetch_tensormap(&E[0].tm_codes);
    if (E[0].scale_rows) prefetch_tensormap(&E[0].tm_scales);
    if (QUANT == kW4) prefetch_tensormap(&E[0].tm_zeros);
  }
  if (warp == C::kXProd && lane == 0) prefetch_tensormap(&E[0].tm_x);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  pdl_launch_dependents();

  const Ctl ctl{abort_flag, p.abort_all, p.err, p.wait_ns};

  if (warp == C::kWProd) {
    // ------------------------------------------------------------ weight producer
    // (the whole warp walks; one elected lane issues)
    const bool leader = elect_one();
    const uint64_t pol = policy_evict_first();
    // a GEMM's tensor maps and stage sizes, cached while the walk stays in it
    struct Src {
      int e = -1;
      const CUtensorMap *codes = nullptr, *scales = nullptr, *zeros = nullptr;
      uint32_t tx = 0;
      int rows = 0, gshift = 0;
      __device__ __forceinline__ void at(const GemmEntry* E, int nE, int e_, bool lead) {
        if (e_ == e) return;
        e = e_;
        if (lead && e + 1 < nE) {
          // the next GEMM's descriptors, so that its first copies do not wait for them
          prefetch_tensormap(&E[e + 1].tm_codes);
          prefetch_tensormap(&E[e + 1].tm_scales);
          prefetch_tensormap(&E[e + 1].tm_zeros);
        }
        codes = &E[e].tm_codes;
        scales = &E[e].tm_scales;
        zeros = &E[e].tm_zeros;
        tx = E[e].tx_w;
        rows = E[e].scale_rows;
        gshift = E[e].gshift;
      }
    };
    Walk w(E, nE, G, cta);
    Walk pf(E, nE, G, cta);
    Src sw, spf;
    int pf_n = 0;
    Ring<SW> r;
    int n = 0, skipped = -1;
    const int last_e = last_entry_of(E, nE, G, cta);
    bool from0 = false;
    auto prefetch_next = [&]() {
      spf.at(E, nE, pf.e, false);
      if (leader) {
        tma_prefetch_2d(spf.codes, pf.kst * 128, pf.tile * kTileM);
        if (spf.rows) {
          const int g0 = (pf.kst * C::kStageKK) >> spf.gshift;
          tma_prefetch_2d(spf.scales, pf.tile * kTileM, g0);
          if (QUANT == kW4) tma_prefetch_2d(spf.zeros, pf.tile * (kTileM / 2), g0);
        }
      }
      pf.next();
      ++pf_n;
    };
    for (; w.valid(); w.next(), r.next(), ++n) {
      while (pf.valid() && pf_n < n + p.pf_dist) prefetch_next();
      if (!__all_sync(0xffffffffu, mbar_test_wait(&wempty[r.slot], r.phase ^ 1))) {
        // the ring is full: run the L2 stream further ahead meanwhile
        while (pf.valid() && pf_n < n + p.pf_max &&
               !__all_sync(0xffffffffu, mbar_test_wait(&wempty[r.slot], r.phase ^ 1)))
          prefetch_next();
        if (!wait_warp(&wempty[r.slot], r.phase ^ 1, ctl)) break;
      }
      if (n == p.skip_unit && cta == 0) {
        skipped = n;   // test hook: this stage's weights never arrive
        continue;
      }
      sw.at(E, nE, w.e, leader);
      const bool seg_start = w.kst == 0 || w.u == w.ub;
      if (seg_start) from0 = w.kst == 0;
      const bool seg_end = w.kst == w.ks - 1 || w.u == w.ue - 1;
      // a segment from the tile's first k that stops before its last one
      // finishes a tile split over several CTAs
      const bool fin_start = seg_start && w.kst == 0 && w.u - w.kst + w.ks > w.ue;
      const uint32_t rec = (uint32_t)w.e | (seg_end ? kStageSegEnd : 0u) |
                           (seg_end && from0 && w.kst == w.ks - 1 ? kStageWhole : 0u) |
                           (seg_end && from0 ? kStageFrom0 : 0u) | (fin_start ? kStageFinStart : 0u) |
                           (w.e == last_e && w.u == w.ue - 1 ? kStageLast : 0u);
      if (leader) {
        uint8_t* st = wreg + r.slot * C::kWSlot;
        *reinterpret_cast<uint2*>(st + C::kCtlOff) = make_uint2(rec, (uint32_t)w.tile);
        mbar_arrive_expect_tx(&wfull[r.slot], sw.tx);
        tma_load_2d_hint(st, sw.codes, &wfull[r.slot], w.kst * 128, w.tile * kTileM, pol);
        if (sw.rows) {
          const int g0 = (w.kst * C::kStageKK) >> sw.gshift;
          tma_load_2d_hint(st + C::kScaleOff, sw.scales, &wfull[r.slot], w.tile * kTileM, g0, pol);
          if (QUANT == kW4)
            tma_load_2d_hint(st + C::kZeroOff, sw.zeros, &wfull[r.slot], w.tile * (kTileM / 2), g0, pol);
        }
      }
      __syncwarp();
    }
    if (*abort_flag && leader) {
      // copies still in flight into this CTA's shared memory land before it exits
      for (int j = (n > SW ? n - SW : 0); j < n; ++j)
        if (j != skipped) drain_bar(&wfull[j % SW], (uint32_t)((j / SW) & 1));
    }
  } else if (warp == C::kXProd) {
    // ------------------------------------------------------------ activation producer
    // activations (and the rotation's scratch) may be written by the previous kernel
    pdl_wait_prior();
    const bool leader = elect_one();
    Ring<SX> r;
    Ring<C::kDM> rdone;     // stage whose MMAs free the slot: n - SX
    int n = 0, verified = 0;
    bool ok = true;
    const int last_e = last_entry_of(E, nE, G, cta);
    for (int e = 0; e < nE && ok; ++e) {
      const GemmEntry& en = E[e];
      const int ub = unit_begin(cta, en.units, G), ue = unit_begin(cta + 1, en.units, G);
      const bool gate = p.gate && en.wait_prev && e > 0;
      if (ub < ue && lane == 0) {
        // while the gate is closed: the GEMM's activation descriptor, and
        // (activations read as given) its first boxes into L2 -- a hint
        // only, still correct if an earlier GEMM writes them meanwhile
        prefetch_tensormap(&en.tm_x);
        if (!en.prep) {
          const int ks0 = en.ks;
          int k0 = ub % ks0;
          for (int u = ub; u < ue && u < ub + SX; ++u) {
#pragma unroll
            for (int j = 0; j < SUB; ++j) tma_prefetch_2d(&en.tm_x, k0 * C::kStageKK + kGroupK * j, 0);
            if (++k0 == ks0) k0 = 0;
          }
        }
      }
      if (gate && (en.prep || ub < ue)) {
        // this GEMM reads what the earlier ones wrote: wait until every one
        // of their tiles is finished
        while (verified < e) {
          if (!__all_sync(0xffffffffu, wait_count(&p.done[verified], kGemmWorkers * E[verified].tiles, ctl))) {
            ok = false;
            break;
          }
          ++verified;
        }
        if (!ok) break;
      }
      if (en.prep) {
        // this CTA's share of the activations in the MMA's operand form,
        // written into the scratch copy, then published
        const int K = en.K, kind = en.kind;
        const uint16_t* x = en.x;
        uint16_t* xp = en.xprep;
        if (en.prep == 1 && en.rot_block == 32) {
          // rotation, 32-element blocks: one lane per (row, block), the
          // block in its registers (a warp rotates 32 blocks at once)
          const int8_t* signs = en.signs;
          const float rscale = en.rot_scale;
          const int nblk = K / 32;
          const int pairs = en.T * nblk;
          for (int pp = cta * 32 + lane; pp < pairs; pp += G * 32) {
            const int t = pp / nblk, b = pp - t * nblk;
            const size_t col = (size_t)b * 32;
            const uint16_t* xs = x + (size_t)t * K + col;
            if (kind == kGemmBf16)
              fwht_thread<32, kFwhtBf16Split>(xs, xp + (size_t)(2 * t) * K + col, signs + col, rscale, (size_t)K);
            else if (kind == kGemmF16Nib)
              fwht_thread<32, kFwhtF16Nib>(xs, xp + (size_t)t * K + col, signs + col, rscale);
            else
              fwht_thread<32, kFwhtF16>(xs, xp + (size_t)t * K + col, signs + col, rscale);
          }
        } else if (en.prep == 1) {
          // rotation: one warp per (row, block)
          const int B = en.rot_block;
          const int8_t* signs = en.signs;
          const float rscale = en.rot_scale;
          const int nblk = K / B;
          const int pairs = en.T * nblk;
          for (int pp = cta; pp < pairs; pp += G) {
            const int t = pp / nblk, b = pp - t * nblk;
            const size_t col = (size_t)b * B;
            const uint16_t* xs = x + (size_t)t * K + col;
            if (kind == kGemmBf16) {
              // bf16 operands: row t as two rows, 2t (rounded) and 2t+1 (remainder)
              fwht_warp_any<kFwhtBf16Split>(B, xs, xp + (size_t)(2 * t) * K + col, signs + col, rscale,
                                            lane, (size_t)K);
            } else if (kind == kGemmF16Nib) {
              fwht_warp_any<kFwhtF16Nib>(B, xs, xp + (size_t)t * K + col, signs + col, rscale, lane);
            } else {
              fwht_warp_any<kFwhtF16>(B, xs, xp + (size_t)t * K + col, signs + col, rscale, lane);
            }
          }
        } else {
          // conversion to fp16: 16-byte chunks of 8 consecutive k spread
          // over every lane of every CTA
          const bool nib = kind == kGemmF16Nib;
          const int chunks = en.T * (K / 8);
          for (int i = cta * 32 + lane; i < chunks; i += G * 32) {
            const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)i * 8);
            *reinterpret_cast<uint4*>(xp + (size_t)i * 8) = chunk_bf16_to_f16(v, nib);
          }
        }
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) red_release_gpu_add(&p.rot_done[e], 1);
      }
      if (ub >= ue) continue;
      if (en.prep && !__all_sync(0xffffffffu, wait_count(&p.rot_done[e], G, ctl))) {
        ok = false;
        break;
      }
      if (gate || en.prep) fence_proxy_async_global();
      const CUtensorMap* tmx = &en.tm_x;
      const uint32_t xmode = (uint32_t)en.xconv << kStageConvShift;
      const uint32_t xidesc = en.idesc;
      const int ks = en.ks;
      int kst = ub % ks;
      for (int u = ub; u < ue; ++u, r.next(), ++n) {
        if (n >= SX) {
          if (!wait_warp(&mdone[rdone.slot], rdone.phase, ctl)) {
            ok = false;
            break;
          }
          rdone.next();
        }
        if (leader) {
          uint8_t* st = xreg + r.slot * C::kXSlot;
          const bool seg_end = kst == ks - 1 || u == ue - 1;
          xrec[r.slot] = make_uint2((uint32_t)e | (seg_end ? kStageSegEnd : 0u) |
                                        (e == last_e && u == ue - 1 ? kStageLast : 0u) | xmode,
                                    xidesc);
          mbar_arrive_expect_tx(&xfull[r.slot], (uint32_t)(SUB * C::kXBox));
#pragma unroll
          for (int j = 0; j < SUB; ++j)
            tma_load_2d(st + j * C::kXBox, tmx, &xfull[r.slot], kst * C::kStageKK + kGroupK * j, 0);
        }
        __syncwarp();
        if (++kst == ks) kst = 0;
      }
    }
    if (*abort_flag && leader) {
      for (int j = (n > SX ? n - SX : 0); j < n; ++j) drain_bar(&xfull[j % SX], (uint32_t)((j / SX) & 1));
    }
  } else if (warp < C::kMma0) {
    // ------------------------------------------------------------ converters
    // (warps 2 and 3 when there are two MMA warps; else they wait at the
    // final barrier)
    if (C::kConv0 == 2 && (p.prep_flags & kAnyConv)) {
      Ring<SX> r;
      int mode = 0;
      for (bool more = last_entry_of(E, nE, G, cta) >= 0; more; r.next()) {
        if (!wait_warp(&xfull[r.slot], r.phase, ctl)) break;
        const uint32_t rec = xrec[r.slot].x;
        mode = (int)((rec >> kStageConvShift) & 3u);
        convert_share<C>(mode, xreg + r.slot * C::kXSlot, &xconv[r.slot], warp - C::kConv0, lane);
        if (rec & kStageLast) more = false;
      }
    }
  } else if (warp < C::kWorker0) {
    // ------------------------------------------------------------ MMA issue
    // warp kMma0 + k issues the K16 MMAs of groups k*kGpm .. into the
    // current segment's accumulator (the whole warp follows the activation
    // slots' control records; one elected lane issues)
    const int k = warp - C::kMma0;
    const bool leader = elect_one();
    const uint64_t xdesc0 = smem_desc_sw128(xreg);
    Ring<NA> ra;
    Ring<SX> rx;
    Ring<C::kDM> rm;
    Ring<2> rs;
    int last_m = -1, xconv_mode = 0;
    const bool any_conv = (p.prep_flags & kAnyConv) != 0;
    uint32_t idesc = 0, last_mph = 0;
    bool seg_start = true;
    for (bool more = last_entry_of(E, nE, G, cta) >= 0; more;) {
      // the stage's activations (and its control record) have landed
      if (!wait_warp(&xfull[rx.slot], rx.phase, ctl)) break;
      const uint2 xr = xrec[rx.slot];
      const uint32_t rec = xr.x;
      idesc = xr.y;
      xconv_mode = (int)((rec >> kStageConvShift) & 3u);
      if (any_conv) convert_share<C>(xconv_mode, xreg + rx.slot * C::kXSlot, &xconv[rx.slot], warp - C::kConv0, lane);
      // a segment starts on a zeroed accumulator (zeroed at the start of the
      // launch, then by the workers after they read it)
      if (seg_start && !wait_warp(&sempty[rs.slot], rs.phase, ctl)) break;
      if (!wait_warp(&afull[ra.slot], ra.phase, ctl)) break;
      // a converted slot is ready once every converting warp has done its share
      if (xconv_mode && !wait_warp(&xconv[rx.slot], rx.phase, ctl)) break;
      tc_fence_after();
      const bool seg_end = (rec & kStageSegEnd) != 0;
      if (leader) {
        const uint32_t d = tbase + rs.slot * C::kDCols;
        const uint32_t a0 = tbase + C::kA0 + ra.slot * C::kACols;
        const uint64_t xd = xdesc0 + (uint64_t)((rx.slot * C::kXSlot) >> 4);
#pragma unroll
        for (int gi = 0; gi < C::kGpm; ++gi) {
          const int g = k * C::kGpm + gi;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: 8 TMEM columns (16 elements) per K16 step; B: +32 bytes inside the swizzled row
            mma_ts(d, a0 + g * 32 + kk * 8, xd + (uint64_t)((g * C::kXBox) >> 4) + kk * 2, idesc, 1u);
          }
        }
        mma_commit(&mdone[rm.slot]);
        if (seg_end) mma_commit(&sfull[rs.slot]);
      }
      __syncwarp();
      last_m = rm.slot;
      last_mph = rm.phase;
      if (seg_end) rs.next();
      seg_start = seg_end;
      ra.next();
      rx.next();
      rm.next();
      if (rec & kStageLast) more = false;
    }
    // the CTA frees its tensor memory and shared memory only after its
    // MMAs have completed and their commits have arrived
    if (last_m >= 0 && leader) drain_bar(&mdone[last_m], last_mph);
  } else {
    // ------------------------------------------------------------ workers
    const int wk = warp - C::kWorker0;
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int h = wk >> 2;
    const int m = q * 32 + lane;                  // weight row inside the tile
    const int j0 = h * C::kGpw;                   // first 64-k group this warp dequantises
    const int c0 = h * kCols;                     // first accumulator column this warp reads
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t zshift = (m & 1) * 4;
    const uint32_t wbase = smem_u32(wreg);
    // per-entry shared-memory offsets inside a weight slot: this row's zero
    // byte and scale of each dequantised group
    uint32_t zoff[C::kGpw] = {}, soff[C::kGpw] = {};
    int ed = -1, ee = -1, kind = 0;
    EpiEntry epi{};
    auto enter_d = [&](int e) {
      ed = e;
      if (p.entries) {
        // the fields the epilogue reads for this GEMM, into L1 ahead of it
        const uint8_t* fe = reinterpret_cast<const uint8_t*>(&E[e].x);
        prefetch_l1(fe);
        prefetch_l1(fe + 64);
      }
      const int gsh = E[e].gsh;
      kind = E[e].kind;
#pragma unroll
      for (int i = 0; i < C::kGpw; ++i) {
        const int row = (kGroupK * (j0 + i)) >> gsh;
        zoff[i] = C::kZeroOff + row * 64 + (m >> 1);
        soff[i] = C::kScaleOff + row * (kTileM * 2) + m * 2;
      }
    };
    auto enter_e = [&](int e) {
      ee = e;
      const GemmEntry& en = E[e];
      epi.y = en.y;
      epi.chscale = en.chscale;
      epi.e = e;
      epi.N = en.N;
      epi.T = en.T;
      epi.y_f32 = en.y_f32;
      epi.pair = en.rot_block && en.kind == kGemmBf16 ? 1 : 0;
      epi.per_channel = en.scale_rows == 0;
      const int U = en.units, ks = en.ks;
      const int ub = unit_begin(cta, U, G), ue = unit_begin(cta + 1, U, G);
      if (ub < ue) {
        epi.tile_a = ub / ks;
        epi.first_a = cta_of_unit(epi.tile_a * ks, U, G);
        epi.last_a = cta_of_unit(epi.tile_a * ks + ks - 1, U, G);
        epi.tile_b = (ue - 1) / ks;
        epi.first_b = cta_of_unit(epi.tile_b * ks, U, G);
        epi.last_b = cta_of_unit(epi.tile_b * ks + ks - 1, U, G);
      }
    };
    Ring<SW> rw;
    Ring<NA> ra;
    // stage n reuses the A slot of stage n - NA once that stage's MMAs are
    // done: ring position n - NA + kDM, so the first NA waits name the phase
    // before a barrier's first one, which counts as complete
    Ring<C::kDM> rm;
    rm.slot = C::kDM - NA;
    rm.phase = 1;
    Ring<2> rs;
    bool ok = true, pdl_done = false;
    bool more = last_entry_of(E, nE, G, cta) >= 0;   // this CTA owns any stage
    uint32_t prec = 0, ptile = 0;                     // the previous stage's control record
    // the other contributors' sum of the split tile this CTA finishes next
    // is copied into shared memory when that segment starts, if they have
    // all counted in by then (up to 16 columns a worker; wider tiles read it
    // at the epilogue)
    bool pre_ok = false;
    uint32_t pre_phase = 0;
    const float* pre_row = C::kPreBytes ? pre_s + (size_t)m * TPAD + c0 : nullptr;
    // both accumulators start at zero
#pragma unroll
    for (int sl = 0; sl < 2; ++sl) tmem_zero_cols<kCols>(tbase + lane_base + sl * C::kDCols + c0);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sempty[0]);
      mbar_arrive(&sempty[1]);
    }
    for (;;) {
      const bool has_d = more;
      uint32_t rec = 0, tile = 0;
      if (has_d) {
        // ---- dequantise the next stage into its A slot
        if (!wait_warp(&wfull[rw.slot], rw.phase, ctl)) {
          ok = false;
          break;
        }
        const uint32_t st = wbase + rw.slot * C::kWSlot;
        {
          const uint2 r2 = lds64(st + C::kCtlOff);
          rec = r2.x;
          tile = r2.y;
        }
        if ((int)(rec & 0xFFFFu) != ed) enter_d((int)(rec & 0xFFFFu));
        uint32_t words[C::kGpw][8];
        uint32_t zb[C::kGpw], s2[C::kGpw];
        if constexpr (QUANT == kW4) {
#pragma unroll
          for (int i = 0; i < C::kGpw; ++i) {
            load_w4(st + m * 128, m, j0 + i, words[i]);
            zb[i] = (lds_u8(st + zoff[i]) >> zshift) & 0xFu;
            s2[i] = (uint32_t)lds_u16(st + soff[i]) * 0x00010001u;
          }
        } else {
#pragma unroll
          for (int i = 0; i < C::kGpw; ++i) s2[i] = kind == kGemmF16 ? (uint32_t)lds_u16(st + soff[i]) * 0x00010001u : 0u;
        }
        // the A slot is free once the MMAs that read it (NA stages back) have completed
        if (!wait_warp(&mdone[rm.slot], rm.phase, ctl)) {
          ok = false;
          break;
        }
        rm.next();
        tc_fence_after();
        const uint32_t aslot = tbase + lane_base + C::kA0 + ra.slot * C::kACols;
#pragma unroll
        for (int i = 0; i < C::kGpw; ++i) {
          uint32_t a[32];
          if constexpr (QUANT == kW4) {
            dequant_w4_f16(words[i], zb[i], s2[i], a);
          } else {
            if (kind == kGemmF16)
              dequant_w8_f16(st + m * 128, m, j0 + i, s2[i], a);
            else
              dequant_w8(st + m * 128, m, j0 + i, a);
          }
          tmem_st_32x32b_x32(aslot + (j0 + i) * 32, a);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&afull[ra.slot]);
          mbar_arrive(&wempty[rw.slot]);   // codes, scales and zero points read
        }
        rw.next();
        ra.next();
        if (rec & kStageLast) more = false;
      }
      // ---- the previous stage: the end of a segment reads the accumulator
      // (one stage late, so that its MMAs complete behind this dequantisation)
      if (prec & kStageSegEnd) {
        if (!pdl_done) {
          // outputs and split-tile sums may still be used by the previous kernel
          pdl_wait_prior();
          pdl_done = true;
        }
        if ((int)(prec & 0xFFFFu) != ee) enter_e((int)(prec & 0xFFFFu));
        if (!wait_warp(&sfull[rs.slot], rs.phase, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dbase = tbase + lane_base + rs.slot * C::kDCols + c0;
        float v[kCols];
        tmem_ld_cols<kCols>(dbase, v);
        tmem_wait_ld();
        tmem_zero_cols<kCols>(dbase);     // the next segment on this accumulator adds from zero
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[rs.slot]);
        rs.next();
        const bool fin = (prec & (kStageWhole | kStageFrom0)) == kStageFrom0;
        const bool use_pre = fin && pre_ok;
        if (use_pre) {
          if (!wait_warp(&prebar[wk], pre_phase, ctl)) {
            ok = false;
            break;
          }
          pre_phase ^= 1u;
          pre_ok = false;
        }
        if (!finish_segment<QUANT, TPAD>(epi, (int)ptile, (prec & kStageWhole) != 0, (prec & kStageFrom0) != 0, v,
                                         use_pre ? pre_row : nullptr, p, m, c0, wk, lane, ctl)) {
          ok = false;
          break;
        }
      }
      if (C::kPreBytes && has_d && (rec & kStageFinStart)) {
        // this stage starts the segment that finishes a split tile: if the
        // other contributors have all counted in, fetch their sum now, so
        // that it lands while this segment's MMAs run
        if (!pdl_done) {
          // split-tile sums and counters may still be used by the previous kernel
          pdl_wait_prior();
          pdl_done = true;
        }
        const int e = (int)(rec & 0xFFFFu);
        const int U = E[e].units, ks = E[e].ks;
        const int need = cta_of_unit((int)tile * ks + ks - 1, U, G) - cta;
        const size_t key = (size_t)(e % kSplitKeys) * p.slot_ctas + cta;
        int ready = 0;
        if (lane == 0) ready = ld_acquire_gpu(p.split_cnt + key * kGemmWorkers + wk) >= need;
        ready = __shfl_sync(0xffffffffu, ready, 0);
        __syncwarp();   // orders lane 0's acquire before the other lanes' reads
        if (ready) {
          // one bulk copy per row of this warp's part, issued by lane 0
          // after its acquire (the async proxy reads what the acquire made
          // visible; this warp's earlier reads of the buffer come first)
          if (lane == 0) {
            fence_proxy_async_global();
            fence_proxy_async_smem();
            const int r0 = (warp & 3) * 32;
            mbar_arrive_expect_tx(&prebar[wk], (uint32_t)(32 * kCols * 4));
            for (int r = 0; r < 32; ++r)
              bulk_g2s(pre_s + (size_t)(r0 + r) * TPAD + c0,
                       p.partials + ((key * kTileM + r0 + r) * TPAD + c0), (uint32_t)(kCols * 4), &prebar[wk]);
          }
          __syncwarp();
          pre_ok = true;
        }
      }
      if (!has_d) break;
      prec = rec;
      ptile = tile;
    }
    if (!ok) {
      tmem_wait_st();
      tmem_wait_ld();
    }
    // a split-tile sum still being copied in lands before the CTA exits
    if (pre_ok && lane == 0) drain_bar(&prebar[wk], pre_phase);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kAlloc) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  if (threadIdx.x == 0 && (p.gate || (p.prep_flags & kAnyPrep))) {
    // the last CTA to leave resets the per-entry counters for the next launch
    __threadfence();
    const int old = atomic_add_acq_rel_gpu(p.exit_cnt, 1);
    if (old == G - 1) {
      for (int e = 0; e < nE; ++e) {
        p.done[e] = 0;
        p.rot_done[e] = 0;
      }
      *p.exit_cnt = 0;
      __threadfence();
    }
  }
}

template <int QUANT, int TPAD>
int launch_t(spec_ctx* ctx, const GemmEntry& e0, const GemmEntry* dev_entries, int n, int gate,
             int prep_flags, int G, cudaStream_t stream) {
  using C = Cfg<QUANT, TPAD>;
  Params p;
  p.entries = dev_entries;
  p.n_entries = n;
  p.gate = gate;
  p.prep_flags = prep_flags;
  p.slot_ctas = ctx->num_sms;
  p.partials = ctx->partials;
  p.split_cnt = ctx->split_cnt;
  p.done = ctx->done;
  p.rot_done = ctx->rot_done;
  p.exit_cnt = ctx->exit_cnt;
  p.err = ctx->err;
  p.abort_all = ctx->abort_all;
  p.wait_ns = ctx->test_wait_ns ? ctx->test_wait_ns : kWaitLimitNs;
  p.skip_unit = ctx->test_skip_unit;
  p.pf_dist = ctx->pf_dist;
  p.pf_max = ctx->pf_max;
  ctx->test_wait_ns = 0;
  ctx->test_skip_unit = -1;

  static std::atomic<uint32_t> attr_done{0};   // per instantiation, one bit per device
  const uint32_t bit = ctx->device < 32 ? (1u << ctx->device) : 0u;
  if (!bit || !(attr_done.load() & bit)) {
    int rc = check_cuda(cudaFuncSetAttribute(qgemm_kernel<QUANT, TPAD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes),
                        "cudaFuncSetAttribute(qgemm)");
    if (rc) return rc;
    attr_done.fetch_or(bit);
  }
  // programmatic stream serialisation: the launch may start while the
  // previous kernel finishes; every read of its results waits for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return check_cuda(cudaLaunchKernelEx(&cfg, qgemm_kernel<QUANT, TPAD>, e0, p), "qgemm launch");
}

template <int QUANT>
int launch_q(spec_ctx* ctx, int tpad, const GemmEntry& e0, const GemmEntry* dev, int n, int gate,
             int prep_flags, int G, cudaStream_t s) {
  switch (tpad) {
    case 16: return launch_t<QUANT, 16>(ctx, e0, dev, n, gate, prep_flags, G, s);
    case 32: return launch_t<QUANT, 32>(ctx, e0, dev, n, gate, prep_flags, G, s);
    case 48: return launch_t<QUANT, 48>(ctx, e0, dev, n, gate, prep_flags, G, s);
    case 64: return launch_t<QUANT, 64>(ctx, e0, dev, n, gate, prep_flags, G, s);
    default: return set_error(SPEC_ERR_SHAPE, "padded T=%d outside 16..64", tpad);
  }
}

int stage_k(int quant) { return quant == kW4 ? 256 : 128; }

// The MMA operand form of a GEMM (see GemmKind).
int kind_of(const GemmArgs& a) {
  return a.quant == kW4 ? kGemmF16Nib : (a.group_size ? kGemmF16 : kGemmBf16);
}

}  // namespace

int build_entry(spec_ctx* ctx, const GemmArgs& a, int tpad, int index, GemmEntry* out) {
  GemmEntry e;
  std::memset(&e, 0, sizeof(e));
  const int SK = stage_k(a.quant);
  const bool rot = a.signs != nullptr;
  const int kind = kind_of(a);
  // activations the MMA reads in another form are prepared inside the launch
  // into the scratch copy of this GEMM's key (a rotated bf16 GEMM's as 2T
  // rows, (rounded, remainder) per token)
  // small GEMMs convert each CTA's activation slots in shared memory; large
  // ones (many stages per CTA, each slot read many times) convert once, with
  // every CTA taking a share, into the scratch copy
  const long long units = (long long)((a.K + SK - 1) / SK) * ((a.N + kTileM - 1) / kTileM);
  const int xconv = !rot && kind != kGemmBf16 && units <= (long long)kLocalConvStages * ctx->num_sms
                        ? (kind == kGemmF16Nib ? 2 : 1)
                        : 0;
  const int prep = rot ? 1 : (kind != kGemmBf16 && !xconv ? 2 : 0);
  uint16_t* xp = prep ? ctx->xprep + (size_t)(index % kSplitKeys) * kMaxT * kMaxK : nullptr;
  const uint16_t* xsrc = prep ? xp : a.x;
  const uint64_t xrows = rot && kind == kGemmBf16 ? 2 * (uint64_t)a.T : (uint64_t)a.T;
  if ((int)xrows > tpad) return set_error(SPEC_ERR_SHAPE, "internal: padded T %d below %d rows", tpad, (int)xrows);
  int rc = encode_tmap_2d(&e.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xsrc, (uint64_t)a.K, xrows,
                          (uint64_t)a.K * 2, kGroupK, tpad, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t row_bytes = a.quant == kW4 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
  rc = encode_tmap_2d(&e.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qcodes, row_bytes, (uint64_t)a.N,
                      row_bytes, 128, kTileM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  int sr = 0;
  if (a.group_size) {
    const uint64_t groups = (uint64_t)(a.K / a.group_size);
    sr = a.group_size < SK ? SK / a.group_size : 1;
    rc = encode_tmap_2d(&e.tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)a.N, groups,
                        (uint64_t)a.N * 2, kTileM, sr, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
    if (a.quant == kW4) {
      rc = encode_tmap_2d(&e.tm_zeros, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.zeros, (uint64_t)a.N / 2, groups,
                          (uint64_t)a.N / 2, kTileM / 2, sr, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc) return rc;
    }
  }
  e.x = a.x;
  e.signs = a.signs;
  e.xprep = xp;
  e.chscale = a.group_size ? nullptr : a.scales;
  e.y = a.y;
  e.T = a.T;
  e.N = a.N;
  e.K = a.K;
  e.rot_block = rot ? a.rot_block : 0;
  e.rot_scale = rot ? (float)(1.0 / std::sqrt((double)a.rot_block)) : 0.f;
  e.ks = (a.K + SK - 1) / SK;
  e.tiles = (a.N + kTileM - 1) / kTileM;
  e.units = e.ks * e.tiles;
  e.gshift = 0;
  while (a.group_size && (1 << e.gshift) < a.group_size) ++e.gshift;
  e.gsh = (a.group_size == 0 || a.group_size > SK) ? 31 : e.gshift;
  e.scale_rows = sr;
  e.tx_w = kTileM * 128 + (uint32_t)sr * kTileM * 2 + (a.quant == kW4 ? (uint32_t)sr * 64 : 0u);
  e.y_f32 = a.y_f32;
  e.wait_prev = a.wait_prev;
  e.kind = kind;
  e.prep = prep;
  e.xconv = xconv;
  e.idesc = kind == kGemmBf16 ? idesc_bf16_f32(128, tpad) : idesc_f16_f32(128, tpad);
  *out = e;
  return SPEC_OK;
}

int gemm_tpad(const GemmArgs& a) {
  const int rows = a.signs && kind_of(a) == kGemmBf16 ? 2 * a.T : a.T;
  return (rows + 15) / 16 * 16;
}

int launch_qgemm(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s) {
  const int tpad = gemm_tpad(a);
  GemmEntry e;
  int rc = build_entry(ctx, a, tpad, 0, &e);
  if (rc) return rc;
  // persistent grid of at most one CTA per SM with an even share of units each
  long long G = ctx->num_sms;
  if (G > e.units) G = e.units;
  const long long per = (e.units + G - 1) / G;
  G = (e.units + per - 1) / per;
  if (e.prep) G = ctx->num_sms < e.units ? ctx->num_sms : e.units;
  const int flags = (e.prep ? kAnyPrep : 0) | (e.xconv ? kAnyConv : 0);
  return a.quant == kW4 ? launch_q<kW4>(ctx, tpad, e, nullptr, 1, 0, flags, (int)G, s)
                        : launch_q<kW8>(ctx, tpad, e, nullptr, 1, 0, flags, (int)G, s);
}

int launch_qgemm_stack(spec_ctx* ctx, const spec_gemm_stack* st, cudaStream_t s) {
  GemmEntry dummy;
  std::memset(&dummy, 0, sizeof(dummy));
  return st->quant == kW4
             ? launch_q<kW4>(ctx, st->tpad, dummy, st->dev_entries, st->n, 1, st->prep_flags, ctx->num_sms, s)
             : launch_q<kW8>(ctx, st->tpad, dummy, st->dev_entries, st->n, 1, st->prep_flags, ctx->num_sms, s);
}

}  // namespace sv
