// The split engine of the verify GEMM (the default; the persistent engine is
// in qgemm.cu): one launch per GEMM, low-bit weights times the T drafted
// positions' activations, on the sm_103a tensor cores.
//
// What it computes ("Karpathy's Trick for Faster Local LLMs Finally Has Proper
// Tooling", section "How Uzu optimizes bytes and tokens per pass": 4-bit
// asymmetric Medium tier, 8-bit symmetric Large tier, one scale per group):
//   y[t][n] = sum_k x[t][k] * (code[n][k] - zero[g][n]) * scale[g][n]   (int4)
//   y[t][n] = sum_k x[t][k] *  code[n][k]              * scale         (int8)
// A rotated GEMM reads activations that the standalone rotation kernel
// wrote just before it on the same stream.
//
// Design (swap-AB: 128 weight rows are the MMA's M dimension, the T drafted
// positions its N dimension; one CTA per SM owns all 512 TMEM columns):
//  * two TMA warps stream stages into a shared-memory ring: one issues per
//    stage the 128-byte line of codes of each of the 128 weight rows (256 k
//    of int4 or 128 k of int8 -- full-width HBM bursts) and the stage's scale
//    and zero rows, the other the stage's bf16 activation boxes, each on its
//    own barrier (one issuing thread that also issued the activation boxes
//    kept too few weight bytes in flight to stream at full HBM rate);
//  * eight dequantisation warps (two per TMEM lane quadrant, one weight row
//    per thread) turn codes into exact bf16 integers (code - zero, or the
//    int8 code) and write them straight into a TMEM ring with tcgen05.st --
//    the MMA's A operand lives in TMEM, so dequantised weights never touch
//    shared memory, and the activations are used as stored;
//  * one MMA warp per 64-k group issues that group's four K16 MMAs into the
//    group's own fp32 partial (a ring of per-stage partial sets in TMEM);
//  * four epilogue warps read each stage's partials back (tcgen05.ld) and add
//    scale * partial into fp32 registers, so group scales are applied
//    exactly in fp32: apart from the order of fp32 additions the result is
//    the exact product sum (rounding the weights to bf16 instead would put
//    the largest output error near the 1e-2 * RMS parity bound);
//  * work is split stream-K style: the (tile, stage) units of the GEMM are
//    divided evenly over the persistent grid; a tile cut between CTAs is
//    summed with red.global.add into an fp32 slot and finished by the last
//    contributor to arrive (no CTA ever waits for another);
//  * launches overlap: the kernel is launched with programmatic stream
//    serialisation, lets the next kernel be scheduled at once, and waits for
//    the previous kernel only before it reads activations or writes outputs
//    and split-tile sums -- the weight stream (which no kernel writes) never
//    waits, so a CTA that starts on an SM freed by the previous GEMM fills
//    its ring with weights while that GEMM's last CTAs finish.
// Every wait is bounded (see ptx.cuh); a timeout records an error, drains the
// CTA's in-flight copies/MMAs and frees its tensor memory before returning.
// A test hook (spec_test_stall) shortens the limit and withholds one stage's
// weights from CTA 0 for one launch.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "internal.hpp"
#include "ptx.cuh"

namespace sv {
namespace {

constexpr int kTmemCols = 512;

template <int QUANT, int TPAD>
struct Cfg {
  static constexpr int kSub = QUANT == kW4 ? 4 : 2;             // 64-k groups per stage
  static constexpr int kStageKK = 64 * kSub;                    // k per stage
  static constexpr int kCodeBytes = kTileM * 128;               // 128 code bytes per row
  static constexpr int kXBoxBytes = TPAD * 128;                 // TPAD rows x 64 activations
  static constexpr int kXOff = 0;
  static constexpr int kCodeOff = kSub * kXBoxBytes;
  static constexpr int kScaleOff = kCodeOff + kCodeBytes;       // [SR][128] fp16
  static constexpr int kMaxSR = kSub;                           // scale rows per stage (g = 64)
  static constexpr int kZeroOff = kScaleOff + kMaxSR * kTileM * 2;   // [SR][64] bytes
  static constexpr int kStageBytes =
      (kZeroOff + (QUANT == kW4 ? kMaxSR * 64 : 0) + 1023) / 1024 * 1024;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kSmemBudget = 224 * 1024;
  static constexpr int kStagesFit = (kSmemBudget - kCtrlBytes - 1024) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kCtrlBytes;
  // warps: weight producer, dequant, MMA issue (one per 64-k group),
  // epilogue, activation producer
  static constexpr int kDqWarps = 8;                            // two per TMEM lane quadrant
  static constexpr int kGroupsPerDq = kSub / 2;                 // 64-k groups of a stage per dequant warp
  static constexpr int kMmaWarps = kSub;
  static constexpr int kDqWarp0 = 1;
  static constexpr int kMmaWarp0 = kDqWarp0 + kDqWarps;
  static constexpr int kEpWarp0 = kMmaWarp0 + kMmaWarps;
  static constexpr int kXWarp = kEpWarp0 + 4;
  static constexpr int kThreads = 32 * (kXWarp + 1);
  // TMEM: a ring of A slots (one stage each, 32 columns per group) and a ring
  // of partial sets (one stage each, TPAD columns per group).
  static constexpr int kACols = 32 * kSub;
  static constexpr int kDCols = TPAD * kSub;
  static constexpr int kNumDFit = (kTmemCols - 2 * kACols) / kDCols;
  static constexpr int kNumD = kNumDFit > 4 ? 4 : kNumDFit;
  static constexpr int kNumAFit = (kTmemCols - kNumD * kDCols) / kACols;
  static constexpr int kNumA = kNumAFit > 4 ? 4 : kNumAFit;
  static constexpr int kD0 = kNumA * kACols;
  // When the A ring is no deeper than the partial ring, the completion of
  // stage n's MMAs (the partial ring's "full" barrier) also frees stage n's A
  // slot, so the MMA warps commit one barrier per stage instead of two.
  static constexpr bool kAFromD = kNumA <= kNumD;
  static_assert(kStages >= 3, "pipeline too shallow");
  static_assert(kNumA >= 2 && kNumD >= 1, "TMEM rings too shallow");
  static_assert(kD0 + kNumD * kDCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert((3 * kStages + 2 * kNumA + 2 * kNumD) * 8 + 8 <= kCtrlBytes, "barrier block");
};

struct Params {
  int T, N, K;
  int group_size;      // 0 = per output channel
  int gshift;          // log2(group_size) (group_size is a power of two)
  int ks;              // stages per tile = ceil(K / stage k)
  int last_nsub;       // valid 64-k groups in a tile's last stage
  int gsh;             // row of group j in a stage's scale/zero box = (64 j) >> gsh
  int total;           // tiles * ks units (< 2^28)
  uint32_t tx_w;       // TMA bytes of a stage's codes, scales and zero points
  const uint16_t* scales;   // per-channel int8 scales (applied at the end of a segment)
  void* y;
  int y_f32;
  float* partials;     // split tiles: [first contributor CTA][TPAD][128] fp32, kept zeroed
  int* counters;       // per tile arrival counters, kept zeroed
  int* err;
  unsigned long long wait_ns;   // limit of every wait
  int skip_unit;       // test hook: CTA 0 never loads the weights of this unit (-1: none)
};

__device__ __forceinline__ int unit_begin(int c, int total, int G) {
  return (int)((long long)c * total / G);
}

__device__ __forceinline__ int cta_of_unit(int u, int total, int G) {
  int c = (int)((long long)u * G / total);
  while (c + 1 < G && unit_begin(c + 1, total, G) <= u) ++c;
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

// Walks a CTA's range of (tile, stage) units without per-unit division.
struct UnitIter {
  int tile, kst, ks;
  __device__ __forceinline__ UnitIter(int u, int ks_) : ks(ks_) {
    tile = u / ks_;
    kst = u - tile * ks_;
  }
  __device__ __forceinline__ void next() {
    if (++kst == ks) {
      kst = 0;
      ++tile;
    }
  }
};

// int4: 64 codes (group j of the row's 128-byte stage line) to exact bf16
// pairs (code - zero) in natural k order: a[i] holds k = 2i (low half) and
// 2i+1 (high half).  Code layout: nibble p (0..7, from the least significant
// end) of each little-endian 32-bit word holds k = 8w + 2*(p % 4) + p / 4, so
// the pairs (k0, k1), (k2, k3), (k4, k5), (k6, k7) sit at bit offsets 0, 4, 8
// and 12 of both 16-bit halves.  Shifted to offset 0 and merged under the
// bf16 exponent of 128, a nibble c becomes 128 + c exactly (bf16 keeps 7
// fraction bits); subtracting 128 + zero leaves the exact integer.
// The line was written by TMA with the 128-byte swizzle: 16-byte chunk c of
// row m sits at chunk position c ^ (m & 7).
__device__ __forceinline__ void load_w4(uint32_t row_addr, uint32_t m, int j, uint32_t (&words)[8]) {
  const uint32_t sw = m & 7u;
  const uint4 c0 = lds128(row_addr + (((2u * j) ^ sw) << 4));
  const uint4 c1 = lds128(row_addr + (((2u * j + 1u) ^ sw) << 4));
  words[0] = c0.x; words[1] = c0.y; words[2] = c0.z; words[3] = c0.w;
  words[4] = c1.x; words[5] = c1.y; words[6] = c1.z; words[7] = c1.w;
}

__device__ __forceinline__ void dequant_w4(const uint32_t (&words)[8], uint32_t z, uint32_t (&a)[32]) {
  const uint32_t zz = (0x4300u | z) * 0x00010001u;             // bf16x2 (128 + z)
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = words[w];
#pragma unroll
    for (int o = 0; o < 4; ++o)
      a[4 * w + o] = sub_bf16x2(lop3_and_or(q >> (4 * o), 0x000F000Fu, 0x43004300u), zz);
  }
}

// int8: 64 codes (group j of the row's 128-byte stage line, 128-byte swizzle
// as above) to exact bf16.  A biased byte b = code + 128 becomes the fp32
// 2^23 + b, minus 2^23 + 128 gives the code exactly, and |code| <= 127 fits
// bf16's 8-bit significand.
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

template <int QUANT, int TPAD>
__global__ void __launch_bounds__(Cfg<QUANT, TPAD>::kThreads, 1)
    qgemm_split_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_codes,
                 const __grid_constant__ CUtensorMap tm_scales,
                 const __grid_constant__ CUtensorMap tm_zeros, const Params p) {
  using C = Cfg<QUANT, TPAD>;
  constexpr int S = C::kStages, NA = C::kNumA, SUB = C::kSub, ND = C::kNumD;
  constexpr int kMmaWarps = C::kMmaWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ctrl = smem + S * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* a_full = empty + S;
  uint64_t* a_empty = a_full + NA;
  uint64_t* d_full = a_empty + NA;
  uint64_t* d_empty = d_full + ND;
  uint64_t* x_full = d_empty + ND;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x_full + S);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int begin = unit_begin(blockIdx.x, p.total, G);
  const int end = unit_begin(blockIdx.x + 1, p.total, G);
  const bool per_channel = (QUANT == kW8) && p.group_size == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&x_full[s], 1);
      // released by the dequant warps and by the epilogue warps once the
      // stage's MMAs have completed (they read the stage's scales)
      mbar_init(&empty[s], C::kDqWarps + 4);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&a_full[s], C::kDqWarps);
      mbar_init(&a_empty[s], kMmaWarps);
    }
    for (int b = 0; b < ND; ++b) {
      mbar_init(&d_full[b], kMmaWarps);
      mbar_init(&d_empty[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_codes);
      prefetch_tensormap(&tm_scales);
      if (QUANT == kW4) prefetch_tensormap(&tm_zeros);
    }
    __syncwarp();
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  pdl_launch_dependents();

  const int nunits = end - begin;
  // valid 64-k groups of stage kst (only a tile's last stage may be partial)
  auto nsub_of = [&](int kst) { return kst == p.ks - 1 ? p.last_nsub : SUB; };

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    // (the whole warp walks the ring; lane 0 issues the copies)
    const uint64_t pol_w = policy_evict_first();
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    int n = 0;
    for (; n < nunits; ++n, it.next(), st_ring.next()) {
      const int s = st_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], st_ring.phase ^ 1, abort_flag, p.err, p.wait_ns))) break;
      if (n == p.skip_unit && blockIdx.x == 0) continue;   // test hook: this stage's weights never arrive
      if (lane == 0) {
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], p.tx_w);
        tma_load_2d_hint(st + C::kCodeOff, &tm_codes, &full[s], it.kst * 128, it.tile * kTileM, pol_w);
        const int g0 = p.group_size ? (it.kst * C::kStageKK) >> p.gshift : 0;
        tma_load_2d(st + C::kScaleOff, &tm_scales, &full[s], it.tile * kTileM, g0);
        if (QUANT == kW4) tma_load_2d(st + C::kZeroOff, &tm_zeros, &full[s], it.tile * (kTileM / 2), g0);
      }
      __syncwarp();
    }
    if (*abort_flag && lane == 0) {
      // drain copies still in flight into this CTA's shared memory
      for (int j = (n > S ? n - S : 0); j < n; ++j) {
        volatile int no_abort = 0;
        mbar_wait(&full[j % S], (j / S) & 1, &no_abort, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp < C::kMmaWarp0) {
    // ------------------------------------------------------------ dequant
    const int dq = warp - C::kDqWarp0;
    const int q = warp & 3;                   // TMEM lane quadrant this warp may access
    const int j0 = (dq >> 2) * C::kGroupsPerDq;   // first 64-k group of a stage this warp handles
    const int m = q * 32 + lane;              // weight row inside the tile
    const uint32_t a_addr0 = tbase + ((uint32_t)(q * 32) << 16) + j0 * 32;
    const uint32_t row_off = C::kCodeOff + m * 128;
    const uint32_t zshift = (m & 1) * 4;
    uint32_t zero_off[C::kGroupsPerDq];
#pragma unroll
    for (int i = 0; i < C::kGroupsPerDq; ++i)
      zero_off[i] = C::kZeroOff + ((64 * (j0 + i)) >> p.gsh) * 64 + (m >> 1);
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    Ring<NA> a_ring;
    Ring<ND> dprev;   // partial slot of stage n - NA (whose MMAs free this stage's A slot)
    for (int n = 0; n < nunits; ++n, it.next(), st_ring.next(), a_ring.next()) {
      const int nsub = nsub_of(it.kst);
      const int s = st_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], st_ring.phase, abort_flag, p.err, p.wait_ns))) break;
      const uint8_t* st = smem + s * C::kStageBytes;
      const int sa = a_ring.slot;
      bool ok = true;
      // all of this stage's shared-memory reads first (one exposed latency),
      // then one group at a time: dequantise into registers, store to TMEM
      // (the first store waits for the A slot to be free; one wait for both)
      uint32_t words[C::kGroupsPerDq][8];
      uint32_t zb[C::kGroupsPerDq];
      if constexpr (QUANT == kW4) {
#pragma unroll
        for (int i = 0; i < C::kGroupsPerDq; ++i) {
          if (j0 + i < nsub) {
            load_w4(smem_u32(st) + row_off, m, j0 + i, words[i]);
            zb[i] = st[zero_off[i]];
          }
        }
      }
#pragma unroll
      for (int i = 0; i < C::kGroupsPerDq; ++i) {
        const int j = j0 + i;
        uint32_t a[32];
        if (j < nsub) {
          if constexpr (QUANT == kW4) {
            dequant_w4(words[i], (zb[i] >> zshift) & 0xFu, a);
          } else {
            dequant_w8(smem_u32(st) + row_off, m, j, a);
          }
        }
        if (i == 0) {
          if constexpr (C::kAFromD) {
            if (n >= NA) {
              ok = __all_sync(0xffffffffu, mbar_wait(&d_full[dprev.slot], dprev.phase, abort_flag, p.err, p.wait_ns));
              dprev.next();
            }
          } else {
            ok = __all_sync(0xffffffffu, mbar_wait(&a_empty[sa], a_ring.phase ^ 1, abort_flag, p.err, p.wait_ns));
          }
          if (!ok) break;
          tc_fence_after();
        }
        if (j < nsub) tmem_st_32x32b_x32(a_addr0 + sa * C::kACols + i * 32, a);
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[sa]);
        mbar_arrive(&empty[s]);
      }
    }
  } else if (warp < C::kEpWarp0) {
    // ------------------------------------------------------------ MMA issue
    // (the whole warp walks the rings; lane 0 issues the MMAs and commits)
    const int jg = warp - C::kMmaWarp0;       // the 64-k group of each stage this warp issues
    constexpr uint32_t idesc = idesc_bf16_f32(128, TPAD);
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    Ring<NA> a_ring;
    Ring<ND> d_ring;
    int last_sa = -1;
    uint32_t last_phase = 0;
    for (int n = 0; n < nunits; ++n, it.next(), st_ring.next(), a_ring.next(), d_ring.next()) {
      const int s = st_ring.slot, sa = a_ring.slot, b = d_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&d_empty[b], d_ring.phase ^ 1, abort_flag, p.err, p.wait_ns))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(&a_full[sa], a_ring.phase, abort_flag, p.err, p.wait_ns))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(&x_full[s], st_ring.phase, abort_flag, p.err, p.wait_ns))) break;
      tc_fence_after();
      if (lane == 0) {
        if (jg < nsub_of(it.kst)) {
          const uint32_t d_col = tbase + C::kD0 + b * C::kDCols + jg * TPAD;
          const uint32_t a_col = tbase + sa * C::kACols + jg * 32;
          const uint64_t bdesc =
              smem_desc_sw128(smem + s * C::kStageBytes + C::kXOff) + (uint64_t)((jg * C::kXBoxBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: 8 TMEM columns (16 bf16) per K16 step; B: +32 bytes inside the swizzled row.
            mma_ts(d_col, a_col + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, kk > 0 ? 1u : 0u);
          }
        }
        if constexpr (!C::kAFromD) mma_commit(&a_empty[sa]);
        mma_commit(&d_full[b]);
      }
      __syncwarp();
      last_sa = b;
      last_phase = d_ring.phase;
    }
    if (*abort_flag && last_sa >= 0 && lane == 0) {
      // wait for this warp's own MMAs before the CTA frees its tensor memory
      volatile int no_abort = 0;
      mbar_wait(&d_full[last_sa], last_phase, &no_abort, nullptr, kDrainLimitNs);
    }
  } else if (warp < C::kXWarp) {
    // ------------------------------------------------------------ epilogue
    // outputs and split-tile sums may be read or cleared by the previous kernel
    pdl_wait_prior();
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    constexpr int kW = TPAD < 32 ? TPAD : (TPAD > 32 ? 16 : 32);   // columns read per wait (register budget)

    float acc[TPAD];
#pragma unroll
    for (int t = 0; t < TPAD; ++t) acc[t] = 0.f;

    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    Ring<ND> d_ring;
    bool ok = true;
    int n = 0;
    while (ok && n < nunits) {
      const int tile = it.tile;
      const int tile_first = tile * p.ks;
      const int u0 = begin + n;
      const int seg_end = min(end, tile_first + p.ks);
      const bool whole_tile = (u0 == tile_first) && (seg_end == tile_first + p.ks);
      const int nrow = tile * kTileM + m;
      for (int u = u0; u < seg_end; ++u, ++n, it.next(), st_ring.next(), d_ring.next()) {
        const int nsub = nsub_of(it.kst);
        // this stage's group scales (fp32, exact), read while its slot is still held
        const int s = st_ring.slot;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], st_ring.phase, abort_flag, p.err, p.wait_ns));
        if (!ok) break;
        float sc[SUB];
        {
          const __half* srow = reinterpret_cast<const __half*>(smem + s * C::kStageBytes + C::kScaleOff) + m;
#pragma unroll
          for (int j = 0; j < SUB; ++j)
            sc[j] = per_channel ? 1.f : __half2float(srow[((64 * j) >> p.gsh) * kTileM]);
        }
        // this stage's partials; once they are complete the stage's MMAs have
        // finished reading its activations, so the slot can be released
        const int b = d_ring.slot;
        ok = __all_sync(0xffffffffu, mbar_wait(&d_full[b], d_ring.phase, abort_flag, p.err, p.wait_ns));
        if (!ok) break;
        if (lane == 0) mbar_arrive(&empty[s]);
        tc_fence_after();
        const uint32_t dbase = tbase + lane_base + C::kD0 + b * C::kDCols;
#pragma unroll
        for (int j = 0; j < SUB; ++j) {
          if (j < nsub) {
            const uint64_t s2 = pack_f32x2(__float_as_uint(sc[j]), __float_as_uint(sc[j]));
#pragma unroll
            for (int c0 = 0; c0 < TPAD; c0 += kW) {
              uint32_t r[kW];
#pragma unroll
              for (int h = 0; h < kW / 16; ++h)
                tmem_ld_32x32b_x16(dbase + j * TPAD + c0 + h * 16, *reinterpret_cast<uint32_t(*)[16]>(&r[h * 16]));
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < kW; c += 2) {
                // columns (t, t + 1) in one fma.rn.f32x2
                const uint64_t d = fma_f32x2(s2, pack_f32x2(r[c], r[c + 1]),
                                             pack_f32x2(__float_as_uint(acc[c0 + c]), __float_as_uint(acc[c0 + c + 1])));
                acc[c0 + c] = __uint_as_float((uint32_t)d);
                acc[c0 + c + 1] = __uint_as_float((uint32_t)(d >> 32));
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[b]);
      }
      if (!ok) break;

      float v[TPAD];
      const float osc = per_channel && nrow < p.N ? __half2float(__ushort_as_half(p.scales[nrow])) : 1.f;
#pragma unroll
      for (int t = 0; t < TPAD; ++t) {
        v[t] = acc[t] * osc;
        acc[t] = 0.f;
      }
      if (whole_tile) {
        if (nrow < p.N) {
#pragma unroll
          for (int t = 0; t < TPAD; ++t) {
            if (t < p.T) {
              if (p.y_f32)
                reinterpret_cast<float*>(p.y)[(size_t)t * p.N + nrow] = v[t];
              else
                reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)t * p.N + nrow] = __float2bfloat16_rn(v[t]);
            }
          }
        }
      } else {
        // Split tile: add this warp's 32 rows of the CTA's partial into the
        // tile's fp32 slot (keyed by the tile's first contributor, unique per
        // split tile).  Arrivals are counted per lane quadrant, so each warp
        // finishes its own rows: the last to arrive converts the sum and
        // clears the slot, with no barrier between the epilogue warps.
        const int c_first = cta_of_unit(tile_first, p.total, G);
        const int c_last = cta_of_unit(tile_first + p.ks - 1, p.total, G);
        // slot layout [128 rows][TPAD]: a thread's values are contiguous, so
        // the sums travel as 16-byte vector reductions and loads
        float* slot = p.partials + (size_t)c_first * kPartialSlotFloats + (size_t)m * TPAD;
#pragma unroll
        for (int t = 0; t < TPAD; t += 4)
          if (t < p.T) red_add_f32x4(slot + t, v[t], v[t + 1], v[t + 2], v[t + 3]);
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomic_add_acq_rel_gpu(&p.counters[tile * 4 + q], 1) == c_last - c_first;
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();   // orders lane 0's acquire before the other lanes' reads
        if (last) {
          // every read before any store (one L2 round trip for T <= 32): the
          // stores may alias the slot as far as the compiler knows
          constexpr int kB = TPAD % 32 == 0 ? 32 : 16;
#pragma unroll
          for (int h = 0; h < TPAD / kB; ++h) {
            float4 w[kB / 4];
#pragma unroll
            for (int c = 0; c < kB / 4; ++c)
              w[c] = (h * kB + 4 * c < p.T) ? ldcg_f32x4(slot + h * kB + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kB / 4; ++c) {
              const int t0 = h * kB + 4 * c;
              if (t0 < p.T) {
                __stcg(reinterpret_cast<float4*>(slot + t0), make_float4(0.f, 0.f, 0.f, 0.f));
                const float wv[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int t = t0 + e;
                  if (t < p.T && nrow < p.N) {
                    if (p.y_f32)
                      reinterpret_cast<float*>(p.y)[(size_t)t * p.N + nrow] = wv[e];
                    else
                      reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)t * p.N + nrow] = __float2bfloat16_rn(wv[e]);
                  }
                }
              }
            }
          }
          // only this warp touches the counter until the kernel ends
          if (lane == 0) __stcg(&p.counters[tile * 4 + q], 0);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ activation producer
    // (the activations may be written by the previous kernel; a slot is
    // refilled once the epilogue has seen that stage's MMAs complete)
    pdl_wait_prior();
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    int n = 0;
    for (; n < nunits; ++n, it.next(), st_ring.next()) {
      const int s = st_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], st_ring.phase ^ 1, abort_flag, p.err, p.wait_ns))) break;
      if (lane == 0) {
        const int nsub = nsub_of(it.kst);
        uint8_t* st = smem + s * C::kStageBytes + C::kXOff;
        mbar_arrive_expect_tx(&x_full[s], (uint32_t)(nsub * C::kXBoxBytes));
        for (int j = 0; j < nsub; ++j)
          tma_load_2d(st + j * C::kXBoxBytes, &tm_x, &x_full[s], it.kst * C::kStageKK + 64 * j, 0);
      }
      __syncwarp();
    }
    if (*abort_flag && lane == 0) {
      for (int j = (n > S ? n - S : 0); j < n; ++j) {
        volatile int no_abort = 0;
        mbar_wait(&x_full[j % S], (j / S) & 1, &no_abort, nullptr, kDrainLimitNs);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int QUANT, int TPAD>
int launch_t(spec_ctx* ctx, const GemmArgs& a, cudaStream_t stream) {
  using C = Cfg<QUANT, TPAD>;
  CUtensorMap tx, tc, ts, tz;
  int rc;
  rc = encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.T,
                      (uint64_t)a.K * 2, kGroupK, TPAD, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t row_bytes = QUANT == kW4 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
  rc = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qcodes, row_bytes, (uint64_t)a.N,
                      row_bytes, 128, kTileM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t groups = a.group_size ? (uint64_t)(a.K / a.group_size) : 1;
  const int sr = a.group_size && a.group_size < C::kStageKK ? C::kStageKK / a.group_size : 1;
  rc = encode_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)a.N, groups,
                      (uint64_t)a.N * 2, kTileM, sr, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc) return rc;
  if (QUANT == kW4) {
    rc = encode_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.zeros, (uint64_t)a.N / 2, groups,
                        (uint64_t)a.N / 2, kTileM / 2, sr, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  } else {
    tz = ts;
  }

  Params p;
  p.T = a.T;
  p.N = a.N;
  p.K = a.K;
  p.group_size = a.group_size;
  p.gshift = 0;
  while (a.group_size && (1 << p.gshift) < a.group_size) ++p.gshift;
  p.ks = (a.K + C::kStageKK - 1) / C::kStageKK;
  p.last_nsub = (a.K - (p.ks - 1) * C::kStageKK) / 64;
  p.gsh = (a.group_size == 0 || a.group_size > C::kStageKK) ? 31 : p.gshift;
  const long long tiles = (a.N + kTileM - 1) / kTileM;
  p.total = tiles * p.ks;
  p.tx_w = C::kCodeBytes + sr * kTileM * 2 + (QUANT == kW4 ? sr * 64 : 0);
  p.scales = a.scales;
  p.y = a.y;
  p.y_f32 = a.y_f32;
  p.partials = ctx->split_partials;
  p.counters = ctx->tile_counters;
  p.err = ctx->err;
  p.wait_ns = ctx->test_wait_ns ? ctx->test_wait_ns : kWaitLimitNs;
  p.skip_unit = ctx->test_skip_unit;
  ctx->test_wait_ns = 0;
  ctx->test_skip_unit = -1;
  // persistent grid of one CTA per SM with an even share of units each
  long long G = ctx->num_sms;
  if (G > p.total) G = p.total;
  const long long per = (p.total + G - 1) / G;
  G = (p.total + per - 1) / per;
  if (G > ctx->max_slots) return set_error(SPEC_ERR_OOM, "workspace has too few partial slots");

  static std::atomic<uint32_t> attr_done{0};   // per instantiation, one bit per device
  const uint32_t bit = ctx->device < 32 ? (1u << ctx->device) : 0u;
  if (!bit || !(attr_done.load() & bit)) {
    rc = check_cuda(cudaFuncSetAttribute(qgemm_split_kernel<QUANT, TPAD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes),
                    "cudaFuncSetAttribute(qgemm)");
    if (rc) return rc;
    attr_done.fetch_or(bit);
  }
  // programmatic stream serialisation: see the design notes at the top
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
  return check_cuda(cudaLaunchKernelEx(&cfg, qgemm_split_kernel<QUANT, TPAD>, tx, tc, ts, tz, p), "qgemm_split launch");
}

template <int QUANT>
int launch_q(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s) {
  const int tpad = (a.T + 15) / 16 * 16;
  switch (tpad) {
    case 16: return launch_t<QUANT, 16>(ctx, a, s);
    case 32: return launch_t<QUANT, 32>(ctx, a, s);
    case 48: return launch_t<QUANT, 48>(ctx, a, s);
    case 64: return launch_t<QUANT, 64>(ctx, a, s);
    default: return set_error(SPEC_ERR_SHAPE, "T=%d outside 1..64", a.T);
  }
}

}  // namespace

int launch_qgemm_split(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s) {
  return a.quant == kW4 ? launch_q<kW4>(ctx, a, s) : launch_q<kW8>(ctx, a, s);
}

}  // namespace sv
