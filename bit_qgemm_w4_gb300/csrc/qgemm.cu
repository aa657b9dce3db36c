// Verify GEMM for the speculative-decoding verification step: low-bit weights
// times the T drafted positions' activations, on the sm_103a tensor cores.
//
// What it computes ("Karpathy's Trick for Faster Local LLMs Finally Has Proper
// Tooling", section "How Uzu optimizes bytes and tokens per pass": 4-bit
// asymmetric Medium tier, 8-bit symmetric Large tier, one scale per group):
//   y[t][n] = sum_k x[t][k] * (code[n][k] - zero[g][n]) * scale[g][n]   (int4)
//   y[t][n] = sum_k x[t][k] *  code[n][k]              * scale[g][n]   (int8)
//
// Design (swap-AB, weight rows are the MMA's M dimension, the T drafted
// positions its N dimension):
//  * one pipeline stage = 128 weight rows x 64 k.  A TMA warp streams the
//    packed codes (swizzled so that each row's bytes are bank-conflict free),
//    the group's scales/zeros and the 64-wide activation slice into a ring of
//    shared-memory stages;
//  * four dequantisation warps (one per TMEM lane quadrant, one weight row per
//    thread) turn a row's 64 codes into exact bf16 integers (code - zero, or
//    the int8 code) and write them straight into tensor memory with
//    tcgen05.st -- the MMA's A operand lives in TMEM, so the dequantised tile
//    never touches shared memory;
//  * one thread issues tcgen05.mma (A from TMEM, B = activations from shared
//    memory, D = fp32 in TMEM), 4 x K16 per stage, into a per-stage partial
//    accumulator;
//  * the same dequantisation warps read each stage's partial back
//    (tcgen05.ld) and add scale * partial into fp32 registers, so group scales
//    are applied exactly in fp32 (no bf16 rounding of the weights at all);
//  * work is split stream-K style: the (tile, stage) units of the whole GEMM
//    are divided evenly over a persistent grid of two CTAs per SM; a tile cut
//    between CTAs is finished by the last CTA to arrive (deterministic sum of
//    per-CTA fp32 partials in CTA order, no spin-waiting on other CTAs).
// Every wait is bounded (see ptx.cuh); a timeout records an error, drains the
// CTA's in-flight copies/MMAs and frees its tensor memory before returning.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "internal.hpp"
#include "ptx.cuh"

namespace sv {
namespace {

// Roles: warp 0 owns TMEM and streams stages with TMA; then 4*kSG dequant
// warps (one per TMEM lane quadrant and k group of a step); then kSG MMA
// warps (warp j issues the MMAs of k group j -- several issuing warps keep
// the tensor core fed, a single one cannot with small-N MMAs); then four
// epilogue warps (one per quadrant) that fold the group partials into fp32
// accumulators and write the output.  One CTA per SM owns all of TMEM.
constexpr int kTmemCols = 512;

template <int QUANT, int TPAD>
struct Cfg {
  // One pipeline stage streams 128 contiguous code bytes of each of the 128
  // weight rows (full-width HBM bursts): 256 k for int4, 128 k for int8.
  // Within a stage, work is handed between roles in steps of kSG groups of
  // 64 k; each 64-k group gets its own fp32 partial so its scale can be
  // applied exactly.
  static constexpr int kSub = QUANT == kW4 ? 4 : 2;             // 64-k groups per stage
  static constexpr int kStageKK = 64 * kSub;                    // k per stage
  static constexpr int kSG = (QUANT == kW4 && TPAD <= 32) ? 4 : 2;   // 64-k groups per step
  static constexpr int kSteps = kSub / kSG;                     // steps per stage
  static constexpr int kCodeBytes = kTileM * 128;
  static constexpr int kXBoxBytes = TPAD * 128;                 // TPAD rows x 64 bf16
  static constexpr int kXOff = 0;
  static constexpr int kCodeOff = kSub * kXBoxBytes;
  static constexpr int kScaleOff = kCodeOff + kCodeBytes;       // [SR][128] fp16
  static constexpr int kMaxSR = kSub;                           // scale rows per stage (g = 64)
  static constexpr int kZeroOff = kScaleOff + kMaxSR * kTileM * 2;   // [SR][64] bytes
  static constexpr int kStageBytes = (kZeroOff + kMaxSR * 64 + 1023) / 1024 * 1024;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kSmemBudget = 224 * 1024;
  static constexpr int kStagesFit = (kSmemBudget - kCtrlBytes - 1024) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kACols = 32 * kSG;                       // one A slot: a step's groups
  static constexpr int kPCols = TPAD * kSG;                     // one P slot: a step's partials
  static constexpr int kNumA = 2, kNumP = 2;
  static constexpr int kPCols0 = kNumA * kACols;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kCtrlBytes;
  static constexpr int kDqWarps = 4 * kSG;
  static constexpr int kDqWarp0 = 1;
  static constexpr int kMmaWarp0 = kDqWarp0 + kDqWarps;
  static constexpr int kEpWarp0 = kMmaWarp0 + kSG;
  static constexpr int kThreads = 32 * (kEpWarp0 + 4);
  static_assert(kStages >= 3, "pipeline too shallow");
  static_assert(kPCols0 + kNumP * kPCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Params {
  int T, N, K;
  int group_size;      // 0 = per output channel
  int gshift;          // log2(group_size) (group_size is a power of two)
  int ks;              // stages per tile = ceil(K / stage k)
  int sr;              // scale/zero rows per stage box
  long long total;     // tiles * ks units
  uint32_t tx;         // TMA bytes per full stage
  void* y;
  int y_f32;
  float* partials;     // split tiles: [first contributor CTA][TPAD][128] fp32, kept zeroed
  int* counters;       // per tile arrival counters, kept zeroed
  int* err;
};

__device__ __forceinline__ long long unit_begin(int c, long long total, int G) {
  return (long long)c * total / G;
}

__device__ __forceinline__ int cta_of_unit(long long u, long long total, int G) {
  long long c = u * G / total;
  while (c + 1 < G && unit_begin((int)c + 1, total, G) <= u) ++c;
  while (c > 0 && unit_begin((int)c, total, G) > u) --c;
  return (int)c;
}

// int4: one thread dequantises 64 codes (sub-step j of its row's 128-byte
// stage line) to bf16 pairs of (code - zero) in natural k order: a[i] holds
// k = 2i (low half) and 2i+1 (high half).  Storage: byte b of each 4-byte
// word holds k = 8w+b in its low nibble and k = 8w+b+4 in its high nibble.
// The line was written by TMA with the 128-byte swizzle: 16-byte chunk c of
// row m sits at chunk position c ^ (m & 7).
__device__ __forceinline__ void dequant_sub_w4(uint32_t row_addr, uint32_t m, int j, uint32_t z,
                                               uint32_t (&a)[32]) {
  const uint32_t sw = m & 7u;
  const uint4 c0 = lds128(row_addr + (((2u * j) ^ sw) << 4));
  const uint4 c1 = lds128(row_addr + (((2u * j + 1u) ^ sw) << 4));
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const uint32_t zz = (0x4300u | z) * 0x00010001u;     // bf16x2 (128 + z, 128 + z)
  const uint32_t magic = 0x43434343u;                  // high byte of bf16 128.0
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t lo = words[w] & 0x0F0F0F0Fu;         // bytes: k0 k1 k2 k3
    const uint32_t hi = (words[w] >> 4) & 0x0F0F0F0Fu;  // bytes: k4 k5 k6 k7
    // bf16x2 (128 + c_a, 128 + c_b) = bytes {c_a, 0x43, c_b, 0x43}
    a[4 * w + 0] = sub_bf16x2(__byte_perm(lo, magic, 0x4140u), zz);
    a[4 * w + 1] = sub_bf16x2(__byte_perm(lo, magic, 0x4342u), zz);
    a[4 * w + 2] = sub_bf16x2(__byte_perm(hi, magic, 0x4140u), zz);
    a[4 * w + 3] = sub_bf16x2(__byte_perm(hi, magic, 0x4342u), zz);
  }
}

// int8: one thread converts 64 codes (sub-step j of its row's 128-byte stage
// line, 128-byte swizzle as above) to exact bf16.
__device__ __forceinline__ void dequant_sub_w8(uint32_t row_addr, uint32_t m, int j,
                                               uint32_t (&a)[32]) {
  const uint32_t sw = m & 7u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = lds128(row_addr + (((uint32_t)(4 * j + c) ^ sw) << 4));
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t u = words[w] ^ 0x80808080u;       // biased bytes code + 128
      float f[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // fp32 2^23 + byte, minus 2^23 + 128 = code, exactly
        f[b] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u | b)) - 8388736.0f;
      }
      a[8 * c + 2 * w] = pack_bf16x2(f[0], f[1]);
      a[8 * c + 2 * w + 1] = pack_bf16x2(f[2], f[3]);
    }
  }
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
  __device__ __forceinline__ UnitIter(long long u, int ks_) : ks(ks_) {
    tile = (int)(u / ks_);
    kst = (int)(u - (long long)tile * ks_);
  }
  __device__ __forceinline__ void next() {
    if (++kst == ks) {
      kst = 0;
      ++tile;
    }
  }
};

template <int QUANT, int TPAD>
__global__ void __launch_bounds__(Cfg<QUANT, TPAD>::kThreads, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_codes,
                 const __grid_constant__ CUtensorMap tm_scales,
                 const __grid_constant__ CUtensorMap tm_zeros, const Params p) {
  using C = Cfg<QUANT, TPAD>;
  constexpr int S = C::kStages, NA = C::kNumA, NP = C::kNumP, SUB = C::kSub, SG = C::kSG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ctrl = smem + S * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* a_full = empty + S;
  uint64_t* a_empty = a_full + NA;
  uint64_t* p_full = a_empty + NA;
  uint64_t* p_empty = p_full + NP;
  uint64_t* wg_bar = p_empty + NP;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wg_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* fix_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const long long begin = unit_begin(blockIdx.x, p.total, G);
  const long long end = unit_begin(blockIdx.x + 1, p.total, G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kDqWarps + SG + 4);   // dequant warps, MMA commits, epilogue warps
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&a_full[s], C::kDqWarps);
      mbar_init(&a_empty[s], SG);
    }
    for (int s = 0; s < NP; ++s) {
      mbar_init(&p_full[s], SG);
      mbar_init(&p_empty[s], 4);
    }
    mbar_init(wg_bar, 4);
    *abort_flag = 0;
    *fix_flag = 0;
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

  const long long nunits = end - begin;
  // valid 64-k groups of stage kst (the last stage of a row may be partial)
  // and the scale/zero row of group jg inside the stage's box
  auto nsub_of = [&](int kst) { return min(SUB, (p.K - kst * C::kStageKK) >> 6); };
  auto grow_of = [&](int kst, int jg) {
    return p.group_size ? (((kst * C::kStageKK + 64 * jg) >> p.gshift) - ((kst * C::kStageKK) >> p.gshift))
                        : 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      UnitIter it(begin, p.ks);
      Ring<S> st_ring;
      long long n = 0;
      for (; n < nunits; ++n, it.next(), st_ring.next()) {
        const int nsub = nsub_of(it.kst);
        const int s = st_ring.slot;
        if (!mbar_wait(&empty[s], st_ring.phase ^ 1, abort_flag, p.err)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], p.tx - (SUB - nsub) * C::kXBoxBytes);
        tma_load_2d_hint(st + C::kCodeOff, &tm_codes, &full[s], it.kst * 128, it.tile * kTileM, pol_w);
        const int g0 = p.group_size ? (it.kst * C::kStageKK) >> p.gshift : 0;
        tma_load_2d(st + C::kScaleOff, &tm_scales, &full[s], it.tile * kTileM, g0);
        if (QUANT == kW4) tma_load_2d(st + C::kZeroOff, &tm_zeros, &full[s], it.tile * (kTileM / 2), g0);
        for (int j = 0; j < nsub; ++j)
          tma_load_2d(st + C::kXOff + j * C::kXBoxBytes, &tm_x, &full[s],
                      it.kst * C::kStageKK + 64 * j, 0);
      }
      if (*abort_flag) {
        // drain copies still in flight into this CTA's shared memory
        const int issued = (int)n;
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j) {
          volatile int no_abort = 0;
          mbar_wait(&full[j % S], (j / S) & 1, &no_abort, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp < C::kMmaWarp0) {
    // ------------------------------------------------------------ dequant
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int jj = (warp - C::kDqWarp0) >> 2;     // k group of each step this warp handles
    const int m = q * 32 + lane;                  // weight row inside the tile
    const uint32_t a_addr0 = tbase + ((uint32_t)(q * 32) << 16) + jj * 32;
    const uint32_t zshift = (m & 1) * 4;
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    Ring<NA> a_ring;
    bool ok = true;
    for (long long n = 0; ok && n < nunits; ++n, it.next(), st_ring.next()) {
      const int nsub = nsub_of(it.kst);
      const int s = st_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], st_ring.phase, abort_flag, p.err))) break;
      const uint8_t* st = smem + s * C::kStageBytes;
      const uint32_t row_addr = smem_u32(st + C::kCodeOff) + m * 128;
      for (int ls = 0; ls * SG < nsub; ++ls, a_ring.next()) {
        const int jg = ls * SG + jj;              // group inside the stage
        uint32_t a[32];
        if (jg < nsub) {
          if constexpr (QUANT == kW4) {
            const uint32_t zb = st[C::kZeroOff + grow_of(it.kst, jg) * 64 + (m >> 1)];
            dequant_sub_w4(row_addr, m, jg, (zb >> zshift) & 0xFu, a);
          } else {
            dequant_sub_w8(row_addr, m, jg, a);
          }
        }
        const int sa = a_ring.slot;
        if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[sa], a_ring.phase ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        if (jg < nsub) {
          tc_fence_after();
          tmem_st_32x32b_x32(a_addr0 + sa * C::kACols, a);
          tmem_wait_st();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&empty[s]);
    }
  } else if (warp < C::kEpWarp0) {
    // ------------------------------------------------------------ MMA issue (k group jj)
    if (lane == 0) {
      const int jj = warp - C::kMmaWarp0;
      constexpr uint32_t idesc = idesc_bf16_f32(128, TPAD);
      UnitIter it(begin, p.ks);
      Ring<S> st_ring;
      Ring<NA> a_ring;
      Ring<NP> p_ring;
      bool ok = true, issued_any = false;
      int last_sp = 0;
      uint32_t last_phase = 0;
      for (long long n = 0; ok && n < nunits; ++n, it.next(), st_ring.next()) {
        const int nsub = nsub_of(it.kst);
        const int s = st_ring.slot;
        if (!mbar_wait(&full[s], st_ring.phase, abort_flag, p.err)) break;
        const uint64_t bdesc0 = smem_desc_sw128(smem + s * C::kStageBytes + C::kXOff);
        for (int ls = 0; ls * SG < nsub; ++ls, a_ring.next(), p_ring.next()) {
          const int sa = a_ring.slot, sp = p_ring.slot;
          if (!mbar_wait(&a_full[sa], a_ring.phase, abort_flag, p.err) ||
              !mbar_wait(&p_empty[sp], p_ring.phase ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int jg = ls * SG + jj;
          if (jg < nsub) {
            const uint32_t a_col = tbase + sa * C::kACols + jj * 32;
            const uint32_t d_col = tbase + C::kPCols0 + sp * C::kPCols + jj * TPAD;
            const uint64_t bdesc = bdesc0 + (uint64_t)((jg * C::kXBoxBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // A: 8 TMEM columns (16 bf16) per K16 step; B: +32 bytes inside the swizzled row
              mma_ts(d_col, a_col + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&a_empty[sa]);
          mma_commit(&p_full[sp]);
          issued_any = true;
          last_sp = sp;
          last_phase = p_ring.phase;
        }
        if (!ok) break;
        // the stage's shared memory may be reused once these MMAs are done
        mma_commit(&empty[s]);
      }
      if (*abort_flag && issued_any) {
        // wait for this thread's own MMAs before the CTA frees its tensor memory
        volatile int no_abort = 0;
        mbar_wait(&p_full[last_sp], last_phase, &no_abort, nullptr, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t wg_phase = 0;
    auto wg_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(wg_bar);
      const bool ok = mbar_wait(wg_bar, wg_phase, abort_flag, p.err);
      wg_phase ^= 1;
      return __all_sync(0xffffffffu, ok);
    };

    float acc[TPAD];
#pragma unroll
    for (int t = 0; t < TPAD; ++t) acc[t] = 0.f;
    bool ok = true;
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    Ring<NP> p_ring;
    long long n = 0;
    while (ok && n < nunits) {
      const int tile = it.tile;
      const long long tile_first = (long long)tile * p.ks;
      const long long u0 = begin + n;
      const long long seg_end = min(end, tile_first + p.ks);
      const bool whole_tile = (u0 == tile_first) && (seg_end == tile_first + p.ks);
      for (long long u = u0; u < seg_end; ++u, ++n, it.next(), st_ring.next()) {
        const int kst = it.kst;
        const int nsub = nsub_of(kst);
        const int s = st_ring.slot;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], st_ring.phase, abort_flag, p.err));
        if (!ok) break;
        float sc[SUB];
        {
          const __half* srow = reinterpret_cast<const __half*>(smem + s * C::kStageBytes + C::kScaleOff);
#pragma unroll
          for (int j = 0; j < SUB; ++j)
            sc[j] = (j < nsub) ? __half2float(srow[grow_of(kst, j) * kTileM + m]) : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
        for (int ls = 0; ls < C::kSteps; ++ls) {
          if (ls * SG >= nsub) break;
          const int sp = p_ring.slot;
          ok = __all_sync(0xffffffffu, mbar_wait(&p_full[sp], p_ring.phase, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < SG; ++jj) {
            const int jg = ls * SG + jj;
            if (jg < nsub) {
              const uint32_t d_addr = tbase + lane_base + C::kPCols0 + sp * C::kPCols + jj * TPAD;
              const float scj = sc[jg < SUB ? jg : 0];
#pragma unroll
              for (int h = 0; h < TPAD / 16; ++h) {
                uint32_t rr[16];
                tmem_ld_32x32b_x16(d_addr + h * 16, rr);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; c += 2)
                  fma_f32x2(acc[h * 16 + c], acc[h * 16 + c + 1], scj, __uint_as_float(rr[c]),
                            __uint_as_float(rr[c + 1]));
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_empty[sp]);
          p_ring.next();
        }
        if (!ok) break;
      }
      if (!ok) break;

      // ---- segment epilogue
      const int nrow = tile * kTileM + m;
      bool store = whole_tile;
      if (!whole_tile) {
        // Split tile: add this CTA's partial into the tile's fp32 slot (keyed
        // by the tile's first contributor, unique per split tile); the last
        // contributor to arrive converts the sum and clears the slot.
        const int c_first = cta_of_unit(tile_first, p.total, G);
        const int c_last = cta_of_unit(tile_first + p.ks - 1, p.total, G);
        float* slot = p.partials + (size_t)c_first * kPartialSlotFloats;
#pragma unroll
        for (int t = 0; t < TPAD; ++t) red_add_f32(slot + t * kTileM + m, acc[t]);
        __threadfence();
        ok = wg_sync();
        if (!ok) break;
        if (q == 0 && lane == 0) {
          const int old = atomicAdd(&p.counters[tile], 1);
          *fix_flag = (old == c_last - c_first) ? 1 : 0;
        }
        ok = wg_sync();
        if (!ok) break;
        store = *fix_flag != 0;
        if (store) {
          __threadfence();
#pragma unroll
          for (int t = 0; t < TPAD; ++t) {
            acc[t] = __ldcg(slot + t * kTileM + m);
            __stcg(slot + t * kTileM + m, 0.f);
          }
          if (q == 0 && lane == 0) atomicExch(&p.counters[tile], 0);
        }
        // keep fix_flag stable until every warp has read it
        ok = wg_sync();
        if (!ok) break;
      }
      if (store && nrow < p.N) {
        if (p.y_f32) {
          float* y = reinterpret_cast<float*>(p.y);
#pragma unroll
          for (int t = 0; t < TPAD; ++t)
            if (t < p.T) y[(size_t)t * p.N + nrow] = acc[t];
        } else {
          __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
#pragma unroll
          for (int t = 0; t < TPAD; ++t)
            if (t < p.T) y[(size_t)t * p.N + nrow] = __float2bfloat16_rn(acc[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < TPAD; ++t) acc[t] = 0.f;
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
                      (uint64_t)a.K * 2, kStageK, TPAD, CU_TENSOR_MAP_SWIZZLE_128B);
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
  p.sr = sr;
  const long long tiles = (a.N + kTileM - 1) / kTileM;
  p.total = tiles * p.ks;
  p.tx = C::kSub * C::kXBoxBytes + C::kCodeBytes + sr * kTileM * 2 + (QUANT == kW4 ? sr * 64 : 0);
  p.y = a.y;
  p.y_f32 = a.y_f32;
  p.partials = ctx->partials;
  p.counters = ctx->tile_counters;
  p.err = ctx->err;
  // persistent grid of one CTA per SM with an even share of units each
  long long G = ctx->num_sms;
  if (G > p.total) G = p.total;
  const long long per = (p.total + G - 1) / G;
  G = (p.total + per - 1) / per;
  if (G > ctx->max_slots) return set_error(SPEC_ERR_OOM, "workspace has too few partial slots");

  static std::atomic<uint32_t> attr_done{0};   // per instantiation, one bit per device
  const uint32_t bit = ctx->device < 32 ? (1u << ctx->device) : 0u;
  if (!bit || !(attr_done.load() & bit)) {
    rc = check_cuda(cudaFuncSetAttribute(qgemm_kernel<QUANT, TPAD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes),
                    "cudaFuncSetAttribute(qgemm)");
    if (rc) return rc;
    attr_done.fetch_or(bit);
  }
  qgemm_kernel<QUANT, TPAD><<<(unsigned)G, C::kThreads, C::kSmemBytes, stream>>>(tx, tc, ts, tz, p);
  return check_cuda(cudaGetLastError(), "qgemm launch");
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

int launch_qgemm(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s) {
  return a.quant == kW4 ? launch_q<kW4>(ctx, a, s) : launch_q<kW8>(ctx, a, s);
}

}  // namespace sv
