// Verify GEMM for the speculative-decoding verification step: low-bit weights
// times the T drafted positions' activations, on the sm_103a tensor cores.
//
// What it computes ("Karpathy's Trick for Faster Local LLMs Finally Has Proper
// Tooling", section "How Uzu optimizes bytes and tokens per pass": 4-bit
// asymmetric Medium tier, 8-bit symmetric Large tier, one scale per group):
//   y[t][n] = sum_k x[t][k] * (code[n][k] - zero[g][n]) * scale[g][n]   (int4)
//   y[t][n] = sum_k x[t][k] *  code[n][k]              * scale         (int8)
//
// Design (swap-AB: 128 weight rows are the MMA's M dimension, the T drafted
// positions its N dimension; one CTA per SM owns all 512 TMEM columns):
//  * a TMA warp streams stages into a shared-memory ring: per stage the
//    128-byte line of codes of each of the 128 weight rows (256 k of int4 or
//    128 k of int8 -- full-width HBM bursts), the stage's scale and zero
//    rows, and the stage's activation boxes (bf16);
//  * dequantisation warps, one per (TMEM lane quadrant, 64-k group), turn a
//    row's 64 codes into fp16 weights, (code - zero) * scale rounded once
//    (relative error <= 2^-11), and write them straight into a TMEM ring
//    with tcgen05.st -- the MMA's A operand lives in TMEM, so dequantised
//    weights never touch shared memory.  The same warps convert the stage's
//    activations to fp16 in place (exact inside the fp16 range; a value
//    outside it records an error);
//  * one MMA warp per 64-k group (several issuing warps are needed to keep
//    the tensor core fed with small-N MMAs) accumulates D += A * B in fp32
//    across the whole tile segment into its own TMEM accumulator (double
//    buffered when TMEM allows);
//  * four epilogue warps sum the accumulators at the end of a segment
//    (times the per-channel scale for int8 without groups, which stays exact
//    in fp32), clear them and write the output;
//  * work is split stream-K style: the (tile, stage) units of the GEMM are
//    divided evenly over the persistent grid; a tile cut between CTAs is
//    summed with red.global.add into an fp32 slot and finished by the last
//    contributor to arrive (no CTA ever waits for another).
// Every wait is bounded (see ptx.cuh); a timeout records an error, drains the
// CTA's in-flight copies/MMAs and frees its tensor memory before returning.

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
  static constexpr int kStageBytes = (kZeroOff + kMaxSR * 64 + 1023) / 1024 * 1024;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kSmemBudget = 224 * 1024;
  static constexpr int kStagesFit = (kSmemBudget - kCtrlBytes - 1024) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kCtrlBytes;
  // One MMA-issuing warp per 64-k group of a stage.  TMEM: a ring of A slots
  // (one stage each, 32 columns per group) and one or two accumulator
  // buffers, each holding one TPAD-column D per MMA warp.
  static constexpr int kMmaWarps = kSub;
  static constexpr int kACols = 32 * kSub;
  static constexpr int kDCols = TPAD * kMmaWarps;
  static constexpr int kDBufs = (2 * kDCols + 3 * kACols <= kTmemCols) ? 2 : 1;
  static constexpr int kNumAFit = (kTmemCols - kDBufs * kDCols) / kACols;
  static constexpr int kNumA = kNumAFit > 4 ? 4 : kNumAFit;
  static constexpr int kD0 = kNumA * kACols;
  // warps
  static constexpr int kDqWarps = 4 * kSub;
  static constexpr int kDqWarp0 = 1;
  static constexpr int kMmaWarp0 = kDqWarp0 + kDqWarps;
  static constexpr int kEpWarp0 = kMmaWarp0 + kMmaWarps;
  static constexpr int kThreads = 32 * (kEpWarp0 + 4);
  // activation chunks (16 bytes) each dequant lane converts per stage
  static constexpr int kXChunksPerLane = (kSub * kXBoxBytes / 16) / (kDqWarps * 32);
  static_assert(kStages >= 3, "pipeline too shallow");
  static_assert(kNumA >= 2, "TMEM A ring too shallow");
  static_assert(kD0 + kDBufs * kDCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kXChunksPerLane * kDqWarps * 32 * 16 == kSub * kXBoxBytes, "activation split");
};

struct Params {
  int T, N, K;
  int group_size;      // 0 = per output channel
  int gshift;          // log2(group_size) (group_size is a power of two)
  int ks;              // stages per tile = ceil(K / stage k)
  long long total;     // tiles * ks units
  uint32_t tx;         // TMA bytes per full stage
  const uint16_t* scales;   // per-channel int8 scales (epilogue)
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

// int4: 64 codes (group j of the row's 128-byte stage line) to fp16 weights
// (code - zero) * scale in natural k order: a[i] holds k = 2i (low half) and
// 2i+1 (high half).  Code layout: nibble p (0..7, from the least significant
// end) of each little-endian 32-bit word holds k = 8w + 2*(p % 4) + p / 4, so
// masking nibbles {0, 4} gives the pair (k0, k1), {1, 5} gives (k2, k3), and
// the same on the word shifted by 8 gives (k4, k5), (k6, k7).  A nibble in
// bits 0-3 of a half becomes 1024 + c with the fp16 exponent of 1024, a
// nibble in bits 4-7 becomes 64 + c with the exponent of 64 -- both exact.
// The line was written by TMA with the 128-byte swizzle: 16-byte chunk c of
// row m sits at chunk position c ^ (m & 7).
__device__ __forceinline__ void dequant_w4(uint32_t row_addr, uint32_t m, int j, uint32_t z,
                                           uint32_t s2, uint32_t (&a)[32]) {
  const uint32_t sw = m & 7u;
  const uint4 c0 = lds128(row_addr + (((2u * j) ^ sw) << 4));
  const uint4 c1 = lds128(row_addr + (((2u * j + 1u) ^ sw) << 4));
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const uint32_t zlo = (0x6400u | z) * 0x00010001u;            // fp16x2 (1024 + z)
  const uint32_t zhi = (0x5400u | (z << 4)) * 0x00010001u;     // fp16x2 (64 + z)
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = words[w];
    const uint32_t q8 = q >> 8;
    a[4 * w + 0] = mul_f16x2(sub_f16x2(lop3_and_or(q, 0x000F000Fu, 0x64006400u), zlo), s2);
    a[4 * w + 1] = mul_f16x2(sub_f16x2(lop3_and_or(q, 0x00F000F0u, 0x54005400u), zhi), s2);
    a[4 * w + 2] = mul_f16x2(sub_f16x2(lop3_and_or(q8, 0x000F000Fu, 0x64006400u), zlo), s2);
    a[4 * w + 3] = mul_f16x2(sub_f16x2(lop3_and_or(q8, 0x00F000F0u, 0x54005400u), zhi), s2);
  }
}

// int8: 64 codes (group j of the row's 128-byte stage line) to fp16 code *
// scale (grouped) or the exact code (per channel, scale applied later).  A
// biased byte b = code + 128 becomes the fp16 1024 + b (exact), minus 1152.
template <bool kScaled>
__device__ __forceinline__ void dequant_w8(uint32_t row_addr, uint32_t m, int j, uint32_t s2,
                                           uint32_t (&a)[32]) {
  const uint32_t sw = m & 7u;
  const uint32_t bias = 0x64806480u;                           // fp16x2 (1152, 1152)
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = lds128(row_addr + (((uint32_t)(4 * j + c) ^ sw) << 4));
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t u = words[w] ^ 0x80808080u;
      uint32_t lo = sub_f16x2(__byte_perm(u, 0x64646464u, 0x4140u), bias);
      uint32_t hi = sub_f16x2(__byte_perm(u, 0x64646464u, 0x4342u), bias);
      if (kScaled) {
        lo = mul_f16x2(lo, s2);
        hi = mul_f16x2(hi, s2);
      }
      a[8 * c + 2 * w] = lo;
      a[8 * c + 2 * w + 1] = hi;
    }
  }
}

template <int QUANT, int TPAD>
__global__ void __launch_bounds__(Cfg<QUANT, TPAD>::kThreads, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_codes,
                 const __grid_constant__ CUtensorMap tm_scales,
                 const __grid_constant__ CUtensorMap tm_zeros, const Params p) {
  using C = Cfg<QUANT, TPAD>;
  constexpr int S = C::kStages, NA = C::kNumA, SUB = C::kSub, NDB = C::kDBufs;
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
  uint64_t* d_empty = d_full + NDB;
  uint64_t* wg_bar = d_empty + NDB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wg_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* fix_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const long long begin = unit_begin(blockIdx.x, p.total, G);
  const long long end = unit_begin(blockIdx.x + 1, p.total, G);
  const bool per_channel = (QUANT == kW8) && p.group_size == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kDqWarps + kMmaWarps);   // dequant warps + MMA commits
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&a_full[s], C::kDqWarps);
      mbar_init(&a_empty[s], kMmaWarps);
    }
    for (int b = 0; b < NDB; ++b) {
      mbar_init(&d_full[b], kMmaWarps);
      mbar_init(&d_empty[b], 4);
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
  // and the scale/zero row of group j inside the stage's box
  auto nsub_of = [&](int kst) { return min(SUB, (p.K - kst * C::kStageKK) >> 6); };
  auto grow_of = [&](int kst, int j) {
    return p.group_size ? (((kst * C::kStageKK + 64 * j) >> p.gshift) - ((kst * C::kStageKK) >> p.gshift))
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
    // ------------------------------------------------------------ dequant + activation conversion
    const int dq = warp - C::kDqWarp0;
    const int q = warp & 3;                   // TMEM lane quadrant this warp may access
    const int jj = dq >> 2;                   // 64-k group of each stage this warp handles
    const int m = q * 32 + lane;              // weight row inside the tile
    const uint32_t a_addr0 = tbase + ((uint32_t)(q * 32) << 16) + jj * 32;
    const uint32_t zshift = (m & 1) * 4;
    const int xchunk0 = (dq * 32 + lane) * C::kXChunksPerLane;
    float xmax = 0.f;
    UnitIter it(begin, p.ks);
    Ring<S> st_ring;
    Ring<NA> a_ring;
    for (long long n = 0; n < nunits; ++n, it.next(), st_ring.next(), a_ring.next()) {
      const int nsub = nsub_of(it.kst);
      const int s = st_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], st_ring.phase, abort_flag, p.err))) break;
      const uint8_t* st = smem + s * C::kStageBytes;
      uint32_t a[32];
      if (jj < nsub) {
        const int grow = grow_of(it.kst, jj);
        const __half sc = reinterpret_cast<const __half*>(st + C::kScaleOff)[grow * kTileM + m];
        const uint32_t s2 = (uint32_t)__half_as_ushort(sc) * 0x00010001u;
        const uint32_t row_addr = smem_u32(st + C::kCodeOff) + m * 128;
        if constexpr (QUANT == kW4) {
          const uint32_t zb = st[C::kZeroOff + grow * 64 + (m >> 1)];
          dequant_w4(row_addr, m, jj, (zb >> zshift) & 0xFu, s2, a);
        } else {
          if (per_channel)
            dequant_w8<false>(row_addr, m, jj, s2, a);
          else
            dequant_w8<true>(row_addr, m, jj, s2, a);
        }
      }
      // this lane's share of the stage's activations: bf16 -> fp16 in place
      {
        const uint32_t xbase = smem_u32(st + C::kXOff);
#pragma unroll
        for (int c = 0; c < C::kXChunksPerLane; ++c) {
          const int chunk = xchunk0 + c;
          if (chunk * 16 < nsub * C::kXBoxBytes) {
            const uint32_t addr = xbase + chunk * 16;
            uint4 v = lds128(addr);
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(w[e] << 16);
              const float hi = __uint_as_float(w[e] & 0xFFFF0000u);
              xmax = fmaxf(xmax, fmaxf(fabsf(lo), fabsf(hi)));
              w[e] = pack_f16x2(lo, hi);
            }
            sts128(addr, make_uint4(w[0], w[1], w[2], w[3]));
          }
        }
        fence_proxy_async_smem();
      }
      const int sa = a_ring.slot;
      if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[sa], a_ring.phase ^ 1, abort_flag, p.err))) break;
      if (jj < nsub) {
        tc_fence_after();
        tmem_st_32x32b_x32(a_addr0 + sa * C::kACols, a);
        tmem_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[sa]);
        mbar_arrive(&empty[s]);
      }
    }
    // 65520 and above round to infinity in fp16
    if (!(xmax < 65520.f)) atomicCAS(p.err, 0, kDevErrRange);
  } else if (warp < C::kEpWarp0) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const int mw = warp - C::kMmaWarp0;
      constexpr uint32_t idesc = idesc_f16_f32(128, TPAD);
      UnitIter it(begin, p.ks);
      Ring<S> st_ring;
      Ring<NA> a_ring;
      Ring<NDB> d_ring;
      bool ok = true;
      int last_sa = -1;
      uint32_t last_phase = 0;
      long long n = 0;
      while (ok && n < nunits) {
        // one tile segment into accumulator buffer d_ring.slot
        const long long tile_end = (long long)(it.tile + 1) * p.ks;
        const long long seg_len = min(end, tile_end) - (begin + n);
        const uint32_t d_col = tbase + C::kD0 + d_ring.slot * C::kDCols + mw * TPAD;
        if (!mbar_wait(&d_empty[d_ring.slot], d_ring.phase, abort_flag, p.err)) break;
        for (long long e = 0; e < seg_len; ++e, ++n, it.next(), st_ring.next(), a_ring.next()) {
          const int nsub = nsub_of(it.kst);
          const int s = st_ring.slot, sa = a_ring.slot;
          if (!mbar_wait(&a_full[sa], a_ring.phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc0 = smem_desc_sw128(smem + s * C::kStageBytes + C::kXOff);
          {
            const int jg = mw;
            if (jg < nsub) {
              const uint32_t a_col = tbase + sa * C::kACols + jg * 32;
              const uint64_t bdesc = bdesc0 + (uint64_t)((jg * C::kXBoxBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                // A: 8 TMEM columns (16 fp16) per K16 step; B: +32 bytes inside the swizzled row.
                // The accumulator is cleared by the epilogue, so every MMA accumulates.
                mma_ts(d_col, a_col + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, 1u);
              }
            }
          }
          mma_commit(&a_empty[sa]);
          mma_commit(&empty[s]);
          last_sa = sa;
          last_phase = a_ring.phase;
        }
        if (!ok) break;
        mma_commit(&d_full[d_ring.slot]);
        d_ring.next();
      }
      if (*abort_flag && last_sa >= 0) {
        // wait for this thread's own MMAs before the CTA frees its tensor memory
        volatile int no_abort = 0;
        mbar_wait(&a_empty[last_sa], last_phase, &no_abort, nullptr, kDrainLimitNs);
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
    auto clear_d = [&](int b) {
      uint32_t zeros32[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) zeros32[c] = 0u;
#pragma unroll
      for (int c = 0; c < C::kDCols; c += 32)
        tmem_st_32x32b_x32(tbase + lane_base + C::kD0 + b * C::kDCols + c, zeros32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[b]);
    };
    for (int b = 0; b < NDB; ++b) clear_d(b);

    UnitIter it(begin, p.ks);
    Ring<NDB> d_ring;
    bool ok = true;
    long long n = 0;
    while (ok && n < nunits) {
      const int tile = it.tile;
      const long long tile_first = (long long)tile * p.ks;
      const long long u0 = begin + n;
      const long long seg_end = min(end, tile_first + p.ks);
      const bool whole_tile = (u0 == tile_first) && (seg_end == tile_first + p.ks);
      for (long long u = u0; u < seg_end; ++u, ++n) it.next();
      const int b = d_ring.slot;
      ok = __all_sync(0xffffffffu, mbar_wait(&d_full[b], d_ring.phase, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const int nrow = tile * kTileM + m;
      const float osc = per_channel && nrow < p.N ? __half2float(__ushort_as_half(p.scales[nrow])) : 1.f;
      const uint32_t dbase = tbase + lane_base + C::kD0 + b * C::kDCols;
      // sum of the MMA warps' accumulators, 16 columns at a time
      auto load_chunk = [&](int h, float (&v)[16]) {
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = 0.f;
#pragma unroll
        for (int w = 0; w < kMmaWarps; w += 2) {
          uint32_t r0[16], r1[16];
          tmem_ld_32x32b_x16(dbase + w * TPAD + h * 16, r0);
          tmem_ld_32x32b_x16(dbase + (w + 1) * TPAD + h * 16, r1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] += __uint_as_float(r0[c]) + __uint_as_float(r1[c]);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] *= osc;
      };
      if (whole_tile) {
#pragma unroll
        for (int h = 0; h < TPAD / 16; ++h) {
          float v[16];
          load_chunk(h, v);
          if (nrow < p.N) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int t = h * 16 + c;
              if (t < p.T) {
                if (p.y_f32)
                  reinterpret_cast<float*>(p.y)[(size_t)t * p.N + nrow] = v[c];
                else
                  reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)t * p.N + nrow] = __float2bfloat16_rn(v[c]);
              }
            }
          }
        }
        clear_d(b);
      } else {
        // Split tile: add this CTA's partial into the tile's fp32 slot (keyed
        // by the tile's first contributor, unique per split tile); the last
        // contributor to arrive converts the sum and clears the slot.
        const int c_first = cta_of_unit(tile_first, p.total, G);
        const int c_last = cta_of_unit(tile_first + p.ks - 1, p.total, G);
        float* slot = p.partials + (size_t)c_first * kPartialSlotFloats;
#pragma unroll
        for (int h = 0; h < TPAD / 16; ++h) {
          float v[16];
          load_chunk(h, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) red_add_f32(slot + (h * 16 + c) * kTileM + m, v[c]);
        }
        clear_d(b);
        __threadfence();
        ok = wg_sync();
        if (!ok) break;
        if (q == 0 && lane == 0) {
          const int old = atomicAdd(&p.counters[tile], 1);
          *fix_flag = (old == c_last - c_first) ? 1 : 0;
        }
        ok = wg_sync();
        if (!ok) break;
        if (*fix_flag) {
          __threadfence();
#pragma unroll 4
          for (int t = 0; t < TPAD; ++t) {
            const float v = __ldcg(slot + t * kTileM + m);
            __stcg(slot + t * kTileM + m, 0.f);
            if (t < p.T && nrow < p.N) {
              if (p.y_f32)
                reinterpret_cast<float*>(p.y)[(size_t)t * p.N + nrow] = v;
              else
                reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)t * p.N + nrow] = __float2bfloat16_rn(v);
            }
          }
          if (q == 0 && lane == 0) atomicExch(&p.counters[tile], 0);
        }
        // keep fix_flag stable until every warp has read it
        ok = wg_sync();
        if (!ok) break;
      }
      d_ring.next();
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
  const long long tiles = (a.N + kTileM - 1) / kTileM;
  p.total = tiles * p.ks;
  p.tx = C::kSub * C::kXBoxBytes + C::kCodeBytes + sr * kTileM * 2 + (QUANT == kW4 ? sr * 64 : 0);
  p.scales = a.scales;
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
