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

constexpr int kThreads = 192;      // warp 0: TMA, warp 1: TMEM owner + MMA, warps 2-5: dequant
constexpr int kTmemCols = 256;     // two CTAs per SM share the 512 TMEM columns

template <int QUANT, int TPAD>
struct Cfg {
  static constexpr int kCodeRowBytes = QUANT == kW4 ? 32 : 64;  // one row's codes per stage
  static constexpr int kCodeBytes = kTileM * kCodeRowBytes;
  static constexpr int kXBytes = TPAD * 128;                    // TPAD rows x 64 bf16
  static constexpr int kScaleBytes = kTileM * 2;
  static constexpr int kZeroBytes = QUANT == kW4 ? kTileM / 2 : 0;
  static constexpr int kXOff = 0;
  static constexpr int kCodeOff = kXBytes;
  static constexpr int kScaleOff = kCodeOff + kCodeBytes;
  static constexpr int kZeroOff = kScaleOff + kScaleBytes;
  static constexpr int kStageBytes = (kZeroOff + 128 + 1023) / 1024 * 1024;
  static constexpr uint32_t kTx = kXBytes + kCodeBytes + kScaleBytes + kZeroBytes;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kSmemBudget = 110 * 1024;
  static constexpr int kStagesFit = (kSmemBudget - kCtrlBytes - 1024) / kStageBytes;
  static constexpr int kStages = kStagesFit > 12 ? 12 : kStagesFit;
  static constexpr int kSlotCols = 32 + TPAD;                   // A (32 cols) + partial D
  static constexpr int kTStagesFit = kTmemCols / kSlotCols;
  static constexpr int kTStages = kTStagesFit > 4 ? 4 : kTStagesFit;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kCtrlBytes;
  static_assert(kStages >= 3, "pipeline too shallow");
  static_assert(kTStages >= 2, "TMEM ring too shallow");
};

struct Params {
  int T, N, K;
  int group_size;      // 0 = per output channel
  int ks;              // stages per tile = K / 64
  long long total;     // tiles * ks units
  void* y;
  int y_f32;
  float* partials;
  int* counters;
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

// int4: one thread dequantises one row's 64 codes (32 bytes) to bf16 pairs of
// (code - zero), natural k order: a[j] holds k = 2j (low half), 2j+1 (high).
__device__ __forceinline__ void dequant_row_w4(uint32_t code_addr, uint32_t row, uint32_t z,
                                               uint32_t (&a)[32]) {
  const uint32_t sw = (row >> 2) & 1u;                 // 32-byte swizzle: chunk ^= addr bit 7
  const uint4 c0 = lds128(code_addr + ((0u ^ sw) << 4));
  const uint4 c1 = lds128(code_addr + ((1u ^ sw) << 4));
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const uint32_t zz = (0x4300u | z) * 0x00010001u;     // bf16x2 (128 + z, 128 + z)
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = words[w];
    const uint32_t q4 = q >> 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // byte j of q holds k = 8w+2j (low nibble); byte j of q4 holds k = 8w+2j+1
      const uint32_t t = __byte_perm(q, q4, 0x0400u + 0x0101u * j);
      const uint32_t v = lop3_and_or(t, 0x000F000Fu, 0x43004300u);   // bf16x2 (128+c0, 128+c1)
      a[4 * w + j] = sub_bf16x2(v, zz);                               // exact (c - z)
    }
  }
}

// int8: one thread converts one row's 64 codes (64 bytes) to exact bf16.
__device__ __forceinline__ void dequant_row_w8(uint32_t code_addr, uint32_t row,
                                               uint32_t (&a)[32]) {
  const uint32_t sw = (row >> 1) & 3u;                 // 64-byte swizzle: chunk ^= addr bits 7-8
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = lds128(code_addr + ((uint32_t(c) ^ sw) << 4));
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t u = words[w] ^ 0x80808080u;       // biased bytes code + 128
      float f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // fp32 2^23 + byte, minus 2^23 + 128 = code, exactly
        f[j] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u | j)) - 8388736.0f;
      }
      a[8 * c + 2 * w] = pack_bf16x2(f[0], f[1]);
      a[8 * c + 2 * w + 1] = pack_bf16x2(f[2], f[3]);
    }
  }
}

template <int QUANT, int TPAD>
__global__ void __launch_bounds__(kThreads, 2)
    qgemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_codes,
                 const __grid_constant__ CUtensorMap tm_scales,
                 const __grid_constant__ CUtensorMap tm_zeros, const Params p) {
  using C = Cfg<QUANT, TPAD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ctrl = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + C::kStages;
  uint64_t* a_ready = empty + C::kStages;
  uint64_t* mma_done = a_ready + C::kTStages;
  uint64_t* wg_bar = mma_done + C::kTStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wg_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* fix_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const long long begin = unit_begin(blockIdx.x, p.total, G);
  const long long end = unit_begin(blockIdx.x + 1, p.total, G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4 + 1);   // four dequant warps + one MMA commit
    }
    for (int s = 0; s < C::kTStages; ++s) {
      mbar_init(&a_ready[s], 4);
      mbar_init(&mma_done[s], 1);
    }
    mbar_init(wg_bar, 4);
    *abort_flag = 0;
    *fix_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_codes);
    prefetch_tensormap(&tm_scales);
    if (QUANT == kW4) prefetch_tensormap(&tm_zeros);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      int i = 0;
      for (long long u = begin; u < end; ++u, ++i) {
        const int tile = (int)(u / p.ks);
        const int kst = (int)(u - (long long)tile * p.ks);
        const int s = i % C::kStages;
        if (!mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, abort_flag, p.err)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], C::kTx);
        tma_load_2d(st + C::kXOff, &tm_x, &full[s], kst * kStageK, 0);
        tma_load_2d_hint(st + C::kCodeOff, &tm_codes, &full[s], kst * C::kCodeRowBytes,
                         tile * kTileM, pol_w);
        const int g = p.group_size ? (kst * kStageK) / p.group_size : 0;
        tma_load_2d(st + C::kScaleOff, &tm_scales, &full[s], tile * kTileM, g);
        if (QUANT == kW4) tma_load_2d(st + C::kZeroOff, &tm_zeros, &full[s], tile * (kTileM / 2), g);
      }
      if (*abort_flag) {
        // drain copies still in flight into this CTA's shared memory
        for (int j = (i > C::kStages ? i - C::kStages : 0); j < i; ++j) {
          volatile int no_abort = 0;
          mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, &no_abort, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, TPAD);
      int i = 0;
      for (long long u = begin; u < end; ++u, ++i) {
        const int s = i % C::kStages;
        const int ts = i % C::kTStages;
        if (!mbar_wait(&full[s], (i / C::kStages) & 1, abort_flag, p.err)) break;
        if (!mbar_wait(&a_ready[ts], (i / C::kTStages) & 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t a_col = tbase + ts * C::kSlotCols;
        const uint32_t d_col = a_col + 32;
        const uint64_t bdesc = smem_desc_sw128(smem + s * C::kStageBytes + C::kXOff);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // A: 8 TMEM columns (16 bf16) per K16 step; B: +32 bytes inside the swizzled row
          mma_ts(d_col, a_col + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&mma_done[ts]);
        mma_commit(&empty[s]);
      }
      if (*abort_flag && i > 0) {
        volatile int no_abort = 0;
        const int j = i - 1;
        mbar_wait(&mma_done[j % C::kTStages], (j / C::kTStages) & 1, &no_abort, nullptr,
                  kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int m = q * 32 + lane;             // weight row inside the tile
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int first_tile = (int)(begin / p.ks);
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

    // Add scale * partial(stage j) into acc; false on abort.
    auto consume = [&](int j, float sc) -> bool {
      const int ts = j % C::kTStages;
      bool ok = mbar_wait(&mma_done[ts], (j / C::kTStages) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
      uint32_t r[TPAD / 16][16];
      const uint32_t d_addr = tbase + lane_base + ts * C::kSlotCols + 32;
#pragma unroll
      for (int h = 0; h < TPAD / 16; ++h) tmem_ld_32x32b_x16(d_addr + h * 16, r[h]);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < TPAD / 16; ++h)
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[h * 16 + c] = fmaf(sc, __uint_as_float(r[h][c]), acc[h * 16 + c]);
      return true;
    };

    bool ok = true;
    int i = 0;
    long long u = begin;
    int pend = -1;
    float pend_scale = 0.f;
    while (ok && u < end) {
      const int tile = (int)(u / p.ks);
      const long long tile_first = (long long)tile * p.ks;
      const long long seg_end = min(end, tile_first + p.ks);
      const bool whole_tile = (u == tile_first) && (seg_end == tile_first + p.ks);
      for (; u < seg_end; ++u, ++i) {
        const int s = i % C::kStages;
        const int ts = i % C::kTStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (i / C::kStages) & 1, abort_flag, p.err));
        if (!ok) break;
        const uint8_t* st = smem + s * C::kStageBytes;
        const float sc = __half2float(reinterpret_cast<const __half*>(st + C::kScaleOff)[m]);
        uint32_t a[32];
        if constexpr (QUANT == kW4) {
          const uint32_t zb = st[C::kZeroOff + (m >> 1)];
          const uint32_t z = (zb >> ((m & 1) * 4)) & 0xFu;
          dequant_row_w4(smem_u32(st + C::kCodeOff) + m * C::kCodeRowBytes, m, z, a);
        } else {
          dequant_row_w8(smem_u32(st + C::kCodeOff) + m * C::kCodeRowBytes, m, a);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        // The slot's previous partial (stage i - kTStages) was consumed at
        // iteration i - kTStages + 1 <= i - 1, so A and D may be overwritten.
        tmem_st_32x32b_x32(tbase + lane_base + ts * C::kSlotCols, a);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_ready[ts]);
        if (pend >= 0) {
          ok = consume(pend, pend_scale);
          if (!ok) break;
        }
        pend = i;
        pend_scale = sc;
      }
      if (!ok) break;
      if (pend >= 0) {
        ok = consume(pend, pend_scale);
        if (!ok) break;
        pend = -1;
      }

      // ---- segment epilogue
      const int n = tile * kTileM + m;
      bool store = whole_tile;
      if (!whole_tile) {
        const int slot = 2 * (int)blockIdx.x + (tile == first_tile ? 0 : 1);
        float* w = p.partials + (size_t)slot * kPartialSlotFloats;
#pragma unroll
        for (int t = 0; t < TPAD; ++t) w[t * kTileM + m] = acc[t];
        __threadfence();
        ok = wg_sync();
        if (!ok) break;
        const int c_first = cta_of_unit(tile_first, p.total, G);
        const int c_last = cta_of_unit(tile_first + p.ks - 1, p.total, G);
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
          for (int t = 0; t < TPAD; ++t) acc[t] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const int c_first_tile = (int)(unit_begin(c, p.total, G) / p.ks);
            const int cs = 2 * c + (c_first_tile == tile ? 0 : 1);
            const float* wr = p.partials + (size_t)cs * kPartialSlotFloats;
#pragma unroll
            for (int t = 0; t < TPAD; ++t) acc[t] += __ldcg(wr + t * kTileM + m);
          }
          if (q == 0 && lane == 0) atomicExch(&p.counters[tile], 0);
        }
        // keep fix_flag stable until every warp has read it
        ok = wg_sync();
        if (!ok) break;
      }
      if (store && n < p.N) {
        if (p.y_f32) {
          float* y = reinterpret_cast<float*>(p.y);
#pragma unroll
          for (int t = 0; t < TPAD; ++t)
            if (t < p.T) y[(size_t)t * p.N + n] = acc[t];
        } else {
          __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
#pragma unroll
          for (int t = 0; t < TPAD; ++t)
            if (t < p.T) y[(size_t)t * p.N + n] = __float2bfloat16_rn(acc[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < TPAD; ++t) acc[t] = 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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
  if (QUANT == kW4) {
    rc = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qcodes, (uint64_t)a.K / 2,
                        (uint64_t)a.N, (uint64_t)a.K / 2, 32, kTileM, CU_TENSOR_MAP_SWIZZLE_32B);
  } else {
    rc = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qcodes, (uint64_t)a.K, (uint64_t)a.N,
                        (uint64_t)a.K, 64, kTileM, CU_TENSOR_MAP_SWIZZLE_64B);
  }
  if (rc) return rc;
  const uint64_t groups = a.group_size ? (uint64_t)(a.K / a.group_size) : 1;
  rc = encode_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)a.N, groups,
                      (uint64_t)a.N * 2, kTileM, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc) return rc;
  if (QUANT == kW4) {
    rc = encode_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.zeros, (uint64_t)a.N / 2, groups,
                        (uint64_t)a.N / 2, kTileM / 2, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  } else {
    tz = ts;
  }

  Params p;
  p.T = a.T;
  p.N = a.N;
  p.K = a.K;
  p.group_size = a.group_size;
  p.ks = a.K / kStageK;
  const long long tiles = (a.N + kTileM - 1) / kTileM;
  p.total = tiles * p.ks;
  p.y = a.y;
  p.y_f32 = a.y_f32;
  p.partials = ctx->partials;
  p.counters = ctx->tile_counters;
  p.err = ctx->err;
  long long G = 2LL * ctx->num_sms;
  if (G > p.total) G = p.total;
  if (2 * G > ctx->max_slots) return set_error(SPEC_ERR_OOM, "workspace has too few partial slots");

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
  qgemm_kernel<QUANT, TPAD><<<(unsigned)G, kThreads, C::kSmemBytes, stream>>>(tx, tc, ts, tz, p);
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
