// Standalone block-diagonal random Hadamard rotation of bf16 activations
// (fwht_rotate).  The transform of one (row, block) is fwht_warp (fwht.cuh):
// "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "How Uzu optimizes bytes and tokens per pass".  The split GEMM
// engine runs it before each rotated GEMM (the stack engine rotates inside
// its own launch); it also serves callers that want the rotated activations
// themselves.

#include "fwht.cuh"
#include "internal.hpp"
#include "ptx.cuh"

namespace sv {
namespace {

template <int R>
__global__ void __launch_bounds__(256) fwht_kernel(const uint16_t* __restrict__ x, uint16_t* y,
                                                   int T, int K, const int8_t* __restrict__ signs,
                                                   float scale) {
  // the input may be written by the previous kernel on the stream
  pdl_wait_prior();
  pdl_launch_dependents();
  constexpr int B = 32 * R;
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nblk = K / B;
  if (gw >= (long long)T * nblk) return;   // whole warp leaves together
  const int t = (int)(gw / nblk);
  const int b = (int)(gw % nblk);
  const long long off = (long long)t * K + (long long)b * B;
  fwht_warp<R, kFwhtBf16>(x + off, y + off, signs + (long long)b * B, scale, lane);
}

// Blocks of 256 to 1024: one CTA of B/8 threads per (row, block), eight
// consecutive elements per thread.  The butterfly levels of element
// distance 1-4 run in registers, 8-128 across the warp's lanes (shuffles),
// 256 and 512 across its warps (shared memory); the levels commute, so this
// order gives the same transform as any other.  Many short threads instead
// of one long warp per block: a 1024-block no longer waits on one warp's
// 320 dependent steps.
template <int B>
__global__ void __launch_bounds__(B / 8) fwht_cta_kernel(const uint16_t* __restrict__ x, uint16_t* y, int K,
                                                         const int8_t* __restrict__ signs, float scale) {
  constexpr int NT = B / 8, NW = NT / 32;
  __shared__ float xs[NW > 1 ? B : 1];
  // the input may be written by the previous kernel on the stream
  pdl_wait_prior();
  pdl_launch_dependents();
  const int nblk = K / B;
  const int row = blockIdx.x / nblk;
  const int blk = blockIdx.x - row * nblk;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const long long off = (long long)row * K + (long long)blk * B + tid * 8;
  const uint4 raw = *reinterpret_cast<const uint4*>(x + off);
  const uint32_t ws[4] = {raw.x, raw.y, raw.z, raw.w};
  const int8_t* sg = signs + (long long)blk * B + tid * 8;
  float v[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = fwht_bf16_to_f32(ws[j] & 0xFFFFu);
    v[2 * j + 1] = fwht_bf16_to_f32(ws[j] >> 16);
  }
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (sg[r] < 0) v[r] = -v[r];
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if ((r & h) == 0) {
        const float a = v[r], c = v[r + h];
        v[r] = a + c;
        v[r + h] = a - c;
      }
    }
  }
  // lane bit d holds element bit 3 + log2(d): the lower partner keeps a + b,
  // the upper one a - b
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float o = __shfl_xor_sync(0xffffffffu, v[r], d);
      v[r] = upper ? o - v[r] : v[r] + o;
    }
  }
  if constexpr (NW > 1) {
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
      const bool upper = (w & d) != 0;
#pragma unroll
      for (int r = 0; r < 8; ++r) xs[tid * 8 + r] = v[r];
      __syncthreads();
      const int pt = tid ^ (32 * d);
      float o[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) o[r] = xs[pt * 8 + r];
      __syncthreads();   // every read of this level before the next level's writes
#pragma unroll
      for (int r = 0; r < 8; ++r) v[r] = upper ? o[r] - v[r] : v[r] + o[r];
    }
  }
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    out[j] = fwht_f32_to_bf16(v[2 * j] * scale) | (fwht_f32_to_bf16(v[2 * j + 1] * scale) << 16);
  *reinterpret_cast<uint4*>(y + off) = make_uint4(out[0], out[1], out[2], out[3]);
}

template <int B>
int launch_cta(const uint16_t* x, uint16_t* y, int T, int K, const int8_t* signs, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)T * (K / B)));
  cfg.blockDim = dim3(B / 8);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float scale = (float)(1.0 / sqrt((double)B));
  return check_cuda(cudaLaunchKernelEx(&cfg, fwht_cta_kernel<B>, x, y, K, signs, scale), "fwht launch");
}

template <int R>
int launch_r(const uint16_t* x, uint16_t* y, int T, int K, const int8_t* signs, cudaStream_t s) {
  constexpr int B = 32 * R;
  const long long warps = (long long)T * (K / B);
  const int per_block = 8;
  const long long blocks = (warps + per_block - 1) / per_block;
  const float scale = (float)(1.0 / sqrt((double)B));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(per_block * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return check_cuda(cudaLaunchKernelEx(&cfg, fwht_kernel<R>, x, y, T, K, signs, scale), "fwht launch");
}

}  // namespace

int launch_fwht(spec_ctx*, const uint16_t* x, uint16_t* y, int T, int K, const int8_t* signs,
                int block, cudaStream_t s) {
  switch (block) {
    case 32: return launch_r<1>(x, y, T, K, signs, s);
    case 64: return launch_r<2>(x, y, T, K, signs, s);
    case 128: return launch_r<4>(x, y, T, K, signs, s);
    case 256: return launch_cta<256>(x, y, T, K, signs, s);
    case 512: return launch_cta<512>(x, y, T, K, signs, s);
    case 1024: return launch_cta<1024>(x, y, T, K, signs, s);
    default: return set_error(SPEC_ERR_SHAPE, "hadamard block %d not a power of two in [32, 1024]", block);
  }
}

}  // namespace sv
