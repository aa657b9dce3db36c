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
    case 256: return launch_r<8>(x, y, T, K, signs, s);
    case 512: return launch_r<16>(x, y, T, K, signs, s);
    case 1024: return launch_r<32>(x, y, T, K, signs, s);
    default: return set_error(SPEC_ERR_SHAPE, "hadamard block %d not a power of two in [32, 1024]", block);
  }
}

}  // namespace sv
