// Dequantised-weight export (fp32, exact) for checking a packed checkpoint.
//   int4: w[n][k] = (code[n][k] - zero[k/g][n]) * scale[k/g][n]
//   int8: w[n][k] = code[n][k] * scale
// ("Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
// section "How Uzu optimizes bytes and tokens per pass": asymmetric 4-bit,
// symmetric 8-bit, one scale per group.)  Both products fit fp32 exactly.

#include <cuda_fp16.h>

#include "internal.hpp"

namespace sv {
namespace {

__global__ void dequant_w4_kernel(const uint8_t* __restrict__ qc, const uint16_t* __restrict__ sc,
                                  const uint8_t* __restrict__ zr, int g, int N, int K,
                                  float* __restrict__ w) {
  const long long total = (long long)N * K;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i / K), k = (int)(i % K);
    // nibble p of each 32-bit word holds k = 8w + 2*(p % 4) + p / 4
    const int r = k & 7, pos = 4 * (r & 1) + (r >> 1);
    const uint32_t b = qc[(long long)n * (K / 2) + (k / 8) * 4 + (pos >> 1)];
    const int code = (pos & 1) ? (int)(b >> 4) : (int)(b & 15u);
    const int gi = k / g;
    const uint32_t zb = zr[(long long)gi * (N / 2) + n / 2];
    const int z = (n & 1) ? (int)(zb >> 4) : (int)(zb & 15u);
    const float s = __half2float(__ushort_as_half(sc[(long long)gi * N + n]));
    w[i] = (float)(code - z) * s;
  }
}

__global__ void dequant_w8_kernel(const int8_t* __restrict__ qc, const uint16_t* __restrict__ sc,
                                  int g, int N, int K, float* __restrict__ w) {
  const long long total = (long long)N * K;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i / K), k = (int)(i % K);
    const uint16_t sb = g ? sc[(long long)(k / g) * N + n] : sc[n];
    w[i] = (float)qc[i] * __half2float(__ushort_as_half(sb));
  }
}

}  // namespace

int launch_dequant(spec_ctx* ctx, int quant, const void* qcodes, const uint16_t* scales,
                   const uint8_t* zeros, int group_size, int N, int K, float* w, cudaStream_t s) {
  const long long total = (long long)N * K;
  long long blocks = (total + 255) / 256;
  const long long cap = 8LL * ctx->num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (quant == kW4)
    dequant_w4_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t*>(qcodes), scales,
                                                        zeros, group_size, N, K, w);
  else
    dequant_w8_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const int8_t*>(qcodes), scales,
                                                        group_size, N, K, w);
  return check_cuda(cudaGetLastError(), "dequant launch");
}

}  // namespace sv
