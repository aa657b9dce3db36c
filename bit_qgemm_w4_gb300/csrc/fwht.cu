// Block-diagonal random Hadamard rotation of bf16 activations.
//
// "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling", section
// "How Uzu optimizes bytes and tokens per pass": random sign flips applied
// before the mixing, a Hadamard matrix of +1/-1 entries with one overall
// scale, each block mixed on its own, exactly reversible.
//   y[t][block b] = (1/sqrt(B)) * H_B * (s[block b] .* x[t][block b])
// with H_B the Sylvester matrix in natural order, computed as the in-place
// fast Walsh-Hadamard butterfly (pairs (i, i+h) -> (a+b, a-b), h = 1..B/2).
//
// One warp transforms one (row, block): lane l holds the R = B/32 contiguous
// elements l*R .. l*R+R-1, so the log2(R) low butterfly levels run inside a
// thread's registers and the five high levels are warp shuffles.  fp32 math,
// one rounding to bf16 at the end.

#include <cuda_bf16.h>

#include "internal.hpp"
#include "ptx.cuh"

namespace sv {
namespace {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int R>
__global__ void __launch_bounds__(256) fwht_kernel(const uint16_t* __restrict__ x, uint16_t* y,
                                                   int T, int K, const int8_t* __restrict__ signs,
                                                   float scale) {
  // A GEMM launched after this pre-pass may start streaming its weights at
  // once; it waits for this kernel before it reads the rotated activations.
  pdl_launch_dependents();
  constexpr int B = 32 * R;
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nblk = K / B;
  if (gw >= (long long)T * nblk) return;   // whole warp leaves together
  const int t = (int)(gw / nblk);
  const int b = (int)(gw % nblk);
  const long long col0 = (long long)b * B + (long long)lane * R;
  const uint16_t* xr = x + (long long)t * K + col0;

  float v[R];
  if constexpr (R % 8 == 0) {
#pragma unroll
    for (int r = 0; r < R; r += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(xr + r);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[r + 2 * j] = bf16_bits_to_f32(ws[j] & 0xFFFFu);
        v[r + 2 * j + 1] = bf16_bits_to_f32(ws[j] >> 16);
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = bf16_bits_to_f32(xr[r]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (signs[col0 + r] < 0) v[r] = -v[r];
  }
  // butterfly levels h < R: inside the thread
#pragma unroll
  for (int h = 1; h < R; h <<= 1) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if ((r & h) == 0) {
        const float a = v[r], c = v[r + h];
        v[r] = a + c;
        v[r + h] = a - c;
      }
    }
  }
  // levels h = R .. 16R: partner lane = lane ^ (h / R)
#pragma unroll
  for (int hl = 1; hl < 32; hl <<= 1) {
    const bool upper = (lane & hl) != 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float o = __shfl_xor_sync(0xffffffffu, v[r], hl);
      v[r] = upper ? (o - v[r]) : (v[r] + o);
    }
  }
  uint16_t* yr = y + (long long)t * K + col0;
  if constexpr (R % 8 == 0) {
#pragma unroll
    for (int r = 0; r < R; r += 8) {
      uint32_t ws[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ws[j] = (uint32_t)f32_to_bf16_bits(v[r + 2 * j] * scale) |
                ((uint32_t)f32_to_bf16_bits(v[r + 2 * j + 1] * scale) << 16);
      *reinterpret_cast<uint4*>(yr + r) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) yr[r] = f32_to_bf16_bits(v[r] * scale);
  }
}

template <int R>
int launch_r(const uint16_t* x, uint16_t* y, int T, int K, const int8_t* signs, cudaStream_t s) {
  constexpr int B = 32 * R;
  const long long warps = (long long)T * (K / B);
  const int per_block = 8;
  const long long blocks = (warps + per_block - 1) / per_block;
  const float scale = (float)(1.0 / sqrt((double)B));
  fwht_kernel<R><<<(unsigned)blocks, per_block * 32, 0, s>>>(x, y, T, K, signs, scale);
  return check_cuda(cudaGetLastError(), "fwht launch");
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
