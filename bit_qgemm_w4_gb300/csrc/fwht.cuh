// One warp's block-diagonal random Hadamard rotation of one (row, block).
//
// "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling", section
// "How Uzu optimizes bytes and tokens per pass": random sign flips applied
// before the mixing, a Hadamard matrix of +1/-1 entries with one overall
// scale, each block mixed on its own, exactly reversible.
//   y[block] = (1/sqrt(B)) * H_B * (s[block] .* x[block])
// with H_B the Sylvester matrix in natural order, computed as the in-place
// fast Walsh-Hadamard butterfly (pairs (i, i+h) -> (a+b, a-b), h = 1..B/2).
//
// Lane l holds the R = B/32 contiguous elements l*R .. l*R+R-1, so the
// log2(R) low butterfly levels run inside a thread's registers and the five
// high levels are warp shuffles.  fp32 math, one rounding to bf16 at the end.
// Used by the standalone rotation kernel and, inside the verify GEMM, by the
// activation producer that rotates a GEMM's activations before they are
// loaded.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace sv {

__device__ __forceinline__ float fwht_bf16_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint32_t fwht_f32_to_bf16(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Output forms of the transform:
//  kFwhtBf16      one bf16 row (the standalone rotation)
//  kFwhtBf16Split two bf16 rows y and y + split_stride: the rounded value and
//                 the rounding's remainder, whose sum carries 16 significant
//                 bits (an MMA on bf16 operands multiplies both rows, so the
//                 rotation adds no bf16 rounding of its own)
//  kFwhtF16Nib    one fp16 row in the int4 GEMM's activation form: columns
//                 with k % 8 in {2, 3, 6, 7} divided by 16 (those columns
//                 meet weights that carry a factor 16)
//  kFwhtF16       one fp16 row
enum { kFwhtBf16 = 0, kFwhtBf16Split = 1, kFwhtF16Nib = 2, kFwhtF16 = 3 };

__device__ __forceinline__ uint32_t fwht_f32_to_f16(float f) {
  return (uint32_t)__half_as_ushort(__float2half_rn(f));
}

// Whether column k of a block that starts at a multiple of 8 carries the
// factor 1/16 in the kFwhtF16Nib form.
__device__ __forceinline__ bool fwht_nib(int k) { return (k & 2) != 0; }

// x, y and signs point at the start of the block (row t, columns b*B ..).
template <int R, int MODE>
__device__ __forceinline__ void fwht_warp(const uint16_t* x, uint16_t* y, const int8_t* signs,
                                          float scale, int lane, size_t split_stride = 0) {
  const int col0 = lane * R;
  const uint16_t* xr = x + col0;
  float v[R];
  if constexpr (R % 8 == 0) {
#pragma unroll
    for (int r = 0; r < R; r += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(xr + r);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[r + 2 * j] = fwht_bf16_to_f32(ws[j] & 0xFFFFu);
        v[r + 2 * j + 1] = fwht_bf16_to_f32(ws[j] >> 16);
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = fwht_bf16_to_f32(xr[r]);
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
#pragma unroll
  for (int r = 0; r < R; ++r) {
    v[r] *= scale;
    if (MODE == kFwhtF16Nib && fwht_nib(col0 + r)) v[r] *= 0.0625f;
  }
  uint16_t* yr = y + col0;
  auto enc = [](float f) { return MODE >= kFwhtF16Nib ? fwht_f32_to_f16(f) : fwht_f32_to_bf16(f); };
  if constexpr (R % 8 == 0) {
#pragma unroll
    for (int r = 0; r < R; r += 8) {
      uint32_t ws[4], wl[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a = enc(v[r + 2 * j]), b = enc(v[r + 2 * j + 1]);
        ws[j] = a | (b << 16);
        if (MODE == kFwhtBf16Split)
          wl[j] = fwht_f32_to_bf16(v[r + 2 * j] - fwht_bf16_to_f32(a)) |
                  (fwht_f32_to_bf16(v[r + 2 * j + 1] - fwht_bf16_to_f32(b)) << 16);
      }
      *reinterpret_cast<uint4*>(yr + r) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
      if (MODE == kFwhtBf16Split)
        *reinterpret_cast<uint4*>(yr + split_stride + r) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t a = enc(v[r]);
      yr[r] = (uint16_t)a;
      if (MODE == kFwhtBf16Split)
        yr[split_stride + r] = (uint16_t)fwht_f32_to_bf16(v[r] - fwht_bf16_to_f32(a));
    }
  }
}

// One thread's rotation of one small block (B = 32): the whole block in
// registers, the log2(B) butterfly levels without shuffles, the same output
// forms as fwht_warp.  Used where there are many small blocks, so that a
// warp rotates 32 blocks at once instead of one.  signs must be 16-byte
// aligned.
template <int B, int MODE>
__device__ __forceinline__ void fwht_thread(const uint16_t* x, uint16_t* y, const int8_t* signs,
                                            float scale, size_t split_stride = 0) {
  static_assert(B % 16 == 0, "whole 16-byte loads");
  float v[B];
#pragma unroll
  for (int r = 0; r < B; r += 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + r);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[r + 2 * j] = fwht_bf16_to_f32(ws[j] & 0xFFFFu);
      v[r + 2 * j + 1] = fwht_bf16_to_f32(ws[j] >> 16);
    }
  }
#pragma unroll
  for (int r = 0; r < B; r += 16) {
    const uint4 sg = *reinterpret_cast<const uint4*>(signs + r);
    const uint32_t sw[4] = {sg.x, sg.y, sg.z, sg.w};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if ((sw[j >> 2] >> (8 * (j & 3) + 7)) & 1u) v[r + j] = -v[r + j];
    }
  }
#pragma unroll
  for (int h = 1; h < B; h <<= 1) {
#pragma unroll
    for (int r = 0; r < B; ++r) {
      if ((r & h) == 0) {
        const float a = v[r], c = v[r + h];
        v[r] = a + c;
        v[r + h] = a - c;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < B; ++r) {
    v[r] *= scale;
    if (MODE == kFwhtF16Nib && fwht_nib(r)) v[r] *= 0.0625f;
  }
  auto enc = [](float f) { return MODE >= kFwhtF16Nib ? fwht_f32_to_f16(f) : fwht_f32_to_bf16(f); };
#pragma unroll
  for (int r = 0; r < B; r += 8) {
    uint32_t ws[4], wl[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t a = enc(v[r + 2 * j]), b = enc(v[r + 2 * j + 1]);
      ws[j] = a | (b << 16);
      if (MODE == kFwhtBf16Split)
        wl[j] = fwht_f32_to_bf16(v[r + 2 * j] - fwht_bf16_to_f32(a)) |
                (fwht_f32_to_bf16(v[r + 2 * j + 1] - fwht_bf16_to_f32(b)) << 16);
    }
    *reinterpret_cast<uint4*>(y + r) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    if (MODE == kFwhtBf16Split)
      *reinterpret_cast<uint4*>(y + split_stride + r) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
}

// Runtime block size B in {32, 64, ..., 1024}.
template <int MODE>
__device__ __forceinline__ void fwht_warp_any(int B, const uint16_t* x, uint16_t* y,
                                              const int8_t* signs, float scale, int lane,
                                              size_t split_stride = 0) {
  switch (B) {
    case 32: fwht_warp<1, MODE>(x, y, signs, scale, lane, split_stride); break;
    case 64: fwht_warp<2, MODE>(x, y, signs, scale, lane, split_stride); break;
    case 128: fwht_warp<4, MODE>(x, y, signs, scale, lane, split_stride); break;
    case 256: fwht_warp<8, MODE>(x, y, signs, scale, lane, split_stride); break;
    case 512: fwht_warp<16, MODE>(x, y, signs, scale, lane, split_stride); break;
    default: fwht_warp<32, MODE>(x, y, signs, scale, lane, split_stride); break;
  }
}

}  // namespace sv
