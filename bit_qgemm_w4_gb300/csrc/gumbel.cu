// Shared-seed (Gumbel-max) sampling and acceptance for the verify step.
//
// What it computes (the trymirai post feed, nitterts.pages.dev/trymirai, the
// post with the "random number from 1 to 10" example): the speculator and
// the target model sample with the same seed through the Gumbel-max trick,
// token = argmax_v (logit_v + g_v) with g_v = -log(-log u_v) from shared
// randomness, so that matching distributions give matching tokens and every
// draft is accepted.  Verification keeps the drafts while each equals the
// target's own sample at its position and emits the target's sample at the
// first position that differs, or at the bonus position after the last draft.
//
// Noise: token v at draft position p takes word v mod 4 of Philox4x32-10
// (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011) at counter (v div 4, p mod 2^32, p div 2^32, 0) under key
// (seed mod 2^32, seed div 2^32).  A word w becomes u = (2 floor(w / 2^9) + 1)
// * 2^-24, exact in fp32 and strictly inside (0, 1).  A drafter on this GPU
// draws its tokens with spec_gumbel_sample under the same seed and positions.
//
// One launch, grid (V-chunks, rows): each block streams its chunk of one row
// once (16-byte loads when the rows are aligned), generating one Philox block
// per four tokens, and keeps the best (value, token) and the runner-up value;
// the last block to arrive (atomic counter, no waiting) merges every row's
// chunks, then walks the drafts (acceptance) or writes one token per row
// (sampling).  Equal values go to the smaller token id.

#include <cmath>

#include "internal.hpp"

namespace sv {
namespace {

constexpr int kGBlock = 256;
constexpr float kGTieEps = 1e-4f;   // best minus runner-up below this: a near tie
constexpr int kDevErrBadToken = 2;
constexpr int kNoToken = 0x7fffffff;
constexpr int kMergeBatch = 1024;   // chunk partials staged in shared memory at a time

struct GumbelArgs {
  const float* logits;
  int rows, V, nchunks, chunk;   // chunk: tokens per block, a multiple of 4
  int vec;                       // rows start on 16-byte boundaries
  uint32_t key0, key1;
  uint64_t position;             // draft position of row 0
  int accept;                    // 1: acceptance over rows - 1 drafts; 0: sampling
  const int32_t* drafts;         // acceptance: [rows - 1] (nullptr when there are none)
  float* best;                   // [rows][nchunks] partials
  int* idx;
  float* second;
  int* counter;
  int32_t* tokens;               // acceptance: [n + 1]; sampling: [rows]
  int32_t* n_acc;                // acceptance only
  int32_t* flags;                // nullable [rows]
  int* err;
};

// Ten rounds: the products M0 * x0 and M1 * x2 split into high and low
// words give the next counter (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0), and
// the key advances by the two Weyl constants after each round.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// g = -log(e), e = -log(u).  e needs a small relative error, which the fast
// logarithm (absolute error a few 1e-7 near 1) lacks as u -> 1; there
// e = -log(1 - d) = d + d^2/2 + d^3/3 + ... with d = 1 - u, exact from the
// same integer, truncated after d^6 (relative error below d^6 / 7 < 1e-8 for
// d < 1/16).  The outer logarithm only needs a small absolute error: the
// fast one keeps g within a few 1e-6 of the exact value, far inside the
// 1e-4 near-tie band.
__device__ __forceinline__ float gumbel_of(uint32_t w) {
  const uint32_t m = w >> 9;                                  // u = (2m + 1) / 2^24
  const float u = (float)(2u * m + 1u) * 0x1p-24f;
  const float d = (float)(2u * (0x7FFFFFu - m) + 1u) * 0x1p-24f;   // 1 - u
  const float series =
      d * (1.f + d * (0.5f + d * (1.f / 3.f + d * (0.25f + d * (0.2f + d * (1.f / 6.f))))));
  const float e = u > 0.9375f ? series : -__logf(u);
  return -__logf(e);
}

// The best (value, token) of a set and the largest value of the rest.
struct Top2 {
  float b;
  int i;
  float s;
};

__device__ __forceinline__ bool g_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void top2_add(Top2& t, float z, int v) {
  if (g_better(z, v, t.b, t.i)) {
    t.s = fmaxf(t.s, t.b);
    t.b = z;
    t.i = v;
  } else if (z > t.s) {
    t.s = z;
  }
}

__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b) {
  if (g_better(b.b, b.i, a.b, a.i)) {
    b.s = fmaxf(fmaxf(b.s, a.s), a.b);
    return b;
  }
  a.s = fmaxf(fmaxf(a.s, b.s), b.b);
  return a;
}

__global__ void __launch_bounds__(kGBlock) gumbel_kernel(GumbelArgs a) {
  __shared__ Top2 sh[kGBlock / 32];
  __shared__ int s_last, s_n;
  __shared__ int s_tok[kMaxAcceptT + 1];
  __shared__ int s_draft[kMaxAcceptT];
  __shared__ Top2 s_part[kMergeBatch];

  const int c = blockIdx.x, row = blockIdx.y;
  const int lo = c * a.chunk;
  const int hi = min(a.V, lo + a.chunk);
  const float* l = a.logits + (long long)row * a.V;
  const uint64_t pos = a.position + (uint64_t)row;
  const uint32_t p_lo = (uint32_t)pos, p_hi = (uint32_t)(pos >> 32);

  Top2 t{-INFINITY, kNoToken, -INFINITY};
  for (int v0 = lo + 4 * threadIdx.x; v0 < hi; v0 += 4 * kGBlock) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)(v0 >> 2), p_lo, p_hi, 0u), a.key0, a.key1);
    if (a.vec && v0 + 3 < hi) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(l + v0));
      top2_add(t, x.x + gumbel_of(w.x), v0);
      top2_add(t, x.y + gumbel_of(w.y), v0 + 1);
      top2_add(t, x.z + gumbel_of(w.z), v0 + 2);
      top2_add(t, x.w + gumbel_of(w.w), v0 + 3);
    } else {
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (v0 + j < hi) top2_add(t, __ldg(l + v0 + j) + gumbel_of(ws[j]), v0 + j);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Top2 u{__shfl_xor_sync(0xffffffffu, t.b, o), __shfl_xor_sync(0xffffffffu, t.i, o),
                 __shfl_xor_sync(0xffffffffu, t.s, o)};
    t = top2_merge(t, u);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sh[warp] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kGBlock / 32; ++k) t = top2_merge(t, sh[k]);
    const int at = row * a.nchunks + c;
    a.best[at] = t.b;
    a.idx[at] = t.i;
    a.second[at] = t.s;
    __threadfence();
    s_last = atomicAdd(a.counter, 1) == (int)(gridDim.x * gridDim.y) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last block: the chunk partials in batches of rows, every load of a
  // batch in flight together, then one warp per row merges the row's chunks
  // from shared memory (lanes over chunks)
  const int nc = a.nchunks;
  const int batch_rows = kMergeBatch / nc;
  for (int r0 = 0; r0 < a.rows; r0 += batch_rows) {
    const int r1 = min(a.rows, r0 + batch_rows);
    for (int e = threadIdx.x; e < (r1 - r0) * nc; e += kGBlock) {
      const int at = r0 * nc + e;
      s_part[e] = Top2{__ldcg(a.best + at), __ldcg(a.idx + at), __ldcg(a.second + at)};
    }
    __syncthreads();
    for (int r = r0 + warp; r < r1; r += kGBlock / 32) {
      Top2 m{-INFINITY, kNoToken, -INFINITY};
      for (int k = lane; k < nc; k += 32) m = top2_merge(m, s_part[(r - r0) * nc + k]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const Top2 u{__shfl_xor_sync(0xffffffffu, m.b, o), __shfl_xor_sync(0xffffffffu, m.i, o),
                     __shfl_xor_sync(0xffffffffu, m.s, o)};
        m = top2_merge(m, u);
      }
      if (lane == 0) {
        const int tok = m.i == kNoToken ? 0 : m.i;   // a row of NaNs: token 0
        s_tok[r] = tok;
        if (a.flags) a.flags[r] = (m.b - m.s < kGTieEps) ? 1 : 0;
        if (!a.accept) a.tokens[r] = tok;
      }
    }
    __syncthreads();
  }
  if (a.accept) {
    // every draft tested at once; the first rejection is the smallest
    // failing position
    const int T = a.rows - 1;
    if (threadIdx.x == 0) s_n = T;
    __syncthreads();
    for (int i = threadIdx.x; i < T; i += kGBlock) {
      const int d = a.drafts[i];
      s_draft[i] = d;
      if (d < 0 || d >= a.V || d != s_tok[i]) atomicMin(&s_n, i);
    }
    __syncthreads();
    const int n = s_n;
    for (int i = threadIdx.x; i < n; i += kGBlock) a.tokens[i] = s_draft[i];
    if (threadIdx.x == 0) {
      if (n < T && (s_draft[n] < 0 || s_draft[n] >= a.V))   // never matches; reported
        atomicCAS(a.err, 0, kDevErrBadToken);
      a.tokens[n] = s_tok[n];
      *a.n_acc = n;
    }
  }
  if (threadIdx.x == 0) *a.counter = 0;
}

}  // namespace

int launch_gumbel(spec_ctx* ctx, const float* logits, int rows, int V, uint64_t seed, uint64_t position,
                  int accept, const int32_t* drafts, int32_t* tokens, int32_t* n_acc, int32_t* flags,
                  cudaStream_t s) {
  GumbelArgs a;
  a.logits = logits;
  a.rows = rows;
  a.V = V;
  // one full wave of resident blocks in all, at least 1024 tokens a block
  static int per_sm = 0;
  if (per_sm == 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, gumbel_kernel, kGBlock, 0) != cudaSuccess || b < 1)
      b = 4;
    per_sm = b;
  }
  long long want = (long long)per_sm * ctx->num_sms / rows;
  long long by_size = ((long long)V + 1023) / 1024;
  long long nc = want < by_size ? want : by_size;
  if (nc < 1) nc = 1;
  if (nc > kAcceptChunks) nc = kAcceptChunks;
  const long long chunk = (((long long)V + nc - 1) / nc + 3) / 4 * 4;
  a.chunk = (int)chunk;
  a.nchunks = (int)(((long long)V + chunk - 1) / chunk);
  a.vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  a.key0 = (uint32_t)seed;
  a.key1 = (uint32_t)(seed >> 32);
  a.position = position;
  a.accept = accept;
  a.drafts = drafts;
  a.best = ctx->gum_best;
  a.idx = ctx->gum_idx;
  a.second = ctx->gum_second;
  a.counter = ctx->acc_counters + 2;
  a.tokens = tokens;
  a.n_acc = n_acc;
  a.flags = flags;
  a.err = ctx->err;
  dim3 g(a.nchunks, rows);
  gumbel_kernel<<<g, kGBlock, 0, s>>>(a);
  return check_cuda(cudaGetLastError(), "gumbel launch");
}

}  // namespace sv
