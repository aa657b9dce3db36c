// Softmax over the vocabulary and the acceptance rules of the verify step.
//
// Chain rule ("Speculative Decoding Clearly Explained", the cat-sat
// walkthrough): accept draft i with probability min(1, p/q), left to right,
// stop at the first rejection, draw the replacement from the normalised
// positive part of p - q; if every draft is accepted the target supplies one
// more token.  Tree rule ("Karpathy's Trick for Faster Local LLMs Finally Has
// Proper Tooling", section "Issue with parallel draft generation"): the target
// scores every node of the draft tree in one pass, and of the root paths whose
// nodes it confirms the deepest one is emitted -- here greedily, the target
// confirms a node when its token is the argmax of the row that scores it.
//
// Launch structure (two launches for the chain rule, one for the tree):
//  * row_stats_kernel: grid (chunks, rows); each block reduces one V-chunk of
//    one row to an online-softmax pair (max, sum exp(l - max)) -- one pass over
//    the logits, coalesced; the last block of a row to arrive (per-row
//    counter, no waiting) merges the row's pairs once and stores (max, 1/Z).
//  * accept_kernel: grid = V-chunks of the single row that is sampled.  Every
//    block reads the rows' (max, 1/Z), runs the (at most T) accept tests in
//    parallel and takes the first rejection, and sums its chunk of the
//    residual max(0, p_j - q_j) (or of p_T); the last block to arrive (atomic
//    counter, no waiting) does the inverse-CDF draw: it picks the chunk from
//    the chunk sums by a block-wide scan and scans that chunk only.
//  * tree_kernel: grid (chunks, T+1) argmax partials; the last block merges
//    them and walks the tree.

#include <cfloat>
#include <cmath>
#include <mutex>

#include "internal.hpp"

namespace sv {
namespace {

constexpr int kBlock = 256;
constexpr int kMergeBatch = 1024;   // chunk partials staged in shared memory at a time
constexpr int kDevErrBadToken = 2;
constexpr int kDevErrBadParent = 3;
constexpr double kTieEps = 1e-4;   // |u - p/q| band reported as a near tie
constexpr double kCdfEps = 1e-7;   // final draw within this fraction of a CDF boundary

// Exponentials are fp32 (expf, <= 2 ulp); every sum over the vocabulary is
// accumulated in fp64, so cumulative probabilities carry only the per-term
// exponential error, well inside kCdfEps.
struct MS {
  float m;
  double s;
};

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return {M, 0.0};
  return {M, a.s * (double)expf(a.m - M) + b.s * (double)expf(b.m - M)};
}

// Sum over the block in a fixed order (deterministic).
__device__ double block_sum(double v, double* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kBlock / 32; ++w) t += sh[w];
  __syncthreads();
  if (threadIdx.x == 0) sh[0] = t;
  __syncthreads();
  const double r = sh[0];
  __syncthreads();
  return r;
}

// (max, sum) pairs of a warp merged with few fp64 operations (GB300's fp64
// pipe is slow): the max over the warp in fp32, each lane's sum rescaled to
// it once, then an fp64 butterfly sum.  Lane 0's result is the one used.
__device__ __forceinline__ MS warp_ms(MS v) {
  float M = v.m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  double sum = (M == -INFINITY || v.m == -INFINITY) ? 0.0 : v.s * (double)expf(v.m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  return {M, sum};
}

__device__ MS block_ms(MS v, MS* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_ms(v);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  MS t{-INFINITY, 0.0};
  if (threadIdx.x == 0)
    for (int w = 0; w < kBlock / 32; ++w) t = ms_merge(t, sh[w]);
  __syncthreads();
  if (threadIdx.x == 0) sh[0] = t;
  __syncthreads();
  const MS r = sh[0];
  __syncthreads();
  return r;
}

// Inclusive prefix sum over the block's threads in a fixed order
// (deterministic): a shuffle scan inside each warp, then over the warp totals.
__device__ double block_incl_scan(double v, double* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    double w = lane < kBlock / 32 ? sh[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < kBlock / 32; o <<= 1) {
      const double n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kBlock / 32) sh[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += sh[warp - 1];
  __syncthreads();
  return v;
}

__device__ __forceinline__ void chunk_range(int c, int nchunks, int V, int& lo, int& hi) {
  const long long cs = ((long long)V + nchunks - 1) / nchunks;
  lo = (int)min((long long)V, (long long)c * cs);
  hi = (int)min((long long)V, (long long)(c + 1) * cs);
}

// ---------------------------------------------------------------- row stats

__global__ void __launch_bounds__(kBlock) row_stats_kernel(const float* __restrict__ logits, int V,
                                                           int nchunks, double* __restrict__ stats,
                                                           double* __restrict__ rowstat,
                                                           int* __restrict__ rowcnt) {
  __shared__ MS sh[kBlock / 32];
  __shared__ int s_lastrow;
  const int c = blockIdx.x, row = blockIdx.y;
  int lo, hi;
  chunk_range(c, nchunks, V, lo, hi);
  const float* l = logits + (long long)row * V;
  // Per thread: online max and a compensated (Kahan) fp32 sum of
  // exp(l - max), so its error stays near one fp32 rounding of the thread's
  // total however many terms it holds; threads and chunks then combine in
  // fp64.  (GB300's fp64 pipe is slow: one fp64 add per element would bound
  // this pass, not the bytes.)
  // (two passes over the thread's elements, the second from L1: its max,
  // then the sum, with no rescaling)
  float m = -INFINITY;
  for (int v = lo + threadIdx.x; v < hi; v += kBlock) m = fmaxf(m, __ldg(l + v));
  float sum = 0.f, comp = 0.f;
  if (m != -INFINITY) {
    for (int v = lo + threadIdx.x; v < hi; v += kBlock) {
      const float y = expf(__ldg(l + v) - m) - comp;
      const float t = sum + y;
      comp = (t - sum) - y;
      sum = t;
    }
  }
  MS a{m, (double)sum - (double)comp};
  a = block_ms(a, sh);
  if (threadIdx.x == 0) {
    stats[((long long)row * nchunks + c) * 2 + 0] = a.m;
    stats[((long long)row * nchunks + c) * 2 + 1] = a.s;
    __threadfence();
    s_lastrow = atomicAdd(&rowcnt[row], 1) == nchunks - 1;
  }
  __syncthreads();
  // the row's last chunk to finish merges the row once: (max, 1/Z)
  if (s_lastrow && threadIdx.x < 32) {
    __threadfence();
    MS t{-INFINITY, 0.0};
    for (int k = threadIdx.x; k < nchunks; k += 32) {
      const MS x{(float)__ldcg(stats + ((long long)row * nchunks + k) * 2),
                 __ldcg(stats + ((long long)row * nchunks + k) * 2 + 1)};
      t = ms_merge(t, x);
    }
    t = warp_ms(t);
    if (threadIdx.x == 0) {
      rowstat[row * 2 + 0] = (double)t.m;
      rowstat[row * 2 + 1] = 1.0 / t.s;
      rowcnt[row] = 0;
    }
  }
}

__global__ void __launch_bounds__(kBlock) softmax_norm_kernel(const float* __restrict__ logits,
                                                              float* __restrict__ probs, int V,
                                                              int nchunks,
                                                              const double* __restrict__ rowstat) {
  const int c = blockIdx.x, row = blockIdx.y;
  const float M = (float)__ldcg(rowstat + row * 2);
  const float invZ = (float)__ldcg(rowstat + row * 2 + 1);
  int lo, hi;
  chunk_range(c, nchunks, V, lo, hi);
  const float* l = logits + (long long)row * V;
  float* p = probs + (long long)row * V;
  for (int v = lo + threadIdx.x; v < hi; v += kBlock) p[v] = expf(l[v] - M) * invZ;
}

// ---------------------------------------------------------------- chain accept

struct AcceptArgs {
  const float* logits;   // [T+1][V]
  const float* q;        // [T][V]
  const int32_t* drafts;
  const float* u;        // [T+1]
  int T, V;
  const double* rowstat;  // [T+1][2] per-row (max, 1/Z)
  int nscan;             // blocks of accept_kernel == residual chunks
  double* chunk_sums;    // [nscan]
  int* counter;
  int32_t* n_acc;
  int32_t* tokens;
  int32_t* flags;        // nullable
  int* err;              // device error word
};

// Weight of token v in the final draw: residual max(0, p_j - q_j) at a
// rejection (mode 0), p_j itself (mode 1: fallback when the residual has no
// mass, only reachable through rounding), or p_T when all were accepted.
struct DrawRow {
  const float* l;
  const float* q;   // null unless mode 0
  float M;
  double invZ;
  int mode;
  __device__ __forceinline__ double w(int v) const {
    const double p = (double)expf(__ldg(l + v) - M) * invZ;
    return mode == 0 ? fmax(0.0, p - (double)__ldg(q + v)) : p;
  }
};

__global__ void __launch_bounds__(kBlock) accept_kernel(AcceptArgs a) {
  __shared__ float rowM[kMaxAcceptT + 1];
  __shared__ double rowInvZ[kMaxAcceptT + 1];
  __shared__ double shf[kBlock / 32 + 1];
  __shared__ int s_j, s_last, s_tok;
  __shared__ double s_gap;
  __shared__ int s_flag[kMaxAcceptT + 1];
  __shared__ double s_pref[kScanBlocks + 1];

  const int T = a.T, V = a.V;
  for (int r = threadIdx.x; r <= T; r += kBlock) {
    rowM[r] = (float)__ldcg(a.rowstat + r * 2);
    rowInvZ[r] = __ldcg(a.rowstat + r * 2 + 1);
  }
  __syncthreads();
  // every draft's test at once (one round of loads), then the left-to-right
  // scan for the first rejection
  for (int i = threadIdx.x; i < T; i += kBlock) {
    const int x = a.drafts[i];
    double p = 0.0, qx = 1.0;
    const bool in_range = x >= 0 && x < V;
    if (in_range) {
      p = (double)expf(a.logits[(long long)i * V + x] - rowM[i]) * rowInvZ[i];
      qx = (double)a.q[(long long)i * V + x];
    }
    const double r = qx == 0.0 ? (double)INFINITY : p / qx;
    const double ui = (double)a.u[i];
    // bit 0: accepted; bit 1: near tie; bit 2: out of range (rejected, reported)
    s_flag[i] = (ui < fmin(1.0, r) ? 1 : 0) | (fabs(ui - r) < kTieEps ? 2 : 0) | (in_range ? 0 : 4);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int j = T;
    for (int i = 0; i < T; ++i) {
      if (s_flag[i] & 4) atomicCAS(a.err, 0, kDevErrBadToken);
      if (!(s_flag[i] & 1)) {
        j = i;
        break;
      }
    }
    for (int i = 0; i < T; ++i) s_flag[i] = (i <= j && (s_flag[i] & 2)) ? 1 : 0;
    s_j = j;
  }
  __syncthreads();
  const int j = s_j;
  DrawRow dr;
  dr.l = a.logits + (long long)j * V;
  dr.q = j < T ? a.q + (long long)j * V : nullptr;
  dr.M = rowM[j];
  dr.invZ = rowInvZ[j];
  dr.mode = j < T ? 0 : 1;

  // this block's residual chunk sum
  int lo, hi;
  chunk_range(blockIdx.x, a.nscan, V, lo, hi);
  double part = 0.0;
  for (int v = lo + threadIdx.x; v < hi; v += kBlock) part += dr.w(v);
  part = block_sum(part, shf);
  if (threadIdx.x == 0) {
    a.chunk_sums[blockIdx.x] = part;
    __threadfence();
    const int old = atomicAdd(a.counter, 1);
    s_last = (old == a.nscan - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last block: the single inverse-CDF draw
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (attempt == 1) {
      // residual without mass (rounding only): draw from p_j instead
      dr.mode = 1;
      for (int c = 0; c < a.nscan; ++c) {
        int l2, h2;
        chunk_range(c, a.nscan, V, l2, h2);
        double s = 0.0;
        for (int v = l2 + threadIdx.x; v < h2; v += kBlock) s += dr.w(v);
        s = block_sum(s, shf);
        if (threadIdx.x == 0) a.chunk_sums[c] = s;
      }
      __syncthreads();
    }
    {
      // prefix of the chunk sums (nscan <= kBlock): one block-wide scan
      const double x = threadIdx.x < a.nscan ? __ldcg(a.chunk_sums + threadIdx.x) : 0.0;
      const double incl = block_incl_scan(x, shf);
      if (threadIdx.x < a.nscan) s_pref[threadIdx.x + 1] = incl;
      if (threadIdx.x == 0) s_pref[0] = 0.0;
    }
    __syncthreads();
    if (s_pref[a.nscan] > 0.0 || attempt == 1) break;
  }
  const double Z = s_pref[a.nscan];
  const double target = (double)a.u[T] * Z;
  // chosen chunk: the first with mass whose prefix passes the target (or, by
  // rounding only, the last chunk with mass)
  if (threadIdx.x == 0) {
    s_j = 0x7fffffff;
    s_last = -1;
    s_tok = 0x7fffffff;
    s_gap = 0.0;
  }
  __syncthreads();
  if (threadIdx.x < a.nscan && s_pref[threadIdx.x + 1] > s_pref[threadIdx.x]) {
    if (s_pref[threadIdx.x + 1] > target) atomicMin(&s_j, (int)threadIdx.x);
    atomicMax(&s_last, (int)threadIdx.x);
  }
  __syncthreads();
  const int cstar = s_j != 0x7fffffff ? s_j : (s_last >= 0 ? s_last : 0);
  chunk_range(cstar, a.nscan, V, lo, hi);
  const int len = hi - lo;
  const int per = (len + kBlock - 1) / kBlock;
  const int my_lo = min(hi, lo + threadIdx.x * per);
  const int my_hi = min(hi, my_lo + per);
  double sub = 0.0;
  for (int v = my_lo; v < my_hi; ++v) sub += dr.w(v);
  // this thread's starting cumulative weight: the chunk's prefix plus the
  // exclusive prefix of the threads before it
  double cum = s_pref[cstar] + (block_incl_scan(sub, shf) - sub);
  int cand = 0x7fffffff;
  double cgap = 0.0;
  for (int v = my_lo; v < my_hi; ++v) {
    const double wv = dr.w(v);
    const double nxt = cum + wv;
    if (wv > 0.0 && nxt > target) {
      cand = v;
      cgap = fmin(target - cum, nxt - target);
      atomicMin(&s_tok, v);
      break;
    }
    cum = nxt;
  }
  __syncthreads();
  if (cand != 0x7fffffff && cand == s_tok) s_gap = cgap;
  if (threadIdx.x == 0 && s_tok == 0x7fffffff) {
    // rounding: last token with mass in the chosen chunk, reported as a near tie
    int t = lo;
    for (int v = hi - 1; v >= lo; --v)
      if (dr.w(v) > 0.0) {
        t = v;
        break;
      }
    s_tok = t;
    s_gap = 0.0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.n_acc[0] = j;
    for (int i = 0; i < j; ++i) a.tokens[i] = a.drafts[i];
    a.tokens[j] = s_tok;
    if (a.flags) {
      for (int i = 0; i < T; ++i) a.flags[i] = s_flag[i];
      a.flags[T] = (s_gap < kCdfEps * Z) ? 1 : 0;
    }
    *a.counter = 0;
  }
}

// ---------------------------------------------------------------- greedy tree

struct TreeArgs {
  const float* logits;   // [T+1][V]
  const int32_t* drafts;
  const int32_t* parent;
  int T, V, nchunks;
  int chunk;             // tokens per block, a multiple of 4
  int vec;               // rows start on 16-byte boundaries
  float* argval;         // [T+1][nchunks]
  int* argidx;
  int* counter;
  int32_t* path_len;
  int32_t* tokens;
  int32_t* nodes;
  int* err;
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kBlock) tree_kernel(TreeArgs a) {
  __shared__ float shv[kBlock / 32];
  __shared__ int shi[kBlock / 32];
  __shared__ int s_last;
  __shared__ int amax[kMaxAcceptT + 1];
  __shared__ int depth[kMaxAcceptT];
  __shared__ unsigned char ok[kMaxAcceptT];
  __shared__ int s_draft[kMaxAcceptT];
  __shared__ int s_par[kMaxAcceptT];
  __shared__ float s_mv[kMergeBatch];
  __shared__ int s_mi[kMergeBatch];

  const int c = blockIdx.x, row = blockIdx.y;
  const int lo = c * a.chunk;
  const int hi = min(a.V, lo + a.chunk);
  const float* l = a.logits + (long long)row * a.V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  // four tokens per thread and step, 16-byte loads when the rows are
  // aligned, unrolled so that several loads are in flight per thread
#pragma unroll 4
  for (int v0 = lo + 4 * threadIdx.x; v0 < hi; v0 += 4 * kBlock) {
    float x[4];
    if (a.vec && v0 + 3 < hi) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(l + v0));
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = v0 + j < hi ? __ldg(l + v0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (v0 + j < hi && better(x[j], v0 + j, bv, bi)) {
        bv = x[j];
        bi = v0 + j;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    shv[warp] = bv;
    shi[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kBlock / 32; ++w)
      if (better(shv[w], shi[w], bv, bi)) {
        bv = shv[w];
        bi = shi[w];
      }
    a.argval[row * a.nchunks + c] = bv;
    a.argidx[row * a.nchunks + c] = bi;
    __threadfence();
    const int old = atomicAdd(a.counter, 1);
    s_last = (old == (int)(gridDim.x * gridDim.y) - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int T = a.T;
  // the drafts and parents into shared memory at once; the chunk partials
  // in batches of rows, every load of a batch in flight together, then one
  // warp per row merges the row's chunks from shared memory
  for (int i = threadIdx.x; i < T; i += kBlock) {
    s_draft[i] = a.drafts[i];
    s_par[i] = a.parent[i];
  }
  const int nc = a.nchunks;
  const int batch_rows = kMergeBatch / nc;
  for (int r0 = 0; r0 <= T; r0 += batch_rows) {
    const int r1 = min(T + 1, r0 + batch_rows);
    for (int e = threadIdx.x; e < (r1 - r0) * nc; e += kBlock) {
      s_mv[e] = __ldcg(a.argval + r0 * nc + e);
      s_mi[e] = __ldcg(a.argidx + r0 * nc + e);
    }
    __syncthreads();
    for (int r = r0 + warp; r < r1; r += kBlock / 32) {
      float v = -INFINITY;
      int idx = 0x7fffffff;
      for (int k = lane; k < nc; k += 32) {
        const float cv = s_mv[(r - r0) * nc + k];
        const int ci = s_mi[(r - r0) * nc + k];
        if (better(cv, ci, v, idx)) {
          v = cv;
          idx = ci;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (better(ov, oi, v, idx)) {
          v = ov;
          idx = oi;
        }
      }
      if (lane == 0) amax[r] = idx == 0x7fffffff ? 0 : idx;   // all-NaN row: token 0
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int best = -1;
    for (int i = 0; i < T; ++i) {
      int par = s_par[i];
      int row_i, d;
      bool pok;
      if (par < -1 || par >= i) {   // not a topological parent: node rejected, reported
        atomicCAS(a.err, 0, kDevErrBadParent);
        ok[i] = 0;
        depth[i] = 1;
        continue;
      }
      if (par < 0) {
        pok = true;
        row_i = 0;
        d = 1;
      } else {
        pok = ok[par] != 0;
        row_i = par + 1;
        d = depth[par] + 1;
      }
      ok[i] = (pok && s_draft[i] == amax[row_i]) ? 1 : 0;
      depth[i] = d;
      if (ok[i] && (best < 0 || d > depth[best])) best = i;
    }
    const int len = best < 0 ? 0 : depth[best];
    int n = best;
    for (int k = len - 1; k >= 0; --k) {
      a.nodes[k] = n;
      a.tokens[k] = s_draft[n];
      n = s_par[n];
    }
    a.tokens[len] = amax[best + 1];
    a.path_len[0] = len;
    *a.counter = 0;
  }
}

int stat_chunks(const spec_ctx* ctx, int rows, int V) {
  long long want = (4LL * ctx->num_sms + rows - 1) / rows;
  long long by_size = ((long long)V + 1023) / 1024;
  long long c = want < by_size ? want : by_size;
  if (c < 1) c = 1;
  if (c > kAcceptChunks) c = kAcceptChunks;
  return (int)c;
}

}  // namespace

int launch_softmax(spec_ctx* ctx, const float* logits, float* probs, int rows, int V,
                   cudaStream_t s) {
  const int nc = stat_chunks(ctx, rows, V);
  dim3 g(nc, rows);
  row_stats_kernel<<<g, kBlock, 0, s>>>(logits, V, nc, ctx->acc_stats, ctx->acc_rowstat, ctx->acc_rowcnt);
  int rc = check_cuda(cudaGetLastError(), "row_stats launch");
  if (rc) return rc;
  softmax_norm_kernel<<<g, kBlock, 0, s>>>(logits, probs, V, nc, ctx->acc_rowstat);
  return check_cuda(cudaGetLastError(), "softmax_norm launch");
}

int launch_accept(spec_ctx* ctx, const float* logits, const float* q, const int32_t* drafts,
                  const float* u, int T, int V, int32_t* n_acc, int32_t* tokens, int32_t* flags,
                  cudaStream_t s) {
  const int rows = T + 1;
  const int nc = stat_chunks(ctx, rows, V);
  dim3 g(nc, rows);
  row_stats_kernel<<<g, kBlock, 0, s>>>(logits, V, nc, ctx->acc_stats, ctx->acc_rowstat, ctx->acc_rowcnt);
  int rc = check_cuda(cudaGetLastError(), "row_stats launch");
  if (rc) return rc;
  AcceptArgs a;
  a.logits = logits;
  a.q = q;
  a.drafts = drafts;
  a.u = u;
  a.T = T;
  a.V = V;
  a.rowstat = ctx->acc_rowstat;
  long long ns = ((long long)V + 1023) / 1024;
  if (ns > kScanBlocks) ns = kScanBlocks;
  if (ns < 1) ns = 1;
  a.nscan = (int)ns;
  a.chunk_sums = ctx->acc_chunks;
  a.counter = ctx->acc_counters + 0;
  a.n_acc = n_acc;
  a.tokens = tokens;
  a.flags = flags;
  a.err = ctx->err;
  accept_kernel<<<a.nscan, kBlock, 0, s>>>(a);
  return check_cuda(cudaGetLastError(), "accept launch");
}

int launch_accept_tree(spec_ctx* ctx, const float* logits, const int32_t* drafts,
                       const int32_t* parent, int T, int V, int32_t* path_len, int32_t* tokens,
                       int32_t* nodes, cudaStream_t s) {
  const int rows = T + 1;
  TreeArgs a;
  a.logits = logits;
  a.drafts = drafts;
  a.parent = parent;
  a.T = T;
  a.V = V;
  // one full wave of resident blocks in all, at least 1024 tokens a block
  static int per_sm = 0;
  if (per_sm == 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, tree_kernel, kBlock, 0) != cudaSuccess || b < 1) b = 4;
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
  a.argval = ctx->acc_argval;
  a.argidx = ctx->acc_argmax;
  a.counter = ctx->acc_counters + 1;
  a.path_len = path_len;
  a.tokens = tokens;
  a.nodes = nodes;
  a.err = ctx->err;
  dim3 g(a.nchunks, rows);
  tree_kernel<<<g, kBlock, 0, s>>>(a);
  return check_cuda(cudaGetLastError(), "tree launch");
}

// ---------------------------------------------------------------- without allocation
//
// The same two launches as launch_accept, with their scratch taken from a
// fixed array in this module's static device memory instead of a context's
// workspace, for callers that cannot allocate device memory (see
// spec_accept_noalloc in the public header).  Up to kNoAllocMaxT drafts.

namespace {

constexpr int kNoAllocMaxT = 64;
constexpr size_t kNoAllocStatsBytes = sizeof(double) * 2 * (size_t)(kNoAllocMaxT + 1) * kAcceptChunks;
constexpr size_t kNoAllocChunkBytes = sizeof(double) * kScanBlocks;
constexpr size_t kNoAllocRowBytes = sizeof(double) * 2 * (kNoAllocMaxT + 1);
// stats | chunk sums | row (max, 1/Z) | arrival counter, error word, per-row
// counters (these last start at zero)
constexpr int kNoAllocZeroInts = 2 + kNoAllocMaxT + 1;
constexpr size_t kNoAllocScratchBytes =
    kNoAllocStatsBytes + kNoAllocChunkBytes + kNoAllocRowBytes + kNoAllocZeroInts * sizeof(int);

static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct NoAllocSetup {
  unsigned char* scratch;   // device address of g_accept_scratch
  int num_sms;
};

}  // namespace

// Device address of the static scratch and the SM count of the current
// device, looked up once per device (with that device current).
static int noalloc_setup(NoAllocSetup* out) {
  static std::mutex mu;
  static NoAllocSetup table[kMaxDevices] = {};
  int dev = -1;
  int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kMaxDevices) return set_error(SPEC_ERR_ARG, "device %d outside 0..%d", dev, kMaxDevices - 1);
  std::lock_guard<std::mutex> lock(mu);
  if (!table[dev].scratch) {
    int major = 0, minor = 0, nsm = 0;
    rc = check_cuda(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "device attribute");
    if (rc) return rc;
    rc = check_cuda(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "device attribute");
    if (rc) return rc;
    if (major != 10 || minor != 3)
      return set_error(SPEC_ERR_CUDA, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
    rc = check_cuda(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev), "device attribute");
    if (rc) return rc;
    void* p = nullptr;
    rc = check_cuda(cudaGetSymbolAddress(&p, g_accept_scratch), "cudaGetSymbolAddress(acceptance scratch)");
    if (rc) return rc;
    table[dev].scratch = static_cast<unsigned char*>(p);
    table[dev].num_sms = nsm;
  }
  *out = table[dev];
  return SPEC_OK;
}

int launch_accept_noalloc(const float* logits, const float* q, const int32_t* drafts, const float* u,
                          int T, int V, int32_t* n_acc, int32_t* tokens, int32_t* flags,
                          int32_t* status, cudaStream_t s) {
  if (T > kNoAllocMaxT)
    return set_error(SPEC_ERR_SHAPE,
                     "spec_accept_noalloc takes at most %d drafts (its static scratch is sized for "
                     "that); T=%d -- use spec_accept with a context instead",
                     kNoAllocMaxT, T);
  NoAllocSetup su;
  int rc = noalloc_setup(&su);
  if (rc) return rc;
  double* stats = reinterpret_cast<double*>(su.scratch);
  double* chunks = reinterpret_cast<double*>(su.scratch + kNoAllocStatsBytes);
  double* rowstat = reinterpret_cast<double*>(su.scratch + kNoAllocStatsBytes + kNoAllocChunkBytes);
  int* counter = reinterpret_cast<int*>(su.scratch + kNoAllocStatsBytes + kNoAllocChunkBytes + kNoAllocRowBytes);
  int* err = counter + 1;
  int* rowcnt = counter + 2;
  // the arrival counters and the error word must start at zero
  rc = check_cuda(cudaMemsetAsync(counter, 0, kNoAllocZeroInts * sizeof(int), s), "clear acceptance scratch");
  if (rc) return rc;

  const int rows = T + 1;
  long long want = (4LL * su.num_sms + rows - 1) / rows;
  long long by_size = ((long long)V + 1023) / 1024;
  long long nc = want < by_size ? want : by_size;
  if (nc < 1) nc = 1;
  if (nc > kAcceptChunks) nc = kAcceptChunks;
  dim3 g((unsigned)nc, rows);
  row_stats_kernel<<<g, kBlock, 0, s>>>(logits, V, (int)nc, stats, rowstat, rowcnt);
  rc = check_cuda(cudaGetLastError(), "row_stats launch");
  if (rc) return rc;
  AcceptArgs a;
  a.logits = logits;
  a.q = q;
  a.drafts = drafts;
  a.u = u;
  a.T = T;
  a.V = V;
  a.rowstat = rowstat;
  long long ns = ((long long)V + 1023) / 1024;
  if (ns > kScanBlocks) ns = kScanBlocks;
  if (ns < 1) ns = 1;
  a.nscan = (int)ns;
  a.chunk_sums = chunks;
  a.counter = counter;
  a.n_acc = n_acc;
  a.tokens = tokens;
  a.flags = flags;
  a.err = err;
  accept_kernel<<<a.nscan, kBlock, 0, s>>>(a);
  rc = check_cuda(cudaGetLastError(), "accept launch");
  if (rc) return rc;
  if (status)
    rc = check_cuda(cudaMemcpyAsync(status, err, sizeof(int), cudaMemcpyDeviceToDevice, s),
                    "copy acceptance status");
  return rc;
}

}  // namespace sv
