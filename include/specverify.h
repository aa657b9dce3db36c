/*
 * specverify.h -- C ABI of the speculative-decoding verification step on one
 * NVIDIA GB300 (sm_103a).
 *
 * The verify step scores a block of T drafted tokens in one target-model pass,
 * so every low-bit weight read from memory is used for T tokens instead of one
 * ("Speculative Decoding Clearly Explained", the cat-sat walkthrough; "Karpathy's
 * Trick for Faster Local LLMs Finally Has Proper Tooling", section "Producing
 * several tokens from one model pass": 16 rows of work instead of 1).  The pass
 * is a group-quantised weight GEMM followed by the acceptance rule.
 *
 * Conventions for every entry point
 *  - Status is returned by value: SPEC_OK (0) or a negative SPEC_ERR_* code.
 *    Nothing is thrown across the ABI.  spec_last_error() returns a
 *    thread-local text for the last failure on the calling thread.
 *  - All tensor pointers are DEVICE pointers on the context's device, owned by
 *    the caller.  They must stay valid until the work on `stream` completes.
 *    Every pointer must be 16-byte aligned unless stated otherwise.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls only enqueue work; results are valid once the caller synchronises.
 *  - Shapes and arguments are checked on the host before anything is launched;
 *    a rejected call launches nothing.
 *  - A context owns a device workspace (split-K partial sums, tile counters,
 *    rotated activations, acceptance scratch) and a device error word.  One
 *    context must not be used by two streams at the same time: calls that
 *    overlap on the GPU would race on the workspace.
 *  - Device-side failures (a bounded wait that timed out) set the context's
 *    sticky error word; spec_sync_status() reports and clears it.
 *
 * Storage layouts ("Karpathy's Trick ...", section "How Uzu optimizes bytes
 * and tokens per pass": 4-bit asymmetric Medium tier, 8-bit symmetric Large
 * tier, one scale shared by every value of a group; the byte layouts are this
 * library's own):
 *   int4 codes   uint8 [N][K/2]   row n as little-endian 32-bit words, one per
 *                                 8 consecutive k: nibble p (from the least
 *                                 significant end) of word w holds
 *                                 k = 8w + 2*(p % 4) + p / 4, i.e. the bytes
 *                                 carry (k0|k2<<4), (k4|k6<<4), (k1|k3<<4),
 *                                 (k5|k7<<4) -- one mask turns a pair of
 *                                 nibbles into an fp16 pair
 *   int4 scales  fp16  [K/g][N]   one row per quantisation group of g
 *                                 consecutive k
 *   int4 zeros   uint8 [K/g][N/2] uint4 zero points, low nibble = even n
 *   int8 codes   int8  [N][K]     values -127..127 (-128 is read as -128)
 *   int8 scales  fp16  [N] (g == 0, per output channel) or [K/g][N]
 *   activations  bf16  [T][K]     row-major
 *   outputs      bf16 or fp32 [T][N] row-major
 *   dequantised weight: w[n][k] = (code - zero) * scale (int4),
 *                       w[n][k] = code * scale (int8)
 *   GEMM: y[t][n] = sum_k x[t][k] * w[n][k], fp32 accumulation.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spec_ctx spec_ctx;

enum spec_status {
  SPEC_OK = 0,
  SPEC_ERR_ARG = -1,      /* null or misaligned pointer, bad enum value        */
  SPEC_ERR_SHAPE = -2,    /* unsupported size or divisibility                  */
  SPEC_ERR_ARCH = -3,     /* the device is not sm_103                          */
  SPEC_ERR_CUDA = -4,     /* a CUDA runtime/driver call failed                 */
  SPEC_ERR_OOM = -5,      /* workspace allocation failed or is too small       */
  SPEC_ERR_TIMEOUT = -6,  /* a bounded device-side wait ran out (sticky)       */
  SPEC_ERR_NUMERIC = -7   /* reserved: no call of this version reports it      */
};

enum spec_dtype { SPEC_DTYPE_BF16 = 0, SPEC_DTYPE_F32 = 1 };

enum spec_quant { SPEC_QUANT_W4 = 0, SPEC_QUANT_W8 = 1 };

/* Library version, (major << 16) | minor. */
int spec_version(void);

/* Thread-local description of the last failure on this thread ("" if none). */
const char* spec_last_error(void);

/* Create a context on `device` (must be an sm_103 GPU, else SPEC_ERR_ARCH).
 * workspace_bytes = 0 picks the default (enough for T <= 64, K <= 32768 and
 * any N up to 2^22).  The context allocates its workspace with cudaMalloc and
 * zeroes it.  On success *out receives the context. */
int spec_create(int device, size_t workspace_bytes, spec_ctx** out);

/* Free the context and its workspace.  NULL is accepted. */
int spec_destroy(spec_ctx* ctx);

/* Synchronise `stream`, then read and clear the context's device error word.
 * Returns SPEC_OK or the first device-side error recorded since the last call:
 * SPEC_ERR_TIMEOUT when a bounded wait ran out, SPEC_ERR_ARG when a draft token
 * (spec_accept, spec_accept_gumbel) or parent index (spec_accept_tree) read on
 * the device was out of range (that draft/node was treated as rejected).  After an error the
 * split-K counters and partial sums are re-zeroed so the context is usable
 * again. */
int spec_sync_status(spec_ctx* ctx, void* stream);

/* W4A16 verify GEMM ("How Uzu optimizes bytes and tokens per pass": Medium
 * checkpoint, 4-bit asymmetric integer weights).
 *   y[t][n] = sum_k x'[t][k] * (code[n][k] - zero[k/g][n]) * scale[k/g][n]
 * x' = x, or, when signs != NULL and hadamard_block > 0, the block random
 * Hadamard rotation of x (see fwht_rotate; the weights are taken as stored
 * already rotated), computed in fp32; signs must then be 16-byte aligned.
 * Sizes: 1 <= T <= 64 (T <= 32 with rotation); N % 32 == 0; K % 64 == 0,
 * K <= 32768; group_size a power of two >= 64 with K % group_size == 0.
 * y_dtype is SPEC_DTYPE_BF16 or SPEC_DTYPE_F32.
 * Numerics depend on the context's GEMM engine (spec_set_gemm_engine):
 *  - split engine (the default): code - zero enters the tensor cores
 *    exactly (a bf16 integer) with the bf16 activations as given, each 64-k
 *    group is summed in fp32 and its scale applied in fp32; the result is
 *    the exact sum up to fp32 rounding.  A rotation is a separate launch on
 *    the same stream whose result is rounded once to bf16.
 *  - stack engine: each weight (code - zero) * scale is rounded once to
 *    fp16 (the difference is exact, the product rounded); the activations
 *    enter the tensor cores as fp16 (bf16 magnitudes from 2^-10 to 65504
 *    convert exactly; smaller ones round to fp16's subnormal grid, larger
 *    ones become infinite); the products are summed in fp32.  The error is
 *    that of the fp16 weights, about 1e-3 * RMS(y) at its largest over 10^6
 *    outputs.  A rotation runs inside the same launch, rounded once to fp16.
 * Either way a bf16 output adds its own final rounding. */
int qgemm_w4a16(spec_ctx* ctx, const uint8_t* qcodes, const uint16_t* scales,
                const uint8_t* zeros, int group_size, const uint16_t* x, void* y,
                int y_dtype, int T, int N, int K, const int8_t* signs,
                int hadamard_block, void* stream);

/* W8A16 verify GEMM ("How Uzu optimizes bytes and tokens per pass": Large
 * checkpoint, 8-bit symmetric quantisation, no zero point).
 *   y[t][n] = sum_k x'[t][k] * code[n][k] * scale
 * scale = scale[n] when group_size == 0, else scale[k/g][n] (group_size a
 * power of two >= 64).  Per-channel scales: the int8 codes enter the tensor
 * cores exactly (bf16 holds -127..127) with the bf16 activations as given,
 * and the scale multiplies the fp32 sum.  A rotated activation is rounded
 * once to bf16 (split engine) or enters as the sum of two bf16 values, the
 * rounded value and its remainder (stack engine, which adds no rounding).
 * Grouped scales: the split engine sums each 64-k group in fp32 and applies
 * its scale in fp32; the stack engine rounds code * scale once to fp16 and
 * takes fp16 activations, as in qgemm_w4a16.  Rotation and sizes as
 * qgemm_w4a16, except N % 8 == 0 suffices and per-channel K may reach 2^20
 * (32768 with rotation). */
int qgemm_w8a16(spec_ctx* ctx, const int8_t* qcodes, const uint16_t* scales,
                int group_size, const uint16_t* x, void* y, int y_dtype, int T,
                int N, int K, const int8_t* signs, int hadamard_block,
                void* stream);

/* One GEMM of a stack (see qgemm_stack_create).  Fields as the arguments of
 * qgemm_w4a16 (quant SPEC_QUANT_W4) or qgemm_w8a16 (SPEC_QUANT_W8; zeros is
 * ignored), plus wait_prev: 1 = this GEMM reads its activations (and writes
 * its outputs) only after every earlier GEMM of the stack has written all of
 * its outputs, as if each GEMM were a separate call on one stream; 0 = it
 * does not depend on the GEMMs before it (for example q, k and v projections
 * of one input).  The first entry's wait_prev is ignored: the launch itself
 * follows the previous work on its stream. */
typedef struct spec_gemm_desc {
  int quant;
  const void* qcodes;
  const uint16_t* scales;
  const uint8_t* zeros;
  int group_size;
  const uint16_t* x;
  void* y;
  int y_dtype;
  int T, N, K;
  const int8_t* signs;
  int hadamard_block;
  int wait_prev;
} spec_gemm_desc;

typedef struct spec_gemm_stack spec_gemm_stack;

/* A stack of verify GEMMs: the weight pass of the verify step, every
 * projection of every layer in order ("Karpathy's Trick ...", section "Why
 * batch-one decoding is memory-bound": one pass streams every weight once,
 * so the pass is bounded by memory bandwidth).  With the split engine (the
 * default) qgemm_stack_run enqueues one launch per GEMM (two for a rotated
 * one), each GEMM following the previous one as separate calls would; with
 * the stack engine it is one persistent launch that keeps the weight stream
 * running from one GEMM into the next: a GEMM that waits for its
 * predecessors' outputs (wait_prev) waits on the device while the weights
 * after it keep streaming in.
 * qgemm_stack_create checks and records n descriptors (1 <= n <= 1024); the
 * descriptors' pointers and sizes are fixed from then on (the tensors must
 * stay allocated while the stack is used).  Rules beyond each GEMM's own:
 * one quant for all entries; at most 3 consecutive entries (after the
 * first) with wait_prev = 0.
 * The stack holds a small device array (cudaMalloc at creation) and belongs
 * to `ctx`.  qgemm_stack_run enqueues the whole stack on `stream` with the
 * context's current engine (its launches may be captured in a CUDA graph);
 * the results are those of calling the GEMMs one by one.  qgemm_stack_destroy frees the
 * stack (NULL accepted). */
int qgemm_stack_create(spec_ctx* ctx, const spec_gemm_desc* descs, int n,
                       spec_gemm_stack** out);
int qgemm_stack_run(spec_ctx* ctx, const spec_gemm_stack* stack, void* stream);
int qgemm_stack_destroy(spec_gemm_stack* stack);

/* Tuning of the GEMMs' weight stream on this context: each CTA keeps the L2
 * prefetch of its upcoming weight boxes `lead` stages ahead of its
 * shared-memory loads, and up to `lead_when_full` stages ahead while its
 * shared-memory ring is full (0 <= lead <= lead_when_full <= 256).  Results
 * do not depend on it.  Defaults 4 and 16 (or the environment variables
 * SPEC_PREFETCH_LEAD and SPEC_PREFETCH_LEAD_FULL at spec_create). */
int spec_set_stream_prefetch(spec_ctx* ctx, int lead, int lead_when_full);

/* The kernel design that runs this context's verify GEMMs (qgemm_w4a16,
 * qgemm_w8a16, qgemm_stack_run); the results agree within the numerics
 * stated at qgemm_w4a16.
 *  SPEC_GEMM_ENGINE_SPLIT: one launch per GEMM, its (tile, 256-k stage)
 *    units spread evenly over one CTA per SM, a tile cut between CTAs summed
 *    in fp32 and finished by its last contributor; consecutive launches
 *    overlap (each starts streaming weights while its predecessor ends).
 *  SPEC_GEMM_ENGINE_STACK: one persistent launch per call or stack, with
 *    rotations and activation conversion inside the launch.
 *  SPEC_GEMM_ENGINE_AUTO (the default): the split engine, which measured
 *    faster for every workload of the verify step on GB300.
 * Returns SPEC_ERR_ARG for any other value.  Applies to launches enqueued
 * after the call. */
#define SPEC_GEMM_ENGINE_AUTO 0
#define SPEC_GEMM_ENGINE_SPLIT 1
#define SPEC_GEMM_ENGINE_STACK 2
int spec_set_gemm_engine(spec_ctx* ctx, int engine);

/* Test hook for the failure path of the GEMMs' bounded waits (not for
 * production use): the next GEMM launch on this context (qgemm_w4a16,
 * qgemm_w8a16 or qgemm_stack_run) gives every wait a limit of
 * wait_limit_ns (1e5 .. 2e9 ns) instead of the default 2 s, and, when
 * skip_unit >= 0, its CTA 0 never loads the weights of its skip_unit-th
 * stage (if it owns that many), so the waits for that stage run out.  The kernel then records
 * SPEC_ERR_TIMEOUT, stops (the stack engine: every CTA; the split engine:
 * the CTAs whose waits run out, while the others finish), lets its copies
 * and MMAs complete, frees its tensor memory and returns; spec_sync_status reports the error
 * and resets the workspace, after which the context is usable again.  The
 * hook applies to one launch only. */
int spec_test_stall(spec_ctx* ctx, int skip_unit, uint64_t wait_limit_ns);

/* Block-diagonal random Hadamard rotation ("How Uzu optimizes bytes and tokens
 * per pass": random sign flips applied before the mixing, +1/-1 entries and
 * one overall scale, each block mixed on its own, exactly reversible):
 *   y[t][bB:(b+1)B] = (1/sqrt(B)) * H_B * (s[bB:(b+1)B] .* x[t][bB:(b+1)B])
 * H_B is the Sylvester Hadamard matrix in natural order.  B = block is a power
 * of two in [32, 1024], K % B == 0, signs int8 [K] of +1/-1 (any nonzero
 * negative value counts as -1).  x, y bf16 [T][K]; y may alias x.  fp32 math,
 * one rounding to bf16.  1 <= T. */
int fwht_rotate(spec_ctx* ctx, const uint16_t* x, uint16_t* y, int T, int K,
                const int8_t* signs, int block, void* stream);

/* Row softmax ("Speculative Decoding Clearly Explained": p is the target
 * model's probability): probs[i][v] = exp(l[i][v] - max_i) / sum_w exp(l[i][w]
 * - max_i) for rows x V fp32 logits.  1 <= rows <= 4096, 1 <= V <= 2^26.
 * logits/probs need only 4-byte alignment. */
int spec_softmax(spec_ctx* ctx, const float* logits, float* probs, int rows,
                 int V, void* stream);

/* Chain acceptance ("Speculative Decoding Clearly Explained": accept draft i
 * with probability min(1, p/q) left to right, stop at the first rejection,
 * sample the replacement from normalize(max(0, p - q)); if every draft is
 * accepted the target supplies one more token).
 *   target_logits fp32 [T+1][V]: row i scores draft i, row T follows the last
 *   draft_probs   fp32 [T][V]   (used as given, not renormalised)
 *   draft_tokens  int32 [T]     in [0, V)
 *   uniforms      fp32 [T+1]    in [0, 1): u[i] tests draft i, u[T] drives the
 *                               single final draw (inverse CDF in ascending
 *                               token order)
 * Draft i is accepted iff u[i] < min(1, p_i(x_i) / q_i(x_i)) (q = 0 counts as
 * +inf).  Outputs (device): n_accepted int32 [1]; out_tokens int32 [T+1], the
 * first n_accepted+1 entries valid; near_tie_flags (nullable) int32 [T+1]:
 * entry i < T is 1 when |u[i] - p/q| < 1e-4 at an evaluated position, entry T
 * is 1 when the final draw lies within 1e-7 (relative) of a cumulative
 * boundary.  0 <= T <= 256, 1 <= V <= 2^26.  Pointers need 4-byte alignment. */
int spec_accept(spec_ctx* ctx, const float* target_logits,
                const float* draft_probs, const int32_t* draft_tokens,
                const float* uniforms, int T, int V, int32_t* n_accepted,
                int32_t* out_tokens, int32_t* near_tie_flags, void* stream);

/* spec_accept without a context and without allocating device memory.
 * The pages describe nothing like it: it exists for callers that cannot
 * allocate -- a process whose device memory is reserved by another
 * allocator, a caller that must avoid the device-wide synchronisation that
 * cudaMalloc/cudaFree can bring, or a component that owns no spec_ctx.
 * The scratch the two acceptance kernels need (per-row softmax partials,
 * residual chunk sums, an arrival counter and an error word, 68 KB) is a
 * fixed array in the library's static device memory, which is why T is
 * limited to 64 drafts here (a larger T is rejected with SPEC_ERR_SHAPE);
 * nothing is allocated and nothing is freed.
 * Runs on the calling thread's current device.  The first call on a device
 * looks up the scratch's device address (cudaGetSymbolAddress) and the SM
 * count; make that first call before any stream capture.  Every call clears
 * the counter and error word on `stream` before its kernels.
 * All calls on one device share the scratch: calls whose kernels may
 * overlap (different streams without ordering between them, or several host
 * threads) race and give wrong results -- keep them ordered on one stream.
 * Arguments, layouts, sizes (except T <= 64) and results are those of
 * spec_accept.  device_status (nullable, device int32 [1]) receives 0, or 2
 * when a draft token was outside [0, V) (that draft then counts as
 * rejected); spec_sync_status does not see this entry's errors. */
int spec_accept_noalloc(const float* target_logits, const float* draft_probs,
                        const int32_t* draft_tokens, const float* uniforms,
                        int T, int V, int32_t* n_accepted, int32_t* out_tokens,
                        int32_t* near_tie_flags, int32_t* device_status,
                        void* stream);

/* Greedy tree acceptance.  Sources: "Karpathy's Trick ...", section "Issue
 * with parallel draft generation" (the target scores a whole draft tree in
 * one pass and keeps the deepest root path it agrees with) and "Local LLM 4x
 * Faster ..." (one verification pass over the tree).
 *   target_logits fp32 [T+1][V]: row 0 scores the children of the root (the
 *                  last committed token), row i+1 the children of node i
 *   draft_tokens  int32 [T]; parent int32 [T] with parent[i] < i, -1 = child
 *                  of the root
 * Node i is accepted iff its parent is accepted (the root always is) and its
 * token equals the largest-logit token of the row that scores it (ties go to
 * the smallest token id).  The deepest accepted node wins (ties to the
 * smallest node index).  Outputs (device): path_len int32 [1]; out_tokens
 * int32 [T+1] = the path's tokens then the bonus token (the argmax of the row
 * that follows the last path node, row 0 for an empty path); path_nodes
 * int32 [T], the first path_len entries valid.  1 <= T <= 256,
 * 1 <= V <= 2^26.  Pointers need 4-byte alignment. */
int spec_accept_tree(spec_ctx* ctx, const float* target_logits,
                     const int32_t* draft_tokens, const int32_t* parent, int T,
                     int V, int32_t* path_len, int32_t* out_tokens,
                     int32_t* path_nodes, void* stream);

/* Shared-seed sampling and acceptance (the trymirai post feed, the post with
 * the "random number from 1 to 10" example: sample the speculator and the
 * LLM with the same seed through the Gumbel-max trick, so that matching
 * distributions give matching tokens).
 *
 * Noise: the uniform of token v at draft position p is word v mod 4 of
 * Philox4x32-10 (Salmon et al., SC 2011) at counter (v div 4, p mod 2^32,
 * p div 2^32, 0) under key (seed mod 2^32, seed div 2^32), a word w giving
 * u = (2 floor(w / 2^9) + 1) / 2^24.  The sample of a row is
 * argmax_v (logit_v - log(-log u_v)), computed in fp32, equal values to the
 * smallest token id.  A row's near-tie flag is 1 when its best value exceeds
 * every other token's by less than 1e-4 (another summation order could pick
 * the runner-up there).
 *
 * spec_gumbel_sample: the drafter's side.
 *   logits fp32 [rows][V] (device), row r sampled at position + r.
 *   out_tokens int32 [rows]; near_tie_flags nullable int32 [rows] (device).
 *   1 <= rows <= 257, 1 <= V <= 2^26.  Pointers need 4-byte alignment.
 *
 * spec_accept_gumbel: the verifier's side.
 *   target_logits fp32 [T+1][V]: row i scores draft position i, row T follows
 *                 the last draft; row i is sampled at position + i.
 *   draft_tokens  int32 [T] (nullable when T = 0), drawn by the speculator
 *                 under the same seed and positions.
 * Drafts are accepted left to right while each equals the target's sample at
 * its position; the first position that differs, or position T, emits the
 * target's sample.  Outputs (device): n_accepted int32 [1]; out_tokens int32
 * [T+1], the first n_accepted + 1 valid; near_tie_flags nullable int32 [T+1].
 * A draft outside [0, V) never matches and is reported by spec_sync_status.
 * 0 <= T <= 256, 1 <= V <= 2^26.  One launch; the context's sampling
 * partials are shared by both entries, so keep calls on one context ordered
 * on one stream. */
int spec_gumbel_sample(spec_ctx* ctx, const float* logits, int rows, int V,
                       uint64_t seed, uint64_t position, int32_t* out_tokens,
                       int32_t* near_tie_flags, void* stream);
int spec_accept_gumbel(spec_ctx* ctx, const float* target_logits,
                       const int32_t* draft_tokens, int T, int V, uint64_t seed,
                       uint64_t position, int32_t* n_accepted,
                       int32_t* out_tokens, int32_t* near_tie_flags,
                       void* stream);

/* Dequantised weights as fp32 [N][K] (exact: (code - zero) * scale and
 * code * scale both fit in fp32), for checking a packed checkpoint.  Layouts
 * and size rules as the GEMMs (int4 only needs N % 2 == 0 and K % 8 == 0). */
int qdequant_w4(spec_ctx* ctx, const uint8_t* qcodes, const uint16_t* scales,
                const uint8_t* zeros, int group_size, int N, int K, float* w,
                void* stream);
int qdequant_w8(spec_ctx* ctx, const int8_t* qcodes, const uint16_t* scales,
                int group_size, int N, int K, float* w, void* stream);

/* Checkpoint conversion, on the host (no context, no GPU, no stream): int4
 * codes packed in plain order -- byte i of row n holds k = 2i in its low
 * nibble and k = 2i + 1 in its high nibble, uint8 [N][K/2] -- rewritten in
 * this library's int4 code layout (see "Storage layouts" above).  Every 4
 * source bytes (8 consecutive k) map to the same 4 destination bytes, so dst
 * may equal src (in place); any other overlap is not allowed.  src and dst
 * are host pointers of N * K / 2 bytes owned by the caller.  Returns
 * SPEC_ERR_ARG for a null pointer, SPEC_ERR_SHAPE unless N >= 1, K >= 8 and
 * K % 8 == 0. */
int spec_repack_w4_codes(const uint8_t* src, uint8_t* dst, int N, int K);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
