// The C ABI: context life cycle, argument checks, workspace layout and the
// dispatch of each entry point to its kernels.  Every check runs on the host
// before anything is launched; nothing throws across the ABI.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.hpp"
#include "ptx.cuh"

namespace sv {

namespace {
thread_local char g_err[512] = "";

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Make the context's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_err[0] = '\0'; }

int check_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SPEC_OK;
  return set_error(SPEC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0,
                   uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return set_error(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) dims=%llu,%llu box=%u,%u",
                     (int)r, (unsigned long long)dim0, (unsigned long long)dim1, box0, box1);
  return SPEC_OK;
}

}  // namespace sv

using namespace sv;

namespace {

// Workspace layout (bytes, each region 256-aligned).
struct WsLayout {
  size_t err, abort_all, exit_cnt, split_cnt, partials, done, rot_done, tile_counters, split_slots, xprep,
      stats, chunks, argidx,
      argval, acc_counters, rowstat, rowcnt, gbest, gidx, gsecond, total;
};

WsLayout layout_for(int num_sms) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  L.err = take(sizeof(int));
  L.abort_all = take(sizeof(int));
  L.exit_cnt = take(sizeof(int));
  L.split_cnt = take(sizeof(int) * (size_t)kSplitKeys * num_sms * kGemmWorkers);
  L.partials = take(sizeof(float) * (size_t)kPartialSlotFloats * kSplitKeys * num_sms);
  L.done = take(sizeof(int) * (size_t)kMaxStack);
  L.rot_done = take(sizeof(int) * (size_t)kMaxStack);
  L.tile_counters = take(sizeof(int) * 4 * (size_t)kMaxTiles);
  L.split_slots = take(sizeof(float) * (size_t)kPartialSlotFloats * num_sms);
  L.xprep = take(sizeof(uint16_t) * (size_t)kSplitKeys * kMaxT * kMaxK);
  L.stats = take(sizeof(double) * 2 * (size_t)4096 * kAcceptChunks);
  L.chunks = take(sizeof(double) * kScanBlocks);
  L.argidx = take(sizeof(int) * (size_t)(kMaxAcceptT + 1) * kAcceptChunks);
  L.argval = take(sizeof(float) * (size_t)(kMaxAcceptT + 1) * kAcceptChunks);
  L.acc_counters = take(sizeof(int) * 16);
  L.rowstat = take(sizeof(double) * 2 * (size_t)4096);
  L.rowcnt = take(sizeof(int) * (size_t)4096);
  L.gbest = take(sizeof(float) * (size_t)(kMaxAcceptT + 1) * kAcceptChunks);
  L.gidx = take(sizeof(int) * (size_t)(kMaxAcceptT + 1) * kAcceptChunks);
  L.gsecond = take(sizeof(float) * (size_t)(kMaxAcceptT + 1) * kAcceptChunks);
  L.total = off;
  return L;
}

int check_ctx(spec_ctx* ctx) {
  if (!ctx) return set_error(SPEC_ERR_ARG, "null context");
  return SPEC_OK;
}

int check_ptr(const void* p, size_t align, const char* name) {
  if (!p) return set_error(SPEC_ERR_ARG, "%s is null", name);
  if (!aligned(p, align)) return set_error(SPEC_ERR_ARG, "%s is not %zu-byte aligned", name, align);
  return SPEC_OK;
}

#define SV_TRY(expr)           \
  do {                         \
    const int _rc = (expr);    \
    if (_rc != SPEC_OK) return _rc; \
  } while (0)

int check_rotation(const int8_t* signs, int block, int T, int K) {
  if (!signs && block == 0) return SPEC_OK;
  if (!signs || block == 0)
    return set_error(SPEC_ERR_ARG, "signs and hadamard_block must be given together");
  if (block < 32 || block > 1024 || (block & (block - 1)))
    return set_error(SPEC_ERR_SHAPE, "hadamard_block %d not a power of two in [32, 1024]", block);
  if (K % block) return set_error(SPEC_ERR_SHAPE, "K=%d not a multiple of hadamard_block %d", K, block);
  if (reinterpret_cast<uintptr_t>(signs) % 16)
    return set_error(SPEC_ERR_ARG, "signs must be 16-byte aligned");
  if (K > kMaxK || 2 * T > kMaxT)
    return set_error(SPEC_ERR_SHAPE, "rotated GEMMs take T <= %d, K <= %d", kMaxT / 2, kMaxK);
  return SPEC_OK;
}

int check_gemm_common(const void* x, const void* y, int y_dtype, int T, int N, int K,
                      int group_size, bool w4) {
  SV_TRY(check_ptr(x, 16, "x"));
  SV_TRY(check_ptr(y, 16, "y"));
  if (y_dtype != SPEC_DTYPE_BF16 && y_dtype != SPEC_DTYPE_F32)
    return set_error(SPEC_ERR_ARG, "y_dtype %d is not SPEC_DTYPE_BF16/F32", y_dtype);
  if (T < 1 || T > kMaxT) return set_error(SPEC_ERR_SHAPE, "T=%d outside 1..%d", T, kMaxT);
  if (N < 1 || N > (1 << 22)) return set_error(SPEC_ERR_SHAPE, "N=%d outside 1..2^22", N);
  if (N % (w4 ? 32 : 8)) return set_error(SPEC_ERR_SHAPE, "N=%d not a multiple of %d", N, w4 ? 32 : 8);
  if (K < 64 || K % 64) return set_error(SPEC_ERR_SHAPE, "K=%d not a positive multiple of 64", K);
  if (K > (1 << 20)) return set_error(SPEC_ERR_SHAPE, "K=%d above 2^20", K);
  if (w4 || group_size) {
    if (group_size < 64 || (group_size & (group_size - 1)) || K % group_size)
      return set_error(SPEC_ERR_SHAPE, "group_size=%d must be a power of two >= 64 dividing K=%d",
                       group_size, K);
  }
  if (group_size < 0) return set_error(SPEC_ERR_SHAPE, "negative group_size");
  // int4 and grouped int8 GEMMs read their activations as fp16, prepared in
  // the context's scratch
  if ((w4 || group_size) && K > kMaxK)
    return set_error(SPEC_ERR_SHAPE, "K=%d above %d for int4 or grouped int8 weights", K, kMaxK);
  return SPEC_OK;
}

// The split engine: a rotated GEMM is the standalone rotation into the
// context's scratch, then the GEMM on the rotated bf16 activations; each
// launch lets the next one start early and waits for its predecessor before
// it touches what that one wrote.
int run_split(spec_ctx* ctx, GemmArgs a, cudaStream_t s) {
  if (a.signs) {
    SV_TRY(launch_fwht(ctx, a.x, ctx->xprep, a.T, a.K, a.signs, a.rot_block, s));
    a.x = ctx->xprep;
    a.signs = nullptr;
    a.rot_block = 0;
  }
  return launch_qgemm_split(ctx, a, s);
}

int run_gemm(spec_ctx* ctx, GemmArgs& a, void* stream) {
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  if (ctx->engine == SPEC_GEMM_ENGINE_STACK) return launch_qgemm(ctx, a, static_cast<cudaStream_t>(stream));
  return run_split(ctx, a, static_cast<cudaStream_t>(stream));
}

// Reads a positive integer tuning knob from the environment (0 if unset).
int env_int(const char* name) {
  const char* v = std::getenv(name);
  if (!v || !*v) return 0;
  const long x = std::strtol(v, nullptr, 10);
  return x > 0 && x < 1 << 20 ? (int)x : 0;
}

}  // namespace

extern "C" {

int spec_version(void) { return (0 << 16) | 1; }

const char* spec_last_error(void) { return g_err; }

int spec_create(int device, size_t workspace_bytes, spec_ctx** out) {
  clear_error();
  if (!out) return set_error(SPEC_ERR_ARG, "out is null");
  *out = nullptr;
  int ndev = 0;
  SV_TRY(check_cuda(cudaGetDeviceCount(&ndev), "cudaGetDeviceCount"));
  if (device < 0 || device >= ndev)
    return set_error(SPEC_ERR_ARG, "device %d outside 0..%d", device, ndev - 1);
  cudaDeviceProp prop;
  SV_TRY(check_cuda(cudaGetDeviceProperties(&prop, device), "cudaGetDeviceProperties"));
  if (prop.major != 10 || prop.minor != 3)
    return set_error(SPEC_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a",
                     device, prop.major, prop.minor);
  DeviceGuard dg(device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", device);
  const WsLayout L = layout_for(prop.multiProcessorCount);
  const size_t bytes = workspace_bytes ? workspace_bytes : L.total;
  if (bytes < L.total)
    return set_error(SPEC_ERR_OOM, "workspace of %zu bytes is below the %zu needed", bytes, L.total);
  spec_ctx* ctx = new (std::nothrow) spec_ctx();
  if (!ctx) return set_error(SPEC_ERR_OOM, "host allocation failed");
  ctx->device = device;
  ctx->num_sms = prop.multiProcessorCount;
  if (cudaMalloc(&ctx->ws, bytes) != cudaSuccess) {
    delete ctx;
    return set_error(SPEC_ERR_OOM, "cudaMalloc of %zu workspace bytes failed", bytes);
  }
  ctx->ws_bytes = bytes;
  if (cudaMemset(ctx->ws, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(ctx->ws);
    delete ctx;
    return set_error(SPEC_ERR_CUDA, "workspace initialisation failed");
  }
  ctx->err = reinterpret_cast<int*>(ctx->ws + L.err);
  ctx->abort_all = reinterpret_cast<int*>(ctx->ws + L.abort_all);
  ctx->exit_cnt = reinterpret_cast<int*>(ctx->ws + L.exit_cnt);
  ctx->split_cnt = reinterpret_cast<int*>(ctx->ws + L.split_cnt);
  ctx->partials = reinterpret_cast<float*>(ctx->ws + L.partials);
  ctx->done = reinterpret_cast<int*>(ctx->ws + L.done);
  ctx->rot_done = reinterpret_cast<int*>(ctx->ws + L.rot_done);
  ctx->tile_counters = reinterpret_cast<int*>(ctx->ws + L.tile_counters);
  ctx->split_partials = reinterpret_cast<float*>(ctx->ws + L.split_slots);
  ctx->max_slots = ctx->num_sms;
  if (const int v = env_int("SPEC_PREFETCH_LEAD")) ctx->pf_dist = v;
  if (const int v = env_int("SPEC_PREFETCH_LEAD_FULL")) ctx->pf_max = v;
  ctx->xprep = reinterpret_cast<uint16_t*>(ctx->ws + L.xprep);
  ctx->acc_stats = reinterpret_cast<double*>(ctx->ws + L.stats);
  ctx->acc_chunks = reinterpret_cast<double*>(ctx->ws + L.chunks);
  ctx->acc_argmax = reinterpret_cast<int*>(ctx->ws + L.argidx);
  ctx->acc_argval = reinterpret_cast<float*>(ctx->ws + L.argval);
  ctx->acc_counters = reinterpret_cast<int*>(ctx->ws + L.acc_counters);
  ctx->acc_rowstat = reinterpret_cast<double*>(ctx->ws + L.rowstat);
  ctx->acc_rowcnt = reinterpret_cast<int*>(ctx->ws + L.rowcnt);
  ctx->gum_best = reinterpret_cast<float*>(ctx->ws + L.gbest);
  ctx->gum_idx = reinterpret_cast<int*>(ctx->ws + L.gidx);
  ctx->gum_second = reinterpret_cast<float*>(ctx->ws + L.gsecond);
  *out = ctx;
  return SPEC_OK;
}

int spec_destroy(spec_ctx* ctx) {
  clear_error();
  if (!ctx) return SPEC_OK;
  int rc = SPEC_OK;
  {
    DeviceGuard dg(ctx->device);
    if (ctx->ws && cudaFree(ctx->ws) != cudaSuccess) rc = set_error(SPEC_ERR_CUDA, "cudaFree failed");
  }
  delete ctx;
  return rc;
}

int spec_sync_status(spec_ctx* ctx, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  SV_TRY(check_cuda(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream sync"));
  int err = 0;
  SV_TRY(check_cuda(cudaMemcpy(&err, ctx->err, sizeof(int), cudaMemcpyDeviceToHost), "read error word"));
  if (err == 0) return SPEC_OK;
  const WsLayout L = layout_for(ctx->num_sms);
  cudaMemset(ctx->ws, 0, L.xprep);   // error word, abort flag, split-tile sums and every counter
  cudaMemset(ctx->acc_counters, 0, sizeof(int) * 16);
  cudaMemset(ctx->acc_rowcnt, 0, sizeof(int) * 4096);
  cudaDeviceSynchronize();
  if (err == 1) return set_error(SPEC_ERR_TIMEOUT, "a device-side wait timed out");
  return set_error(SPEC_ERR_ARG, "a draft token or parent index read on the device was out of "
                                 "range (code %d)", err);
}

int qgemm_w4a16(spec_ctx* ctx, const uint8_t* qcodes, const uint16_t* scales, const uint8_t* zeros,
                int group_size, const uint16_t* x, void* y, int y_dtype, int T, int N, int K,
                const int8_t* signs, int hadamard_block, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  SV_TRY(check_ptr(qcodes, 16, "qcodes"));
  SV_TRY(check_ptr(scales, 16, "scales"));
  SV_TRY(check_ptr(zeros, 16, "zeros"));
  SV_TRY(check_gemm_common(x, y, y_dtype, T, N, K, group_size, true));
  SV_TRY(check_rotation(signs, hadamard_block, T, K));
  GemmArgs a{kW4, qcodes, scales, zeros, group_size, x, y, y_dtype == SPEC_DTYPE_F32, T, N, K,
             signs, hadamard_block, 0};
  return run_gemm(ctx, a, stream);
}

int qgemm_w8a16(spec_ctx* ctx, const int8_t* qcodes, const uint16_t* scales, int group_size,
                const uint16_t* x, void* y, int y_dtype, int T, int N, int K, const int8_t* signs,
                int hadamard_block, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  SV_TRY(check_ptr(qcodes, 16, "qcodes"));
  SV_TRY(check_ptr(scales, 16, "scales"));
  SV_TRY(check_gemm_common(x, y, y_dtype, T, N, K, group_size, false));
  SV_TRY(check_rotation(signs, hadamard_block, T, K));
  GemmArgs a{kW8, qcodes, scales, nullptr, group_size, x, y, y_dtype == SPEC_DTYPE_F32, T, N, K,
             signs, hadamard_block, 0};
  return run_gemm(ctx, a, stream);
}

int qgemm_stack_create(spec_ctx* ctx, const spec_gemm_desc* descs, int n, spec_gemm_stack** out) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (!out) return set_error(SPEC_ERR_ARG, "out is null");
  *out = nullptr;
  if (!descs) return set_error(SPEC_ERR_ARG, "descs is null");
  if (n < 1 || n > kMaxStack) return set_error(SPEC_ERR_SHAPE, "n=%d outside 1..%d", n, kMaxStack);
  const int quant = descs[0].quant;
  if (quant != SPEC_QUANT_W4 && quant != SPEC_QUANT_W8)
    return set_error(SPEC_ERR_ARG, "descs[0].quant %d is not SPEC_QUANT_W4/W8", quant);
  int tpad = 16, run = 0;
  for (int i = 0; i < n; ++i) {
    const spec_gemm_desc& d = descs[i];
    const bool w4 = d.quant == SPEC_QUANT_W4;
    if (d.quant != quant) return set_error(SPEC_ERR_ARG, "descs[%d]: every GEMM of a stack has one quant", i);
    SV_TRY(check_ptr(d.qcodes, 16, "qcodes"));
    SV_TRY(check_ptr(d.scales, 16, "scales"));
    if (w4) SV_TRY(check_ptr(d.zeros, 16, "zeros"));
    SV_TRY(check_gemm_common(d.x, d.y, d.y_dtype, d.T, d.N, d.K, d.group_size, w4));
    SV_TRY(check_rotation(d.signs, d.hadamard_block, d.T, d.K));
    GemmArgs probe{};
    probe.quant = quant == SPEC_QUANT_W4 ? kW4 : kW8;
    probe.group_size = d.group_size;
    probe.T = d.T;
    probe.signs = d.signs;
    const int tp = gemm_tpad(probe);
    if (tp > tpad) tpad = tp;
    // split-tile slots are keyed by entry index mod kSplitKeys: at most that
    // many entries may be in flight at once
    run = (i > 0 && !d.wait_prev) ? run + 1 : 0;
    if (run >= kSplitKeys)
      return set_error(SPEC_ERR_ARG, "descs[%d]: more than %d consecutive entries without wait_prev", i,
                       kSplitKeys - 1);
  }
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  std::vector<GemmEntry> host(n);
  spec_gemm_stack* st = new (std::nothrow) spec_gemm_stack();
  if (!st) return set_error(SPEC_ERR_OOM, "host allocation failed");
  st->ctx = ctx;
  st->quant = quant == SPEC_QUANT_W4 ? kW4 : kW8;
  st->tpad = tpad;
  st->n = n;
  for (int i = 0; i < n; ++i) {
    const spec_gemm_desc& d = descs[i];
    GemmArgs a{st->quant, d.qcodes, d.scales, d.zeros, d.group_size, d.x, d.y,
               d.y_dtype == SPEC_DTYPE_F32, d.T, d.N, d.K, d.signs, d.hadamard_block, d.wait_prev};
    st->args.push_back(a);
    const int rc = build_entry(ctx, a, tpad, i % kSplitKeys, &host[i]);
    if (rc) {
      delete st;
      return rc;
    }
    if (host[i].prep) st->prep_flags |= kAnyPrep;
    if (host[i].xconv) st->prep_flags |= kAnyConv;
  }
  if (cudaMalloc(&st->dev_entries, sizeof(GemmEntry) * (size_t)n) != cudaSuccess) {
    delete st;
    return set_error(SPEC_ERR_OOM, "cudaMalloc of the stack's %d entries failed", n);
  }
  if (cudaMemcpy(st->dev_entries, host.data(), sizeof(GemmEntry) * (size_t)n, cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    cudaFree(st->dev_entries);
    delete st;
    return set_error(SPEC_ERR_CUDA, "copy of the stack's entries failed");
  }
  *out = st;
  return SPEC_OK;
}

int qgemm_stack_run(spec_ctx* ctx, const spec_gemm_stack* stack, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (!stack) return set_error(SPEC_ERR_ARG, "stack is null");
  if (stack->ctx != ctx) return set_error(SPEC_ERR_ARG, "stack was created on another context");
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ctx->engine == SPEC_GEMM_ENGINE_STACK) return launch_qgemm_stack(ctx, stack, s);
  for (const GemmArgs& a : stack->args) SV_TRY(run_split(ctx, a, s));
  return SPEC_OK;
}

int spec_set_gemm_engine(spec_ctx* ctx, int engine) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (engine != SPEC_GEMM_ENGINE_AUTO && engine != SPEC_GEMM_ENGINE_SPLIT && engine != SPEC_GEMM_ENGINE_STACK)
    return set_error(SPEC_ERR_ARG, "engine %d is not SPEC_GEMM_ENGINE_AUTO/SPLIT/STACK", engine);
  ctx->engine = engine;
  return SPEC_OK;
}

int qgemm_stack_destroy(spec_gemm_stack* stack) {
  clear_error();
  if (!stack) return SPEC_OK;
  int rc = SPEC_OK;
  {
    DeviceGuard dg(stack->ctx->device);
    if (stack->dev_entries && cudaFree(stack->dev_entries) != cudaSuccess)
      rc = set_error(SPEC_ERR_CUDA, "cudaFree failed");
  }
  delete stack;
  return rc;
}

int spec_set_stream_prefetch(spec_ctx* ctx, int lead, int lead_when_full) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (lead < 0 || lead_when_full < lead || lead_when_full > 256)
    return set_error(SPEC_ERR_ARG, "prefetch leads %d/%d outside 0 <= lead <= lead_when_full <= 256",
                     lead, lead_when_full);
  ctx->pf_dist = lead;
  ctx->pf_max = lead_when_full;
  return SPEC_OK;
}

int spec_test_stall(spec_ctx* ctx, int skip_unit, uint64_t wait_limit_ns) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (skip_unit < -1) return set_error(SPEC_ERR_ARG, "skip_unit %d < -1", skip_unit);
  if (wait_limit_ns < 100000ull || wait_limit_ns > kWaitLimitNs)
    return set_error(SPEC_ERR_ARG, "wait limit %llu ns outside [1e5, %llu]",
                     (unsigned long long)wait_limit_ns, (unsigned long long)kWaitLimitNs);
  ctx->test_skip_unit = skip_unit;
  ctx->test_wait_ns = wait_limit_ns;
  return SPEC_OK;
}

int fwht_rotate(spec_ctx* ctx, const uint16_t* x, uint16_t* y, int T, int K, const int8_t* signs,
                int block, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  SV_TRY(check_ptr(x, 16, "x"));
  SV_TRY(check_ptr(y, 16, "y"));
  SV_TRY(check_ptr(signs, 1, "signs"));
  if (T < 1) return set_error(SPEC_ERR_SHAPE, "T=%d < 1", T);
  if (block < 32 || block > 1024 || (block & (block - 1)))
    return set_error(SPEC_ERR_SHAPE, "block %d not a power of two in [32, 1024]", block);
  if (K < block || K % block) return set_error(SPEC_ERR_SHAPE, "K=%d not a multiple of block %d", K, block);
  if ((long long)T * K > (1LL << 34)) return set_error(SPEC_ERR_SHAPE, "T*K too large");
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_fwht(ctx, x, y, T, K, signs, block, static_cast<cudaStream_t>(stream));
}

int spec_softmax(spec_ctx* ctx, const float* logits, float* probs, int rows, int V, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  SV_TRY(check_ptr(logits, 4, "logits"));
  SV_TRY(check_ptr(probs, 4, "probs"));
  if (rows < 1 || rows > 4096) return set_error(SPEC_ERR_SHAPE, "rows=%d outside 1..4096", rows);
  if (V < 1 || V > (1 << 26)) return set_error(SPEC_ERR_SHAPE, "V=%d outside 1..2^26", V);
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_softmax(ctx, logits, probs, rows, V, static_cast<cudaStream_t>(stream));
}

int spec_accept(spec_ctx* ctx, const float* target_logits, const float* draft_probs,
                const int32_t* draft_tokens, const float* uniforms, int T, int V,
                int32_t* n_accepted, int32_t* out_tokens, int32_t* near_tie_flags, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (T < 0 || T > kMaxAcceptT) return set_error(SPEC_ERR_SHAPE, "T=%d outside 0..%d", T, kMaxAcceptT);
  if (V < 1 || V > (1 << 26)) return set_error(SPEC_ERR_SHAPE, "V=%d outside 1..2^26", V);
  SV_TRY(check_ptr(target_logits, 4, "target_logits"));
  if (T > 0) {
    SV_TRY(check_ptr(draft_probs, 4, "draft_probs"));
    SV_TRY(check_ptr(draft_tokens, 4, "draft_tokens"));
  }
  SV_TRY(check_ptr(uniforms, 4, "uniforms"));
  SV_TRY(check_ptr(n_accepted, 4, "n_accepted"));
  SV_TRY(check_ptr(out_tokens, 4, "out_tokens"));
  if (near_tie_flags) SV_TRY(check_ptr(near_tie_flags, 4, "near_tie_flags"));
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_accept(ctx, target_logits, draft_probs, draft_tokens, uniforms, T, V, n_accepted,
                       out_tokens, near_tie_flags, static_cast<cudaStream_t>(stream));
}

int spec_accept_noalloc(const float* target_logits, const float* draft_probs,
                        const int32_t* draft_tokens, const float* uniforms, int T, int V,
                        int32_t* n_accepted, int32_t* out_tokens, int32_t* near_tie_flags,
                        int32_t* device_status, void* stream) {
  clear_error();
  if (T < 0) return set_error(SPEC_ERR_SHAPE, "T=%d is negative", T);
  if (V < 1 || V > (1 << 26)) return set_error(SPEC_ERR_SHAPE, "V=%d outside 1..2^26", V);
  SV_TRY(check_ptr(target_logits, 4, "target_logits"));
  if (T > 0) {
    SV_TRY(check_ptr(draft_probs, 4, "draft_probs"));
    SV_TRY(check_ptr(draft_tokens, 4, "draft_tokens"));
  }
  SV_TRY(check_ptr(uniforms, 4, "uniforms"));
  SV_TRY(check_ptr(n_accepted, 4, "n_accepted"));
  SV_TRY(check_ptr(out_tokens, 4, "out_tokens"));
  if (near_tie_flags) SV_TRY(check_ptr(near_tie_flags, 4, "near_tie_flags"));
  if (device_status) SV_TRY(check_ptr(device_status, 4, "device_status"));
  return launch_accept_noalloc(target_logits, draft_probs, draft_tokens, uniforms, T, V, n_accepted,
                               out_tokens, near_tie_flags, device_status,
                               static_cast<cudaStream_t>(stream));
}

int spec_accept_tree(spec_ctx* ctx, const float* target_logits, const int32_t* draft_tokens,
                     const int32_t* parent, int T, int V, int32_t* path_len, int32_t* out_tokens,
                     int32_t* path_nodes, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (T < 1 || T > kMaxAcceptT) return set_error(SPEC_ERR_SHAPE, "T=%d outside 1..%d", T, kMaxAcceptT);
  if (V < 1 || V > (1 << 26)) return set_error(SPEC_ERR_SHAPE, "V=%d outside 1..2^26", V);
  SV_TRY(check_ptr(target_logits, 4, "target_logits"));
  SV_TRY(check_ptr(draft_tokens, 4, "draft_tokens"));
  SV_TRY(check_ptr(parent, 4, "parent"));
  SV_TRY(check_ptr(path_len, 4, "path_len"));
  SV_TRY(check_ptr(out_tokens, 4, "out_tokens"));
  SV_TRY(check_ptr(path_nodes, 4, "path_nodes"));
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_accept_tree(ctx, target_logits, draft_tokens, parent, T, V, path_len, out_tokens,
                            path_nodes, static_cast<cudaStream_t>(stream));
}

int spec_gumbel_sample(spec_ctx* ctx, const float* logits, int rows, int V, uint64_t seed,
                       uint64_t position, int32_t* out_tokens, int32_t* near_tie_flags, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (rows < 1 || rows > kMaxAcceptT + 1)
    return set_error(SPEC_ERR_SHAPE, "rows=%d outside 1..%d", rows, kMaxAcceptT + 1);
  if (V < 1 || V > (1 << 26)) return set_error(SPEC_ERR_SHAPE, "V=%d outside 1..2^26", V);
  SV_TRY(check_ptr(logits, 4, "logits"));
  SV_TRY(check_ptr(out_tokens, 4, "out_tokens"));
  if (near_tie_flags) SV_TRY(check_ptr(near_tie_flags, 4, "near_tie_flags"));
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_gumbel(ctx, logits, rows, V, seed, position, 0, nullptr, out_tokens, nullptr,
                       near_tie_flags, static_cast<cudaStream_t>(stream));
}

int spec_accept_gumbel(spec_ctx* ctx, const float* target_logits, const int32_t* draft_tokens, int T,
                       int V, uint64_t seed, uint64_t position, int32_t* n_accepted,
                       int32_t* out_tokens, int32_t* near_tie_flags, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  if (T < 0 || T > kMaxAcceptT) return set_error(SPEC_ERR_SHAPE, "T=%d outside 0..%d", T, kMaxAcceptT);
  if (V < 1 || V > (1 << 26)) return set_error(SPEC_ERR_SHAPE, "V=%d outside 1..2^26", V);
  SV_TRY(check_ptr(target_logits, 4, "target_logits"));
  if (T > 0) SV_TRY(check_ptr(draft_tokens, 4, "draft_tokens"));
  SV_TRY(check_ptr(n_accepted, 4, "n_accepted"));
  SV_TRY(check_ptr(out_tokens, 4, "out_tokens"));
  if (near_tie_flags) SV_TRY(check_ptr(near_tie_flags, 4, "near_tie_flags"));
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_gumbel(ctx, target_logits, T + 1, V, seed, position, 1, draft_tokens, out_tokens,
                       n_accepted, near_tie_flags, static_cast<cudaStream_t>(stream));
}

int qdequant_w4(spec_ctx* ctx, const uint8_t* qcodes, const uint16_t* scales, const uint8_t* zeros,
                int group_size, int N, int K, float* w, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  SV_TRY(check_ptr(qcodes, 1, "qcodes"));
  SV_TRY(check_ptr(scales, 2, "scales"));
  SV_TRY(check_ptr(zeros, 1, "zeros"));
  SV_TRY(check_ptr(w, 4, "w"));
  if (N < 2 || N % 2 || K < 8 || K % 8 || group_size < 1 || K % group_size)
    return set_error(SPEC_ERR_SHAPE, "bad int4 shape N=%d K=%d g=%d", N, K, group_size);
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_dequant(ctx, kW4, qcodes, scales, zeros, group_size, N, K, w,
                        static_cast<cudaStream_t>(stream));
}

int qdequant_w8(spec_ctx* ctx, const int8_t* qcodes, const uint16_t* scales, int group_size, int N,
                int K, float* w, void* stream) {
  clear_error();
  SV_TRY(check_ctx(ctx));
  SV_TRY(check_ptr(qcodes, 1, "qcodes"));
  SV_TRY(check_ptr(scales, 2, "scales"));
  SV_TRY(check_ptr(w, 4, "w"));
  if (N < 1 || K < 1 || group_size < 0 || (group_size && K % group_size))
    return set_error(SPEC_ERR_SHAPE, "bad int8 shape N=%d K=%d g=%d", N, K, group_size);
  DeviceGuard dg(ctx->device);
  if (!dg.ok) return set_error(SPEC_ERR_CUDA, "cudaSetDevice(%d) failed", ctx->device);
  return launch_dequant(ctx, kW8, qcodes, scales, nullptr, group_size, N, K, w,
                        static_cast<cudaStream_t>(stream));
}

int spec_repack_w4_codes(const uint8_t* src, uint8_t* dst, int N, int K) {
  clear_error();
  if (!src || !dst) return set_error(SPEC_ERR_ARG, "src or dst is null");
  if (N < 1 || K < 8 || K % 8) return set_error(SPEC_ERR_SHAPE, "N=%d K=%d: need N >= 1, K >= 8, K %% 8 == 0", N, K);
  const size_t groups = (size_t)N * (size_t)(K / 8);
  for (size_t i = 0; i < groups; ++i) {
    // plain order: s0 = (k0, k1), s1 = (k2, k3), s2 = (k4, k5), s3 = (k6, k7) as (low, high)
    const uint32_t s0 = src[4 * i], s1 = src[4 * i + 1], s2 = src[4 * i + 2], s3 = src[4 * i + 3];
    // library order: (k0, k2), (k4, k6), (k1, k3), (k5, k7)
    dst[4 * i] = (uint8_t)((s0 & 0xFu) | ((s1 & 0xFu) << 4));
    dst[4 * i + 1] = (uint8_t)((s2 & 0xFu) | ((s3 & 0xFu) << 4));
    dst[4 * i + 2] = (uint8_t)((s0 >> 4) | (s1 & 0xF0u));
    dst[4 * i + 3] = (uint8_t)((s2 >> 4) | (s3 & 0xF0u));
  }
  return SPEC_OK;
}

}  // extern "C"
