// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>

#include "specverify.h"

namespace sv {

constexpr int kMaxT = 64;                    // largest draft block of the GEMMs
constexpr int kTileM = 128;                  // weight rows per MMA tile
constexpr int kStageK = 64;                  // k per pipeline stage
constexpr int kPartialSlotFloats = kMaxT * kTileM;
constexpr int kMaxK = 32768;                 // rotated-activation buffer width
constexpr int kMaxTiles = (1 << 22) / kTileM;
constexpr int kMaxAcceptT = 256;
constexpr int kAcceptChunks = 64;            // max V-chunks per row in the acceptance kernels
constexpr int kScanBlocks = 256;             // max blocks of the residual scan

int set_error(int code, const char* fmt, ...);
void clear_error();
int check_cuda(cudaError_t e, const char* what);

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link libcuda directly).
int encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0,
                   uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle sw);

// Quantisation flavour of the verify GEMM kernel.
enum Quant { kW4 = 0, kW8 = 1 };

struct GemmArgs {
  int quant;
  const void* qcodes;
  const uint16_t* scales;
  const uint8_t* zeros;   // W4 only
  int group_size;         // 0 = per output channel (W8 only)
  const uint16_t* x;      // bf16 [T][K] (already rotated if requested)
  void* y;
  int y_f32;
  int T, N, K;
};

}  // namespace sv

struct spec_ctx {
  int device = 0;
  int num_sms = 0;
  size_t ws_bytes = 0;
  uint8_t* ws = nullptr;
  int* err = nullptr;             // device error word
  int* tile_counters = nullptr;   // [kMaxTiles][4] split-K arrival counters (per lane quadrant)
  float* partials = nullptr;      // [max_slots][kPartialSlotFloats]
  int max_slots = 0;
  uint16_t* xrot = nullptr;       // [kMaxT][kMaxK] rotated activations
  double* acc_stats = nullptr;    // [rows][kAcceptChunks][2] (max, sum) partials
  double* acc_chunks = nullptr;   // [kScanBlocks] residual chunk sums
  int* acc_argmax = nullptr;      // [kMaxAcceptT+1][kAcceptChunks] argmax partial index
  float* acc_argval = nullptr;    // [kMaxAcceptT+1][kAcceptChunks] argmax partial value
  int* acc_counters = nullptr;    // [16] arrival counters of the acceptance kernels
  double* acc_rowstat = nullptr;  // [4096][2] per-row (max, 1/Z) merged by row_stats
  int* acc_rowcnt = nullptr;      // [4096] per-row arrival counters of row_stats, kept zeroed
  float* gum_best = nullptr;      // [kMaxAcceptT+1][kAcceptChunks] shared-seed sampling partials
  int* gum_idx = nullptr;
  float* gum_second = nullptr;
};

namespace sv {
int launch_qgemm(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s);
int launch_fwht(spec_ctx* ctx, const uint16_t* x, uint16_t* y, int T, int K, const int8_t* signs,
                int block, cudaStream_t s);
int launch_softmax(spec_ctx* ctx, const float* logits, float* probs, int rows, int V,
                   cudaStream_t s);
int launch_accept(spec_ctx* ctx, const float* logits, const float* q, const int32_t* drafts,
                  const float* u, int T, int V, int32_t* n_acc, int32_t* tokens, int32_t* flags,
                  cudaStream_t s);
int launch_accept_noalloc(const float* logits, const float* q, const int32_t* drafts, const float* u,
                          int T, int V, int32_t* n_acc, int32_t* tokens, int32_t* flags,
                          int32_t* status, cudaStream_t s);
int launch_accept_tree(spec_ctx* ctx, const float* logits, const int32_t* drafts,
                       const int32_t* parent, int T, int V, int32_t* path_len, int32_t* tokens,
                       int32_t* nodes, cudaStream_t s);
int launch_gumbel(spec_ctx* ctx, const float* logits, int rows, int V, uint64_t seed, uint64_t position,
                  int accept, const int32_t* drafts, int32_t* tokens, int32_t* n_acc, int32_t* flags,
                  cudaStream_t s);
int launch_dequant(spec_ctx* ctx, int quant, const void* qcodes, const uint16_t* scales,
                   const uint8_t* zeros, int group_size, int N, int K, float* w, cudaStream_t s);
}  // namespace sv
