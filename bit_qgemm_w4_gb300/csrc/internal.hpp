// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "specverify.h"

namespace sv {

constexpr int kMaxT = 64;                    // largest draft block of the GEMMs
constexpr int kTileM = 128;                  // weight rows per MMA tile
constexpr int kGroupK = 64;                  // k per MMA group (one fp32 partial)
constexpr int kPartialSlotFloats = kMaxT * kTileM;
constexpr int kMaxK = 32768;                 // rotated-activation buffer width
constexpr int kSplitKeys = 4;                // GEMMs of one launch whose split tiles may overlap
enum { kAnyPrep = 1, kAnyConv = 2 };         // a launch's prep_flags
constexpr int kLocalConvStages = 32;         // GEMMs of at most this many stages per SM convert
                                             // their activations in each CTA's shared memory
constexpr int kGemmWorkers = 8;              // dequant/epilogue warps per CTA
constexpr int kMaxStack = 1024;              // GEMMs per stack launch
constexpr int kMaxTiles = (1 << 22) / kTileM;   // 128-row tiles of the largest N
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
  const uint16_t* x;      // bf16 [T][K]
  void* y;
  int y_f32;
  int T, N, K;
  const int8_t* signs;    // rotation signs [K] or null
  int rot_block;          // Hadamard block (0 = no rotation)
  int wait_prev;          // stack entries: read x only after the earlier GEMMs completed
};

// One GEMM as the verify kernel sees it: tensor maps and derived sizes.  A
// single call passes one entry as a kernel parameter; a stack keeps an array
// of them in device memory.
struct alignas(64) GemmEntry {
  CUtensorMap tm_x;        // activations (or their rotated copy) [T][K] bf16, box [TPAD][64]
  CUtensorMap tm_codes;    // codes [N][K/2] (int4) or [N][K] (int8), box [128][128 bytes]
  CUtensorMap tm_scales;   // scales [K/g][N] fp16, box [rows][128]
  CUtensorMap tm_zeros;    // int4 zero points [K/g][N/2], box [rows][64]
  const uint16_t* x;       // activations as given
  const int8_t* signs;     // rotation signs, null = no rotation
  uint16_t* xprep;         // the activations in the MMA's operand form (rotated and/or
                           // converted to fp16), which tm_x then points at; null = x as given
  const uint16_t* chscale; // per-output-channel int8 scales [N] (group_size 0), else null
  void* y;
  int T, N, K;
  int rot_block;           // Hadamard block, 0 = none
  float rot_scale;         // 1/sqrt(rot_block)
  int ks;                  // stages per 128-row tile
  int tiles;
  int units;               // tiles * ks
  int gshift;              // log2(group_size): group row of a stage's first k
  int gsh;                 // row of 64-k group j inside a stage's scale box = (64 j) >> gsh
  int scale_rows;          // rows of a stage's scale box (0 = per-channel scales)
  uint32_t tx_w;           // TMA bytes of one stage's codes, scales and zero points
  int y_f32;
  int wait_prev;
  int kind;                // operand form: kGemmBf16, kGemmF16Nib or kGemmF16
  int prep;                // activations prepared inside the launch by all CTAs into the
                           // scratch copy: 0 none, 1 rotated, 2 converted to fp16
  int xconv;               // activations converted to fp16 in each CTA's own shared-memory
                           // slots as they arrive: 0 none, 1 fp16, 2 fp16 with the int4
                           // column scaling
  uint32_t idesc;          // tcgen05.mma instruction descriptor (operand types, M, N)
};

// Operand forms of the verify GEMM's MMAs:
//  kGemmBf16   exact int8 codes and the bf16 activations as given (int8 with
//              one scale per output channel, applied to the fp32 sums)
//  kGemmF16Nib int4: weights (code - zero) * scale rounded once to fp16;
//              activations in fp16, the columns k % 8 in {2, 3, 6, 7} divided
//              by 16 (their weights are read with a factor 16)
//  kGemmF16    int8 with group scales: code * scale rounded to fp16, fp16
//              activations
enum GemmKind { kGemmBf16 = 0, kGemmF16Nib = 1, kGemmF16 = 2 };

}  // namespace sv

struct spec_ctx {
  int device = 0;
  int num_sms = 0;
  size_t ws_bytes = 0;
  uint8_t* ws = nullptr;
  int* err = nullptr;             // device error word
  int engine = 0;                 // GEMM engine: SPEC_GEMM_ENGINE_* (0 = auto)
  int* tile_counters = nullptr;   // split engine: [kMaxTiles][4] split-tile arrivals per lane quadrant
  float* split_partials = nullptr;   // split engine: [max_slots][kPartialSlotFloats] split-tile sums
  int max_slots = 0;
  float* partials = nullptr;      // [kSplitKeys][num_sms][kPartialSlotFloats] split-tile sums
  int* split_cnt = nullptr;       // [kSplitKeys][num_sms][kGemmWorkers] split-tile arrivals
  int* done = nullptr;            // [kMaxStack] finished tile parts per stack entry
  int* rot_done = nullptr;        // [kMaxStack] CTAs that rotated their share per entry
  int* exit_cnt = nullptr;        // CTAs that left the last launch (resets the two above)
  int* abort_all = nullptr;       // raised by a CTA whose wait ran out
  int pf_dist = 4;                // GEMM weight stream: L2 prefetch lead (stages)
  int pf_max = 16;                // ... and the lead allowed while the shared-memory ring is full
  unsigned long long test_wait_ns = 0;   // test hook: wait limit of the next GEMM launch
  int test_skip_unit = -1;               // test hook: unit whose weights CTA 0 never loads
  uint16_t* xprep = nullptr;      // [kSplitKeys][kMaxT][kMaxK] prepared activations, keyed
                                  // like the split-tile slots by a GEMM's index in its launch
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

struct spec_gemm_stack {
  spec_ctx* ctx = nullptr;
  int quant = 0;
  int tpad = 0;
  int n = 0;
  int prep_flags = 0;   // kAnyPrep | kAnyConv over the entries
  sv::GemmEntry* dev_entries = nullptr;   // [n] in device memory
  std::vector<sv::GemmArgs> args;         // [n] the GEMMs as given (split engine)
};

namespace sv {
int build_entry(spec_ctx* ctx, const GemmArgs& a, int tpad, int index, GemmEntry* out);
int gemm_tpad(const GemmArgs& a);   // MMA N of a GEMM: T (2T when rotated) rounded up to 16
int launch_qgemm(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s);
int launch_qgemm_split(spec_ctx* ctx, const GemmArgs& a, cudaStream_t s);
int launch_qgemm_stack(spec_ctx* ctx, const spec_gemm_stack* st, cudaStream_t s);
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
