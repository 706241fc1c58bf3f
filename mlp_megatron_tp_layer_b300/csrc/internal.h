// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/tpl.h"

namespace tpl {

// NVTX range around one call of the C ABI: a profiler that records NVTX (nsys,
// ncu --nvtx) shows each entry point by name around the kernels it launched.
// Without a tool attached the push/pop calls do nothing.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define TPL_NVTX_RANGE(name) ::tpl::NvtxRange tpl_nvtx_range_(name)

// ---------------------------------------------------------------- epilogues
// How a GEMM-like kernel writes the value v computed for (token t, feature f).
// "token" is the row of the activation operand, "feature" the row of the
// [out, in] weight (the output column).
enum EpiMode : int {
    EPI_STORE = 0,    // out[t*ldo + f] (optionally column-blocked), dtype of the call
    EPI_PARTIAL = 1,  // fp32 out32[split*split_stride + t*ldo + f]
    EPI_SWIGLU = 2,   // out[t*ldo + f] = silu(gate) * up   (needs full sums)
    EPI_QKV = 3,      // scatter packed-QKV row f to each shard block, V rows also to O
    EPI_PARTIAL2 = 4  // two fp32 partial planes (gate, up) for split SwiGLU
};

struct QkvMap {
    int n_q, n_kv, head_dim, tp;
    int nq_s, kv_s;        // Q heads / KV groups held by one shard
    int64_t shard_stride;  // elements between shard blocks of qkv_out ([tp, B, W_s])
    int64_t w_s;           // row length of one shard block: (nq_s + 2 kv_s) * head_dim
    void* qkv_out;         // [tp, B, w_s]
    void* o_out;           // [B, n_q * head_dim] attention stand-in output
    int64_t ldo_o;
};

struct Epilogue {
    int mode;
    int out_bf16;          // output element type for EPI_STORE / EPI_SWIGLU (1 = bf16, 0 = fp32)
    void* out;             // EPI_STORE, EPI_SWIGLU
    float* out32;          // EPI_PARTIAL / EPI_PARTIAL2 (plane 0)
    float* out32b;         // EPI_PARTIAL2 plane 1
    int64_t ldo;           // row pitch of the output in elements
    int64_t col_block;     // > 0: output column f lives at (f / col_block) * block_stride + f % col_block
    int64_t block_stride;
    int64_t split_stride;  // EPI_PARTIAL(2): elements between split planes
    QkvMap qkv;
    const float* row_scale;    // EPI_QKV / EPI_SWIGLU: per-token factor applied to the fp32 products
                               // (the folded RMSNorm scale 1/rms), or null
    unsigned int* zero_words;  // if set, block 0 of the launch zeroes zero_count words at start
    int zero_count;            // (row accumulators of the reduction that consumes this output)
};

// Work split of the contracting dimension: K = tp shards of k_shard elements,
// each shard cut into `sub` chunks of k_chunk elements (the last may be shorter).
// Split index = shard * sub + j.
struct KSplit {
    int64_t k_shard;
    int64_t k_chunk;
    int tp;
    int sub;
};

// Context shared by every launch of the library (per device).
struct DeviceCtx {
    int device = -1;
    int num_sms = 0;
    unsigned int* err_word = nullptr;   // device address of the sticky error word
};
const DeviceCtx* device_ctx();          // nullptr if no CUDA device is usable

// Workspace of one tp_mlp_forward call: the plan for the partials argument
// actually given (null or not), as that call checks it.
size_t mlp_plan_bytes(int64_t B, int64_t D, int64_t F, int tp, int dt, bool want_partials);
// Whether out_dt is an output type tp_mlp_forward accepts for inputs of type dt.
bool mlp_out_dtype_ok(int dt, int out_dt);

// ------------------------------------------------------ CUDA-core kernels
// rows of W (N rows, length K, pitch ldw) dotted with nb tokens of X (pitch ldx);
// W1 non-null only for EPI_SWIGLU (up weights, same shape as W).
struct RowdotArgs {
    const void* X;
    int64_t ldx;
    int nb;
    const void* W;
    const void* W1;
    int64_t ldw;
    int64_t N, K;
    KSplit ks;
    int64_t tok0;      // token offset added when storing
    Epilogue epi;
};
cudaError_t launch_rowdot(const RowdotArgs& a, bool bf16, cudaStream_t st);

// Sum of split partials ws[tp*sub, rows, cols] (fp32): per shard over its sub
// chunks, then over shards in ascending order.  Optional outputs: the shard
// partials [tp, rows, cols] fp32, and y = residual + sum written as dtype
// (layout ALLREDUCE [rows, cols] or REDUCE_SCATTER [tp, rows, cols/tp]).
// Optional scale_out[row] = 1 / sqrt(mean(bf16(y)^2) + eps), the RMSNorm
// scale of each row, which needs the whole row.
struct ReduceArgs {
    const float* ws;
    int64_t rows, cols;
    int tp, sub;
    float* shard_out;
    void* y;
    int y_bf16;
    int mode;              // tpl_reduce_mode
    const void* residual;  // bf16 [rows, cols] or null
    float* scale_out;      // [rows] RMSNorm scales, or null
    float eps;
    const float* ws_up;    // non-null: ws/ws_up are gate/up planes -> y = silu(sum ws) * sum ws_up
    unsigned int* row_cnt; // scale_out only: [rows] block tickets, zero on entry (reset on exit)
    float* row_slots;      // scale_out only: [rows, norm_blocks(cols)] per-block sums of squares
};

// The row-normalising reduction covers kNormCols columns per block; a row's
// sum of squares is the sum of its blocks' slots in block order (deterministic).
// Row accumulator area ("rowacc") used by it: [rows] tickets, then the slots.
constexpr int kNormCols = 512;
inline int64_t norm_blocks(int64_t cols) { return (cols + kNormCols - 1) / kNormCols; }
inline size_t rowacc_bytes(int64_t rows, int64_t cols) { return (size_t)rows * 4 * (1 + norm_blocks(cols)); }
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t st);

// RMSNorm scales of bf16 rows: scale[r] = 1 / sqrt(mean(x[r]^2) + eps) (unit
// gain); zeroes the tickets of rowacc itself.
cudaError_t launch_rmsnorm(const void* x, float* scale, int64_t rows, int64_t cols, float eps,
                           unsigned int* rowacc, cudaStream_t st);

// ---------------------------------------------------- tensor-core GEMM
// D[M, N] = A[M, K] B[N, K]^T, A and B bf16 K-major.  `swap` means A holds the
// weights (M = features) and B the tokens (N = tokens); otherwise A holds the
// tokens.  A2 / B2: second weight operand for SwiGLU (up weights).
struct TcGemmArgs {
    const void* A;  int64_t lda;  int64_t M;
    const void* B;  int64_t ldb;  int64_t N;
    const void* A2; const void* B2;
    int64_t K;
    KSplit ks;
    bool swap;
    Epilogue epi;
    float* tail_ws;          // scratch for the split last wave (tc_tail_ws_bytes), or null
    size_t tail_ws_bytes;
};
bool tc_gemm_supported();
// A plain-store GEMM (normal orientation, one split) whose tiles leave a
// partial last wave splits the tiles of that wave along K over all CTAs; the
// chunks' fp32 partials need this much scratch (0: no split for this shape).
size_t tc_tail_ws_bytes(int64_t M, int64_t N, int64_t K, int sms);
cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st);

// TMA descriptor of a bf16 matrix [rows, cols] (row pitch ld elements), box
// 64 columns x box_rows rows, 128-byte swizzle; cached per argument tuple.
bool tma_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows);

// ------------------------------------------------ vocabulary-parallel lm_head
constexpr int kVocabTopkMax = 8;      // largest k of the candidate exchange

struct VocabTopkArgs {
    const void* X;          // [B, D] bf16 final hidden states
    const void* W;          // [V, D] bf16 lm_head weight, shard s = rows [s V/tp, (s+1) V/tp)
    int64_t B, D, V;
    int tp, k;
    int32_t* top_idx;       // [B, k]
    float* top_val;         // [B, k] or null
    int32_t* shard_idx;     // [tp, B, k] or null
    float* shard_val;       // [tp, B, k] or null
    void* ws;               // vocab_topk_ws_bytes(B, V, tp, k), 256-byte aligned
};
size_t vocab_topk_ws_bytes(int64_t B, int64_t V, int tp, int k);
// The GEMM + per-tile ranking kernel, then the per-shard / exchange merge kernel.
cudaError_t launch_vocab_topk(const VocabTopkArgs& a, cudaStream_t st);

// ------------------------------------------------ fused decode stack
constexpr float kRmsEpsilon = 1e-6f;  // RMSNorm eps of the decoder composition
constexpr int kFusedMaxLayers = 32;   // layers per launch (longer stacks take several launches)
constexpr int kFusedGridCap = 148;    // CTAs per launch at most; the workspace is sized for it

struct FusedShape {
    int64_t B, D, F;
    int n_q, n_kv, hd, tp;
};
// Shapes the fused decode stack handles (B <= 128, widths multiples of 64).
bool fused_stack_shape_ok(const FusedShape& s);
size_t fused_stack_ws_bytes(const FusedShape& s);
// Phase trace of instrumented builds (tpl_fused_trace_read); false otherwise.
constexpr int kFusedTraceEvents = 12;
bool fused_trace_read(void* host, size_t bytes);
// Test hook behind tpl_test_fused_fault (cta < 0: off; wait_ns <= 0: default limit).
void fused_test_fault(int cta, int phase, long long wait_ns);
// The whole stack in persistent cooperative launches (kFusedMaxLayers layers each).
// parallel: the parallel (PaLM) block y = x + Attn(RMSNorm(x)) + MLP(RMSNorm(x)).
cudaError_t launch_fused_stack(const FusedShape& s, const void* x, void* y, const void* const* Wqkv,
                               const void* const* Wo, const void* const* Wg, const void* const* Wu,
                               const void* const* Wd, int n_layers, bool parallel, void* ws, cudaStream_t st);

}  // namespace tpl
