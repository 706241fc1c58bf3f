// Weight-only int8 path: symmetric per-(row, group) quantisation and the
// swapped tensor-core GEMM that streams int8 weights and widens them to bf16 in
// shared memory for tcgen05.mma.kind::f16.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace tpl {

// Q[r, c] = clamp(round_even(W[r, c] / s[r, g]), -127, 127) with
// s[r, g] = amax(|W[r, group g]|) / 127 in float32; g = c / (cols / groups).
cudaError_t launch_quantize_w8(const void* W, int64_t rows, int64_t cols, int groups, int8_t* Q, float* scale,
                               cudaStream_t st);

struct W8GemmArgs {
    const int8_t* Q;   const int8_t* Q2;     // [M, K] int8 weights (Q2: up rows, DUAL only)
    const float* scale; const float* scale2; // [M, groups]
    int groups;                              // 1, or ks.tp (one scale per row and shard)
    int64_t M;                               // weight rows (output features)
    const void* X;  int64_t ldx;  int64_t N; // [N tokens, K] bf16 activations
    int64_t K;
    KSplit ks;
    Epilogue epi;                            // EPI_SWIGLU / EPI_PARTIAL2 (DUAL), EPI_STORE / EPI_PARTIAL
};
cudaError_t launch_w8_gemm(const W8GemmArgs& a, cudaStream_t st);

// The same product on CUDA cores for at most kW8RowdotMaxTokens tokens (fp32
// FMAs on the exactly widened codes); same arguments and epilogues.
constexpr int kW8RowdotMaxTokens = 2;
cudaError_t launch_w8_rowdot(const W8GemmArgs& a, cudaStream_t st);

}  // namespace tpl
