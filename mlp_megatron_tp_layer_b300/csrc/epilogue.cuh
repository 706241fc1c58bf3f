// Device-side output stores shared by the CUDA-core and tensor-core kernels.
#pragma once

#include <cuda_bf16.h>
#include "internal.h"

namespace tpl {

// silu(z) = z * sigmoid(z) = z / (1 + exp(-z)); expf overflows to +inf for very
// negative z, which gives the correct limit -0.
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void put(void* base, int64_t off, float v, int bf16) {
    if (bf16)
        reinterpret_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(base)[off] = v;
}

// Packed QKV row r of token t: write to the shard block(s) holding it; a V row
// of KV group g is also the context-1 attention output of every Q head h with
// floor(h n_kv / n_q) == g (softmax over one key is 1).
__device__ __forceinline__ void store_qkv(const QkvMap& q, int64_t t, int64_t r, float v, int bf16) {
    const int hd = q.head_dim;
    const int head = (int)(r / hd);
    const int d = (int)(r - (int64_t)head * hd);
    // round once to the output type so every copy carries identical bits
    float vr = bf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
    if (head < q.n_q) {
        const int s = head / q.nq_s, j = head - s * q.nq_s;
        if (q.qkv_out) put(q.qkv_out, s * q.shard_stride + t * q.w_s + (int64_t)j * hd + d, vr, bf16);
        return;
    }
    const bool is_v = head >= q.n_q + q.n_kv;
    const int g = head - q.n_q - (is_v ? q.n_kv : 0);
    const int64_t base_col = (int64_t)(q.nq_s + (is_v ? q.kv_s : 0)) * hd + d;
    if (q.qkv_out) {
        if (q.tp <= q.n_kv) {
            const int s = g / q.kv_s, c = g - s * q.kv_s;
            put(q.qkv_out, s * q.shard_stride + t * q.w_s + base_col + (int64_t)c * hd, vr, bf16);
        } else {
            const int copies = q.tp / q.n_kv;
            for (int s = g * copies; s < (g + 1) * copies; ++s)
                put(q.qkv_out, s * q.shard_stride + t * q.w_s + base_col, vr, bf16);
        }
    }
    if (is_v) {
        const int per = q.n_q / q.n_kv;
        for (int h = g * per; h < (g + 1) * per; ++h)
            put(q.o_out, t * q.ldo_o + (int64_t)h * hd + d, vr, bf16);
    }
}

__device__ __forceinline__ void store_value(const Epilogue& e, int split, int64_t t, int64_t f, float v) {
    switch (e.mode) {
    case EPI_STORE: {
        const int64_t off = e.col_block > 0
            ? (f / e.col_block) * e.block_stride + t * e.ldo + (f % e.col_block)
            : t * e.ldo + f;
        put(e.out, off, v, e.out_bf16);
        break;
    }
    case EPI_PARTIAL:
        e.out32[(int64_t)split * e.split_stride + t * e.ldo + f] = v;
        break;
    case EPI_QKV:
        store_qkv(e.qkv, t, f, e.row_scale ? v * e.row_scale[t] : v, e.out_bf16);
        break;
    default:
        break;
    }
}

__device__ __forceinline__ void store_pair(const Epilogue& e, int split, int64_t t, int64_t f, float g, float u) {
    if (e.mode == EPI_SWIGLU) {
        if (e.row_scale) {
            const float s = e.row_scale[t];
            g *= s;
            u *= s;
        }
        put(e.out, t * e.ldo + f, silu_f(g) * u, e.out_bf16);
    } else {  // EPI_PARTIAL2
        const int64_t off = (int64_t)split * e.split_stride + t * e.ldo + f;
        e.out32[off] = g;
        e.out32b[off] = u;
    }
}

}  // namespace tpl
