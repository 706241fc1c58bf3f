// CUDA-core kernels: the weight-streaming row-dot kernel for small token
// counts (and the fp32 path), the ordered shard reduction, and RMSNorm.
#include <cuda_bf16.h>
#include <algorithm>

#include "epilogue.cuh"
#include "internal.h"

namespace tpl {
namespace {

constexpr int kWarps = 8;   // warps per block of the row-dot kernel

// 16-byte load that does not allocate in L1 (weights are read exactly once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_cached(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

template <typename T> struct Lanes;
template <> struct Lanes<__nv_bfloat16> {
    static constexpr int kN = 8;
    __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <> struct Lanes<float> {
    static constexpr int kN = 4;
    __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Each warp owns RW output features (rows of W; with DUAL the same rows of W
// and W1) and computes their dot products with NB tokens over one K split.
// Lanes stride over K in 16-byte vectors; U vectors per lane are in flight per
// row.  The warp's sums are reduced with shuffles and stored by distinct lanes.
template <typename T, int NB, int RW, bool DUAL>
__global__ void __launch_bounds__(kWarps * 32) rowdot_kernel(const RowdotArgs a) {
    constexpr int EPV = Lanes<T>::kN;
    constexpr int R = DUAL ? 2 * RW : RW;
    constexpr int U = 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.epi.zero_words && blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < a.epi.zero_count; i += blockDim.x) a.epi.zero_words[i] = 0u;
    const int64_t f0 = ((int64_t)blockIdx.x * kWarps + warp) * RW;
    if (f0 >= a.N) return;
    const int split = blockIdx.y;
    const int sh = split / a.ks.sub, j = split - sh * a.ks.sub;
    const int64_t kbeg = sh * a.ks.k_shard + (int64_t)j * a.ks.k_chunk;
    const int64_t kend = min(kbeg + a.ks.k_chunk, (int64_t)(sh + 1) * a.ks.k_shard);

    const T* W = reinterpret_cast<const T*>(a.W);
    const T* W1 = reinterpret_cast<const T*>(a.W1);
    const T* X = reinterpret_cast<const T*>(a.X);
    const T* wp[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = min(f0 + (r % RW), a.N - 1);
        wp[r] = ((DUAL && r >= RW) ? W1 : W) + row * a.ldw;
    }
    float acc[R][NB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;

    for (int64_t k = kbeg + lane * EPV; k < kend; k += 32 * EPV * U) {
        uint4 wv[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t kk = k + u * 32 * EPV;
#pragma unroll
            for (int r = 0; r < R; ++r)
                wv[u][r] = kk < kend ? ld_stream(wp[r] + kk) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t kk = k + u * 32 * EPV;
            if (kk >= kend) break;
            float wf[R][EPV];
#pragma unroll
            for (int r = 0; r < R; ++r) Lanes<T>::unpack(wv[u][r], wf[r]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < a.nb) {
                    float xf[EPV];
                    Lanes<T>::unpack(ld_cached(X + (int64_t)b * a.ldx + kk), xf);
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int e = 0; e < EPV; ++e) acc[r][b] = fmaf(wf[r][e], xf[e], acc[r][b]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[r][b] = warp_sum(acc[r][b]);

#pragma unroll
    for (int r = 0; r < RW; ++r) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int idx = r * NB + b;
            const int64_t f = f0 + r;
            if (lane == (idx & 31) && b < a.nb && f < a.N) {
                if (DUAL)
                    store_pair(a.epi, split, a.tok0 + b, f, acc[r][b], acc[r + (DUAL ? RW : 0)][b]);
                else
                    store_value(a.epi, split, a.tok0 + b, f, acc[r][b]);
            }
        }
    }
}

template <typename T, bool DUAL>
cudaError_t launch_rowdot_t(const RowdotArgs& a, cudaStream_t st) {
    constexpr int RW = DUAL ? 2 : 4;
    dim3 grid((unsigned)((a.N + kWarps * RW - 1) / (kWarps * RW)), (unsigned)(a.ks.tp * a.ks.sub));
    dim3 block(kWarps * 32);
    if (a.nb <= 1)
        rowdot_kernel<T, 1, RW, DUAL><<<grid, block, 0, st>>>(a);
    else if (a.nb <= 2)
        rowdot_kernel<T, 2, RW, DUAL><<<grid, block, 0, st>>>(a);
    else if (a.nb <= 4)
        rowdot_kernel<T, 4, RW, DUAL><<<grid, block, 0, st>>>(a);
    else
        rowdot_kernel<T, 8, RW, DUAL><<<grid, block, 0, st>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ reduce

__device__ __forceinline__ float ld_any(const void* p, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
                : reinterpret_cast<const float*>(p)[i];
}

// Sum of the split partials of 4 consecutive elements at flat index i:
// per shard over its chunks in ascending order, then over shards in ascending
// order.  All plane loads of a shard are issued before they are added.
__device__ __forceinline__ float4 sum_planes(const float* ws, int64_t n, int64_t i, int tp, int sub,
                                             float* shard_out) {
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < tp; ++s) {
        const float* base = ws + (int64_t)(s * sub) * n + i;
        float4 p = *reinterpret_cast<const float4*>(base);
        int jj = 1;
        for (; jj + 3 < sub; jj += 4) {
            const float4 q0 = *reinterpret_cast<const float4*>(base + (int64_t)jj * n);
            const float4 q1 = *reinterpret_cast<const float4*>(base + (int64_t)(jj + 1) * n);
            const float4 q2 = *reinterpret_cast<const float4*>(base + (int64_t)(jj + 2) * n);
            const float4 q3 = *reinterpret_cast<const float4*>(base + (int64_t)(jj + 3) * n);
            p.x += q0.x; p.y += q0.y; p.z += q0.z; p.w += q0.w;
            p.x += q1.x; p.y += q1.y; p.z += q1.z; p.w += q1.w;
            p.x += q2.x; p.y += q2.y; p.z += q2.z; p.w += q2.w;
            p.x += q3.x; p.y += q3.y; p.z += q3.z; p.w += q3.w;
        }
        for (; jj < sub; ++jj) {
            const float4 q = *reinterpret_cast<const float4*>(base + (int64_t)jj * n);
            p.x += q.x; p.y += q.y; p.z += q.z; p.w += q.w;
        }
        if (shard_out) *reinterpret_cast<float4*>(shard_out + (int64_t)s * n + i) = p;
        if (s == 0) y = p;
        else { y.x += p.x; y.y += p.y; y.z += p.z; y.w += p.w; }
    }
    return y;
}

// Elementwise: y[i] = residual[i] + sum of partials; with ws_up,
// y = silu(sum ws) * sum ws_up instead.  Four consecutive elements per thread.
__global__ void reduce_kernel(const ReduceArgs a) {
    const int64_t n = a.rows * a.cols;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
        const float4 y = sum_planes(a.ws, n, i, a.tp, a.sub, a.shard_out);
        float v[4] = {y.x, y.y, y.z, y.w};
        if (a.ws_up) {
            const float4 u = sum_planes(a.ws_up, n, i, a.tp, a.sub, nullptr);
            const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = silu_f(v[e]) * uu[e];
        }
        if (a.residual) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] += ld_any(a.residual, i + e, 1);
        }
        if (a.mode == TPL_ALLREDUCE) {
#pragma unroll
            for (int e = 0; e < 4; ++e) put(a.y, i + e, v[e], a.y_bf16);
        } else {
            const int64_t cw = a.cols / a.tp;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t row = (i + e) / a.cols, c = (i + e) - row * a.cols;
                const int64_t s = c / cw;
                put(a.y, s * a.rows * cw + row * cw + (c - s * cw), v[e], a.y_bf16);
            }
        }
    }
}

// The plain shard sum (one split per shard, no gate/up pair, no per-shard
// copies, no RMSNorm): y = residual + P_0 + P_1 + ... + P_{TP-1}, added in
// ascending shard order like reduce_kernel, four consecutive elements per
// item and two items per thread, with all 2 TP partial loads issued before
// the first add (streaming loads: every partial is read once), so enough
// bytes are in flight to keep HBM busy.
template <int TP>
__global__ void __launch_bounds__(256) shard_sum_kernel(const ReduceArgs a) {
    const int64_t n4 = a.rows * a.cols / 4;
    const float4* ws = reinterpret_cast<const float4*>(a.ws);
    const int64_t cw = a.mode == TPL_ALLREDUCE ? a.cols : a.cols / TP;
    const int64_t step = (int64_t)gridDim.x * blockDim.x * 2;
    for (int64_t j0 = (int64_t)blockIdx.x * blockDim.x * 2 + threadIdx.x; j0 < n4; j0 += step) {
        float4 v[2][TP];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t j = j0 + (int64_t)u * blockDim.x;
            if (j < n4) {
#pragma unroll
                for (int s = 0; s < TP; ++s) v[u][s] = __ldcs(ws + (int64_t)s * n4 + j);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t j = j0 + (int64_t)u * blockDim.x;
            if (j >= n4) continue;
            float4 y = v[u][0];
#pragma unroll
            for (int s = 1; s < TP; ++s) { y.x += v[u][s].x; y.y += v[u][s].y; y.z += v[u][s].z; y.w += v[u][s].w; }
            const int64_t i = j * 4;
            if (a.residual) {
                const uint2 r = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.residual) + i);
                y.x += __uint_as_float(r.x << 16); y.y += __uint_as_float(r.x & 0xFFFF0000u);
                y.z += __uint_as_float(r.y << 16); y.w += __uint_as_float(r.y & 0xFFFF0000u);
            }
            // four consecutive elements lie in one row and, for reduce-scatter,
            // in one column block (cw is a multiple of 4)
            int64_t o = i;
            if (a.mode != TPL_ALLREDUCE) {
                const int64_t row = i / a.cols, c = i - row * a.cols, sb = c / cw;
                o = sb * a.rows * cw + row * cw + (c - sb * cw);
            }
            if (a.y_bf16) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y), hi = __floats2bfloat162_rn(y.z, y.w);
                uint2 w;
                w.x = *reinterpret_cast<const uint32_t*>(&lo);
                w.y = *reinterpret_cast<const uint32_t*>(&hi);
                __stcs(reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.y) + o), w);
            } else {
                __stcs(reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + o), y);
            }
        }
    }
}

constexpr int kNormThreads = kNormCols / 4;     // 4 columns per thread

__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    if (threadIdx.x < 32) {
        t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        t = warp_sum(t);
    }
    return t;   // valid in thread 0
}

// Grid (column blocks, rows).  Each block: y = bf16(residual + sum of
// partials) for its kNormCols columns (or y = x when tp == 0), and its share of
// the row's sum of squares of the ROUNDED values, written to its own slot.  The
// last block of a row to finish (atomic ticket; nothing waits) adds the slots
// in block order -- the same sum whatever order the blocks ran in -- and writes
// the row's RMSNorm scale: scale_out = 1 / sqrt(mean(y^2) + eps).  row_cnt
// starts at zero (the kernel that produced the partials zeroes it) and the
// last block resets it.
__global__ void __launch_bounds__(kNormThreads) reduce_norm_kernel(const ReduceArgs a) {
    const int64_t row = blockIdx.y;
    const int64_t n = a.rows * a.cols;
    const int64_t c = ((int64_t)blockIdx.x * kNormThreads + threadIdx.x) * 4;
    const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(a.residual);
    __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(a.y);
    __shared__ float red[32];
    __shared__ unsigned int ticket;
    float ss = 0.f;
    if (c < a.cols) {
        const int64_t i = row * a.cols + c;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (a.tp > 0) {
            const float4 p = sum_planes(a.ws, n, i, a.tp, a.sub, a.shard_out);
            v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
        }
        if (res) {
            const uint2 rv = *reinterpret_cast<const uint2*>(res + i);
            v[0] += __uint_as_float(rv.x << 16); v[1] += __uint_as_float(rv.x & 0xFFFF0000u);
            v[2] += __uint_as_float(rv.y << 16); v[3] += __uint_as_float(rv.y & 0xFFFF0000u);
        }
        __nv_bfloat16 b[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            b[e] = __float2bfloat16_rn(v[e]);
            const float r = __bfloat162float(b[e]);
            ss = fmaf(r, r, ss);
        }
        if (y) {
            uint2 w;
            w.x = (uint32_t)__bfloat16_as_ushort(b[0]) | ((uint32_t)__bfloat16_as_ushort(b[1]) << 16);
            w.y = (uint32_t)__bfloat16_as_ushort(b[2]) | ((uint32_t)__bfloat16_as_ushort(b[3]) << 16);
            *reinterpret_cast<uint2*>(y + i) = w;
        }
    }
    const float bsum = block_sum(ss, red);
    float* slots = a.row_slots + row * gridDim.x;
    if (threadIdx.x == 0) {
        slots[blockIdx.x] = bsum;
        __threadfence();
        ticket = atomicAdd(a.row_cnt + row, 1u);
    }
    __syncthreads();
    if (ticket != gridDim.x - 1) return;
    // last block of this row: every other block's y and slot are visible
    __threadfence();
    if (threadIdx.x == 0) {
        float total = 0.f;
        for (unsigned b = 0; b < gridDim.x; ++b) total += __ldcg(slots + b);
        a.scale_out[row] = 1.0f / sqrtf(total / (float)a.cols + a.eps);
        a.row_cnt[row] = 0u;
    }
}

// Zero the row accumulators before a plain RMSNorm (no producing GEMM precedes it).
__global__ void zero_words_kernel(unsigned int* p, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0u;
}

}  // namespace

cudaError_t launch_rowdot(const RowdotArgs& a, bool bf16, cudaStream_t st) {
    const bool dual = a.epi.mode == EPI_SWIGLU || a.epi.mode == EPI_PARTIAL2;
    if (bf16)
        return dual ? launch_rowdot_t<__nv_bfloat16, true>(a, st) : launch_rowdot_t<__nv_bfloat16, false>(a, st);
    return dual ? launch_rowdot_t<float, true>(a, st) : launch_rowdot_t<float, false>(a, st);
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t st) {
    if (a.scale_out) {
        dim3 grid((unsigned)norm_blocks(a.cols), (unsigned)a.rows);
        reduce_norm_kernel<<<grid, kNormThreads, 0, st>>>(a);
        return cudaGetLastError();
    }
    const int64_t n4 = (a.rows * a.cols + 3) / 4;
    const DeviceCtx* ctx = device_ctx();
    const int64_t sms = ctx ? ctx->num_sms : 148;
    if (a.sub == 1 && !a.ws_up && !a.shard_out && a.tp >= 1 && a.tp <= 8 && a.cols % 4 == 0) {
        const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((n4 + 511) / 512, sms * 8));
        switch (a.tp) {
        case 1: shard_sum_kernel<1><<<blocks, 256, 0, st>>>(a); break;
        case 2: shard_sum_kernel<2><<<blocks, 256, 0, st>>>(a); break;
        case 3: shard_sum_kernel<3><<<blocks, 256, 0, st>>>(a); break;
        case 4: shard_sum_kernel<4><<<blocks, 256, 0, st>>>(a); break;
        case 5: shard_sum_kernel<5><<<blocks, 256, 0, st>>>(a); break;
        case 6: shard_sum_kernel<6><<<blocks, 256, 0, st>>>(a); break;
        case 7: shard_sum_kernel<7><<<blocks, 256, 0, st>>>(a); break;
        default: shard_sum_kernel<8><<<blocks, 256, 0, st>>>(a); break;
        }
        return cudaGetLastError();
    }
    const int64_t max_blocks = sms * 16;
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((n4 + 127) / 128, max_blocks));
    reduce_kernel<<<blocks, 128, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* x, float* scale, int64_t rows, int64_t cols, float eps,
                           unsigned int* rowacc, cudaStream_t st) {
    zero_words_kernel<<<1, 256, 0, st>>>(rowacc, (int)rows);
    ReduceArgs a{};
    a.ws = nullptr;
    a.rows = rows;
    a.cols = cols;
    a.tp = 0;
    a.sub = 1;
    a.residual = x;
    a.y = nullptr;
    a.scale_out = scale;
    a.eps = eps;
    a.row_cnt = rowacc;
    a.row_slots = reinterpret_cast<float*>(rowacc + rows);
    return launch_reduce(a, st);
}

}  // namespace tpl
