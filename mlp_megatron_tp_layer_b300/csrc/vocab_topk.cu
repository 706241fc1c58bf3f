// Vocabulary-parallel lm_head with a candidate exchange instead of a logit
// gather ("Lecture 4 - Distributed Serving", S4.5): shard s owns the vocabulary
// rows [s V/tp, (s+1) V/tp) of W[V, D]; it ranks only its own logits
// x . W[v] and keeps its top-k, and the tp shard lists per token are merged
// into the global top-k.  The logits themselves never reach HBM.
//
// Kernel 1 (vocab_topk_gemm_kernel): persistent TMA + tcgen05 GEMM in the
// swapped orientation -- 128 vocabulary rows of W are the M operand, the
// tokens (padded to N = 16..128 by the TMA zero fill) the N operand -- so W
// streams from HBM once per call for B <= 128.  Tiles never straddle a shard:
// the tile list is shard-major and a shard's last tile masks the rows past its
// end.  The epilogue ranks each tile's 128 logits per token: the four
// epilogue warps turn their TMEM rows into order-preserving integer keys and
// store them transposed in shared memory (one column per token, padded so both
// the writes and the column scans are free of bank conflicts); each of the 128
// threads then scans a slice of one column sequentially, keeping its best k,
// and one thread per token merges the slices.  The tile's k best candidates
// per token go to global memory as packed 64-bit words.  No warp-collective
// rounds are needed, so the ranking stays well inside the time the next tile's
// weights take to arrive.
//
// Kernel 2 (vocab_topk_merge_kernel): one block per (token, shard) reduces
// that shard's tile candidates to the shard's top-k (the list a device would
// send); the last block of each token to finish (an atomic ticket, no
// waiting) merges the tp shard lists into the final top-k.  It is launched as
// a programmatic dependent of kernel 1, so its launch overlaps the GEMM's
// last tiles; its blocks wait (griddepcontrol.wait) for the GEMM grid to
// complete before reading any candidate.
//
// Candidate word: (order key of the fp32 logit) << 32 | (0xFFFFFFFF - index).
// Comparing words as unsigned integers orders by logit, larger first, and
// equal logits by lower vocabulary index; 0 marks an empty slot.  -0 is
// turned into +0 before keying, so the two compare equal.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace tpl {
namespace {

constexpr int VT_BM = 128;          // vocabulary rows per tile (TMEM lanes)
constexpr int VT_BK = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int VT_THREADS = 192;     // warp 0 TMA, warp 1 TMEM + MMA, warps 2..5 epilogue
constexpr int VT_MERGE_THREADS = 256;

struct VtParams {
    int64_t B;              // tokens
    int64_t Vs;             // vocabulary rows per shard
    int k;                  // candidates kept per (tile or shard, token)
    int tiles_per_shard;    // ceil(Vs / 128)
    int m_tiles;            // tp * tiles_per_shard
    int64_t total_tiles;    // m_tiles * token tiles
    int nkb;                // ceil(D / 64)
    unsigned long long* cand;   // [m_tiles][B][k]
    unsigned int* tickets;      // [B], zeroed here for the merge kernel
    int n_tickets;
    unsigned int* err;
};

template <int BN>
struct VtCfg {
    static constexpr int A_BYTES = VT_BM * VT_BK * 2;               // 16 KB of W
    static constexpr int B_BYTES = BN * VT_BK * 2;                  // tokens
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int CH = BN >= 32 ? 32 : 16;                    // columns per TMEM load
    static constexpr int KPAD = VT_BM + 1;                           // padded key column: conflict-free both ways
    static constexpr int KEY_BYTES = CH * KPAD * 4;                  // one chunk's keys, column-major
    static constexpr int CAND_BYTES = VT_BM * kVocabTopkMax * 8;     // (row group, column) lists
    static constexpr int EPI_BYTES = ((KEY_BYTES + 15) & ~15) + CAND_BYTES;
    static constexpr int STAGES_RAW = (218 * 1024 - EPI_BYTES - 1280) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 10 ? 10 : STAGES_RAW;
    static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128 : 256;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 256 + 1024;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "token tile must be 16..128 in steps of 16");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ uint32_t order_key(float f) {
    if (f == 0.0f) f = 0.0f;                                          // -0 ranks with +0
    const uint32_t u = __float_as_uint(f);
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return key > 1u ? key : 1u;                                       // 0 is reserved for "empty"
}
__device__ __forceinline__ unsigned long long pack(uint32_t key, uint32_t index) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - index);
}
__device__ __forceinline__ void unpack(unsigned long long w, int32_t& index, float& value) {
    if (w == 0ull) { index = -1; value = __uint_as_float(0xFF800000u); return; }
    const uint32_t key = (uint32_t)(w >> 32);
    index = (int32_t)(0xFFFFFFFFu - (uint32_t)(w & 0xFFFFFFFFull));
    value = __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// bar.sync / bar.red over the four epilogue warps only (named barrier 1).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_all(bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred a, b;\n\t"
        "setp.ne.u32 a, %1, 0;\n\t"
        "bar.red.and.pred b, 1, 128, a;\n\t"
        "selp.u32 %0, 1, 0, b;\n\t}"
        : "=r"(r) : "r"((uint32_t)p) : "memory");
    return r != 0;
}

// Insert w into the descending list L[0..N), dropping the smallest.
template <int N>
__device__ __forceinline__ void list_insert(unsigned long long (&L)[N], unsigned long long w) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const unsigned long long hi = L[i] > w ? L[i] : w;
        w = L[i] > w ? w : L[i];
        L[i] = hi;
    }
}

// Rank one chunk of CH token columns of a 128-row tile (keys already in
// s_key, column-major with pitch KPAD).  Thread et scans rows
// [g CH, (g+1) CH) of column c = et % CH (g = et / CH) and keeps its KL best
// (KL >= k); after a barrier, thread c < ncols merges the 128 / CH lists of its
// column and writes the column's k best words to gout[c k ..].  Rows are
// scanned in ascending order and words compare by (key, lower index), so
// equal logits resolve to the lower vocabulary index.
template <int KL, int CH, int KPAD>
__device__ __forceinline__ void rank_chunk(const uint32_t* s_key, unsigned long long* s_cand, int et, int k,
                                           uint32_t vtile, unsigned long long* gout, int ncols) {
    constexpr int G = VT_BM / CH;
    const int c = et % CH, g = et / CH;
    const uint32_t* col = s_key + c * KPAD + g * CH;
    const uint32_t row0 = vtile + (uint32_t)(g * CH);
    unsigned long long L[KL];
    if (KL == 1) {
        uint32_t best = 0u;
        int at = 0;
#pragma unroll 8
        for (int r = 0; r < CH; ++r) {
            const uint32_t key = col[r];
            if (key > best) { best = key; at = r; }
        }
        L[0] = best ? pack(best, row0 + at) : 0ull;
    } else {
#pragma unroll
        for (int i = 0; i < KL; ++i) L[i] = 0ull;
#pragma unroll 4
        for (int r = 0; r < CH; ++r) {
            const uint32_t key = col[r];
            if (key) list_insert<KL>(L, pack(key, row0 + r));
        }
    }
#pragma unroll
    for (int i = 0; i < KL; ++i) s_cand[(g * CH + c) * KL + i] = L[i];
    epi_sync();
    if (et < ncols) {                       // et < CH: this thread owns column et (g == 0)
        if (KL == 1) {
            unsigned long long best = 0ull;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const unsigned long long w = s_cand[gg * CH + c];
                best = w > best ? w : best;
            }
            gout[c] = best;
        } else {
            int h[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) h[gg] = 0;
            for (int i = 0; i < k; ++i) {
                unsigned long long best = 0ull;
                int bg = -1;
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    const unsigned long long w = h[gg] < KL ? s_cand[(gg * CH + c) * KL + h[gg]] : 0ull;
                    if (w > best) { best = w; bg = gg; }
                }
                gout[c * k + i] = best;
#pragma unroll
                for (int gg = 0; gg < G; ++gg) h[gg] += (gg == bg) ? 1 : 0;
            }
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(VT_THREADS, 1)
vocab_topk_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const VtParams p) {
    using C = VtCfg<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* s_key = reinterpret_cast<uint32_t*>(smem + C::STAGES * C::STAGE_BYTES);
    unsigned long long* s_cand =
        reinterpret_cast<unsigned long long*>(smem + C::STAGES * C::STAGE_BYTES + ((C::KEY_BYTES + 15) & ~15));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* acc_full = bars + 2 * C::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the merge kernel that follows on the stream counts finished shards here
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.n_tickets; i += blockDim.x) p.tickets[i] = 0u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&acc_full[a]), 1);
            mbar_init(smem_addr(&acc_empty[a]), 4);
        }
        mbar_init(smem_addr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the merge kernel may be scheduled now; it waits for this grid to complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    auto fail = [&]() {
        *abort_flag = 1;
        if (p.err) atomicOr(p.err, TPL_DEVERR_TIMEOUT);
    };
    // tile t -> (shard-major vocabulary tile, token tile)
    auto w_row = [&](int64_t t) {
        const int mg = (int)(t % p.m_tiles);
        const int s = mg / p.tiles_per_shard, lt = mg - s * p.tiles_per_shard;
        return (int)(s * p.Vs + (int64_t)lt * VT_BM);
    };

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int issued_tail = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                const int wr = w_row(t);
                const int xr = (int)(t / p.m_tiles) * BN;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(smem_addr(&empty[stage]), phase ^ 1, abort_flag)) { ok = false; break; }
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_expect_tx(fb, C::STAGE_BYTES);
                    uint8_t* st = smem + stage * C::STAGE_BYTES;
                    tma_load_hint(smem_addr(st), &tmW, fb, kb * VT_BK, wr, pol_w);
                    tma_load_hint(smem_addr(st + C::A_BYTES), &tmX, fb, kb * VT_BK, xr, pol_x);
                    issued_tail = min(issued_tail + 1, C::STAGES);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                fail();
                for (int i = 0; i < issued_tail; ++i) {
                    if (--stage < 0) { stage = C::STAGES - 1; phase ^= 1; }
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_addr(&full[stage]), phase) && globaltimer() - t0 < kWaitLimitNs) {}
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(VT_BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(smem_addr(&acc_empty[acc]), acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(smem_addr(&full[stage]), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < VT_BK / 16; ++kk)
                        mma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), idesc, (kb | kk) ? 1u : 0u);
                    mma_commit(smem_addr(&empty[stage]));
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_addr(&acc_full[acc]));
            }
            if (!ok) fail();
            mma_commit(smem_addr(drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_addr(drain), 0) && globaltimer() - t0 < kWaitLimitNs) {}
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lanes 32q..32q+31 = tile rows
        const int et = threadIdx.x - 64;        // 0..127 across the four epilogue warps
        const int k = p.k;
        int it = 0;
        for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // the four warps leave together, so the named barriers below never
            // wait for a warp that has given up
            const bool ok = epi_all(mbar_wait(smem_addr(&acc_full[acc]), acc_phase, abort_flag));
            if (!ok) { if (et == 0) fail(); break; }
            tc_fence_after();
            const int mg = (int)(t % p.m_tiles);
            const int s = mg / p.tiles_per_shard, lt = mg - s * p.tiles_per_shard;
            const int64_t tok0 = (t / p.m_tiles) * BN;
            const int64_t local0 = (int64_t)lt * VT_BM + q * 32;           // shard-local row of lane 0
            const bool row_ok = local0 + lane < p.Vs;
            const uint32_t vtile = (uint32_t)(s * p.Vs + (int64_t)lt * VT_BM);   // vocabulary index of tile row 0
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            float v[32];
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += C::CH) {
                if (C::CH == 32) tmem_ld32(tbase + c0, v); else tmem_ld16(tbase + c0, v);
                if (c0 + C::CH >= BN) {            // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&acc_empty[acc]));
                }
                // keys to shared memory, transposed: column j holds the tile's 128 rows
#pragma unroll
                for (int j = 0; j < C::CH; ++j) {
                    const bool live = row_ok && tok0 + c0 + j < p.B;
                    s_key[j * C::KPAD + q * 32 + lane] = live ? order_key(v[j]) : 0u;
                }
                epi_sync();
                const int64_t left = p.B - (tok0 + c0);
                const int ncols = left < C::CH ? (int)left : C::CH;
                unsigned long long* gout = p.cand + ((int64_t)mg * p.B + tok0 + c0) * k;
                if (k == 1) rank_chunk<1, C::CH, C::KPAD>(s_key, s_cand, et, k, vtile, gout, ncols);
                else if (k == 2) rank_chunk<2, C::CH, C::KPAD>(s_key, s_cand, et, k, vtile, gout, ncols);
                else if (k <= 4) rank_chunk<4, C::CH, C::KPAD>(s_key, s_cand, et, k, vtile, gout, ncols);
                else rank_chunk<8, C::CH, C::KPAD>(s_key, s_cand, et, k, vtile, gout, ncols);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Block-wide top-k of the union of the threads' descending lists: k rounds of
// block max, the owner of each winner popping it.  Writes out[0..k) (shared).
__device__ void block_topk(unsigned long long (&L)[kVocabTopkMax], int k, unsigned long long* out,
                           unsigned long long* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = VT_MERGE_THREADS / 32;
    for (int i = 0; i < k; ++i) {
        unsigned long long m = L[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, m, o);
            m = y > m ? y : m;
        }
        if (lane == 0) red[warp] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long b = red[0];
            for (int w = 1; w < NW; ++w) b = red[w] > b ? red[w] : b;
            out[i] = b;
        }
        __syncthreads();
        const unsigned long long win = out[i];
        if (win != 0ull && L[0] == win) {            // words are unique, so one owner
#pragma unroll
            for (int j = 0; j + 1 < kVocabTopkMax; ++j) L[j] = L[j + 1];
            L[kVocabTopkMax - 1] = 0ull;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(VT_MERGE_THREADS)
vocab_topk_merge_kernel(const unsigned long long* __restrict__ cand, unsigned long long* shard_best,
                        unsigned int* tickets, int64_t B, int tp, int tiles_per_shard, int k, int32_t* top_idx,
                        float* top_val, int32_t* shard_idx, float* shard_val) {
    __shared__ unsigned long long s_out[kVocabTopkMax];
    __shared__ unsigned long long s_red[VT_MERGE_THREADS / 32];
    __shared__ int s_last;
    const int64_t b = blockIdx.x;
    const int s = blockIdx.y;
    // launched early behind the GEMM: wait until it has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // this shard's top-k for token b: the "local maximum / top-k" of one device
    unsigned long long L[kVocabTopkMax];
#pragma unroll
    for (int i = 0; i < kVocabTopkMax; ++i) L[i] = 0ull;
    const int n = tiles_per_shard * k;
    for (int c = threadIdx.x; c < n; c += VT_MERGE_THREADS) {
        const int lt = c / k, i = c - lt * k;
        list_insert<kVocabTopkMax>(L, cand[(((int64_t)s * tiles_per_shard + lt) * B + b) * k + i]);
    }
    block_topk(L, k, s_out, s_red);
    if (threadIdx.x < k) {
        const unsigned long long w = s_out[threadIdx.x];
        shard_best[((int64_t)s * B + b) * k + threadIdx.x] = w;
        if (shard_idx || shard_val) {
            int32_t ix;
            float val;
            unpack(w, ix, val);
            if (shard_idx) shard_idx[((int64_t)s * B + b) * k + threadIdx.x] = ix;
            if (shard_val) shard_val[((int64_t)s * B + b) * k + threadIdx.x] = val;
        }
    }

    // exchange: the last shard of token b to finish merges the tp lists
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&tickets[b], 1u) == (unsigned)(tp - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < kVocabTopkMax; ++i) L[i] = 0ull;
    for (int c = threadIdx.x; c < tp * k; c += VT_MERGE_THREADS) {
        const int ss = c / k, i = c - ss * k;
        list_insert<kVocabTopkMax>(L, __ldcg(shard_best + ((int64_t)ss * B + b) * k + i));
    }
    block_topk(L, k, s_out, s_red);
    if (threadIdx.x < k) {
        int32_t ix;
        float val;
        unpack(s_out[threadIdx.x], ix, val);
        top_idx[b * k + threadIdx.x] = ix;
        if (top_val) top_val[b * k + threadIdx.x] = val;
    }
}

template <int BN>
cudaError_t launch_bn(const VocabTopkArgs& a, const VtParams& p0, cudaStream_t st) {
    using C = VtCfg<BN>;
    const DeviceCtx* ctx = device_ctx();
    if (!ctx) return cudaErrorNoDevice;
    static bool attr_set[64] = {};
    if (ctx->device < 64 && !attr_set[ctx->device]) {
        const cudaError_t e = cudaFuncSetAttribute(vocab_topk_gemm_kernel<BN>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[ctx->device] = true;
    }
    CUtensorMap mW, mX;
    if (!tma_map_bf16(&mW, a.W, a.V, a.D, a.D, VT_BM)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(&mX, a.X, a.B, a.D, a.D, BN)) return cudaErrorInvalidValue;
    VtParams p = p0;
    const int64_t n_tiles = (a.B + BN - 1) / BN;
    p.total_tiles = (int64_t)p.m_tiles * n_tiles;
    p.err = ctx->err_word;
    const int64_t grid = std::min<int64_t>(p.total_tiles, ctx->num_sms);
    vocab_topk_gemm_kernel<BN><<<(unsigned)grid, VT_THREADS, C::SMEM_BYTES, st>>>(mW, mX, p);
    return cudaGetLastError();
}

}  // namespace

size_t vocab_topk_ws_bytes(int64_t B, int64_t V, int tp, int k) {
    const int64_t tps = (V / tp + VT_BM - 1) / VT_BM;
    const size_t cand = (size_t)tp * tps * B * k * 8;
    const size_t shard = (size_t)tp * B * k * 8;
    const size_t tick = (size_t)B * 4;
    auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
    return up(cand) + up(shard) + up(tick);
}

cudaError_t launch_vocab_topk(const VocabTopkArgs& a, cudaStream_t st) {
    const int64_t Vs = a.V / a.tp;
    const int64_t tps = (Vs + VT_BM - 1) / VT_BM;
    auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(ws);
    unsigned long long* shard_best =
        reinterpret_cast<unsigned long long*>(ws + up((size_t)a.tp * tps * a.B * a.k * 8));
    unsigned int* tickets = reinterpret_cast<unsigned int*>(
        reinterpret_cast<uint8_t*>(shard_best) + up((size_t)a.tp * a.B * a.k * 8));

    VtParams p{};
    p.B = a.B;
    p.Vs = Vs;
    p.k = a.k;
    p.tiles_per_shard = (int)tps;
    p.m_tiles = (int)(a.tp * tps);
    p.nkb = (int)((a.D + VT_BK - 1) / VT_BK);
    p.cand = cand;
    p.tickets = tickets;
    p.n_tickets = (int)a.B;
    cudaError_t e;
    if (a.B <= 16) e = launch_bn<16>(a, p, st);
    else if (a.B <= 32) e = launch_bn<32>(a, p, st);
    else if (a.B <= 64) e = launch_bn<64>(a, p, st);
    else e = launch_bn<128>(a, p, st);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)a.B, (unsigned)a.tp);
    cfg.blockDim = dim3(VT_MERGE_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int tp_i = a.tp, tps_i = (int)tps, k_i = a.k;
    const int64_t B_i = a.B;
    e = cudaLaunchKernelEx(&cfg, vocab_topk_merge_kernel, (const unsigned long long*)cand, shard_best, tickets, B_i,
                           tp_i, tps_i, k_i, a.top_idx, a.top_val, a.shard_idx, a.shard_val);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tpl
