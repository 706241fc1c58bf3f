// Weight-only int8 GEMM for decode (swapped orientation) and the row quantiser.
//
//   D[M, N] = (Q[M, K] . X[N, K]^T) * scale[M, group]
//
// Q streams from HBM as int8, half the bytes of bf16 ("Lecture 4 - Distributed
// Serving", S5.5: only the weights are quantised, to cut the time spent
// reading them).  tcgen05.mma has no int8 x bf16 form, so converter warps
// widen the weights to bf16 -- exactly: every integer in [-127, 127] is a bf16
// value -- and store them into tensor memory, where the MMA reads its A
// operand (weights are the M = 128 side, one row per TMEM lane); the tokens
// stay in shared memory as the B operand, and the per-row scale multiplies the
// fp32 accumulator in the epilogue.  Shared memory then carries only the TMA
// writes and one read of each int8 byte; a widened copy in shared memory
// would cost three times the int8 bytes again and makes shared-memory
// bandwidth, not HBM, the limit.
//
// Rings: the TMA ring (shared memory) carries the int8 weight tile(s) and the
// bf16 token tiles of one 128-wide K block per stage -- 128 bytes of each
// weight row, so every copy request moves as many bytes as on the bf16 path.
// The operand ring (TMEM columns) holds widened 64-wide K halves.  A TMA stage
// is released by the commit of the MMAs that read its token tiles, which
// come after the converters have read its weights.
//
// Warp roles (448 threads): 0 TMA producer; 1 TMEM owner + MMA issuer;
// 2-5 epilogue; 6-13 converters.  A warp reaches only the TMEM lanes
// 32*(w%4)..+31, so epilogue warp w reads and converter warp w writes the rows
// of that lane quarter; converter warps 6-9 take the first 32 K elements of a
// half, 10-13 the second.  Every wait is bounded; on expiry the CTA sets the
// sticky device error word, drains what it started, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "w8.h"

namespace tpl {
namespace {

constexpr int W8_BM = 128;          // weight rows per tile (TMEM lanes)
constexpr int W8_BK = 64;           // K elements per widened operand stage (one MMA group)
constexpr int W8_RK = 128;          // K elements per TMA stage (128 int8 bytes per row)
constexpr int W8_THREADS = 448;
constexpr int W8_CONV_WARPS = 8;
constexpr int W8_TMEM_COLS = 512;   // the whole TMEM of the SM (one CTA per SM)

struct W8Params {
    int64_t M, NB;
    int m_tiles, n_tiles, splits;
    int64_t total_tiles;
    KSplit ks;
    Epilogue epi;
    const float* scale;
    const float* scale2;
    int groups;
    unsigned int* err;
};

template <int BN, bool DUAL>
struct W8Cfg {
    static constexpr int NA = DUAL ? 2 : 1;
    static constexpr int Q_BYTES = W8_BM * W8_RK;                 // 16 KB int8 tile (128B-swizzled)
    static constexpr int X_HALF = BN * W8_BK * 2;                 // token tile of one 64-wide K half
    static constexpr int X_BYTES = 2 * X_HALF;                    // token tiles first in the stage
    static constexpr int RAW_BYTES = X_BYTES + NA * Q_BYTES;
    static constexpr int STAGES_RAW = (200 * 1024) / RAW_BYTES;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    // TMEM: accumulators (two if they fit beside four operand stages), then operand stages.
    // NCHAIN > 1 would spread the K slices over independent accumulators that
    // the epilogue adds up; measured back to back, MMAs into one accumulator run
    // as fast as into four, so one chain is used.
    static constexpr int NCHAIN = 1;
    static constexpr int ACC1 = DUAL ? 2 * BN : BN;               // one chain: [gate | up] or [out]
    static constexpr int ACC_COLS = NCHAIN * ACC1;
    static constexpr int A_COLS = NA * (W8_BK / 2);               // 64 bf16 = 32 columns per operand
    static constexpr int NACC = (2 * ACC_COLS + 4 * A_COLS <= W8_TMEM_COLS) ? 2 : 1;
    static constexpr int A_BASE = NACC * ACC_COLS;
    static constexpr int CSTAGES_RAW = (W8_TMEM_COLS - A_BASE) / A_COLS;
    static constexpr int CSTAGES = CSTAGES_RAW > 4 ? 4 : CSTAGES_RAW;
    static constexpr int SMEM_BYTES = STAGES * RAW_BYTES + 512 + 1024;
    static_assert(RAW_BYTES % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
    static_assert(STAGES >= 2 && CSTAGES >= 2, "ring depths");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "token tile 16..128 in steps of 16");
};

struct TileCoord { int sp, mt, nt; };
__device__ __forceinline__ TileCoord tile_coord(const W8Params& p, int64_t t) {
    const int64_t per_split = (int64_t)p.m_tiles * p.n_tiles;
    TileCoord c;
    c.sp = (int)(t / per_split);
    const int64_t r = t - (int64_t)c.sp * per_split;
    c.mt = (int)(r % p.m_tiles);      // m fastest: concurrent CTAs share the token tile
    c.nt = (int)(r / p.m_tiles);
    return c;
}
__device__ __forceinline__ void split_range(const W8Params& p, int sp, int64_t& k0, int& nkb) {
    const int sh = sp / p.ks.sub, j = sp - sh * p.ks.sub;
    k0 = sh * p.ks.k_shard + (int64_t)j * p.ks.k_chunk;
    const int64_t k1 = min(k0 + p.ks.k_chunk, (int64_t)(sh + 1) * p.ks.k_shard);
    nkb = (int)((k1 - k0 + W8_BK - 1) / W8_BK);
}

// The bounded wait, which first tests the phase without blocking (most waits
// of the MMA warp find their phase long complete).
__device__ __forceinline__ bool fast_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait(bar, parity, abort_flag);
}

// tcgen05.mma with the A operand in tensor memory (kind::f16, bf16 x bf16 -> fp32).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp writes lane base+i.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Widen 32 int8 weights of row r -- K elements 64 hh + 32 kq .. +31 of the
// 128-wide int8 row, itself 128B-swizzled by the copy (16-byte chunk c at
// position c ^ (r % 8)) -- into 16 words of bf16 pairs, lower K in the low
// half.  An int8 q becomes the float 2^23 + (q + 128) by placing its biased
// byte under the exponent bits of 2^23; subtracting 2^23 + 128 leaves q
// exactly, and since |q| <= 128 has at most eight significant bits its bf16
// value is the float's upper half.
__device__ __forceinline__ void widen(const uint8_t* q_row, int r, int hh, int kq, uint32_t (&out)[16]) {
    const int sw = r & 7;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int ci = 4 * hh + 2 * kq + j;                     // int8 chunk: 16 K elements
        const uint4 w = *reinterpret_cast<const uint4*>(q_row + ((ci ^ sw) << 4));
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t b = words[i] ^ 0x80808080u;
            const float f0 = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7540)) - 8388736.0f;
            const float f1 = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7541)) - 8388736.0f;
            const float f2 = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7542)) - 8388736.0f;
            const float f3 = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7543)) - 8388736.0f;
            out[8 * j + 2 * i] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
            out[8 * j + 2 * i + 1] = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
        }
    }
}

template <int BN, bool DUAL>
__global__ void __launch_bounds__(W8_THREADS, 1)
w8_gemm_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQ2,
               const __grid_constant__ CUtensorMap tmX, const W8Params p) {
    using C = W8Cfg<BN, DUAL>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw + C::STAGES * C::RAW_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* cfull = bars + 2 * C::STAGES;
    uint64_t* cempty = cfull + C::CSTAGES;
    uint64_t* acc_full = cempty + C::CSTAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int s = 0; s < C::CSTAGES; ++s) {
            mbar_init(smem_addr(&cfull[s]), W8_CONV_WARPS);   // one arrival per converter warp
            mbar_init(smem_addr(&cempty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&acc_full[a]), 1);
            mbar_init(smem_addr(&acc_empty[a]), 4);
        }
        mbar_init(smem_addr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmX);
        if (DUAL) prefetch_tmap(&tmQ2);
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), W8_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        if (p.err) atomicOr(p.err, TPL_DEVERR_TIMEOUT);
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
                const TileCoord c = tile_coord(p, t);
                int64_t k0;
                int nkb;
                split_range(p, c.sp, k0, nkb);
                const int am = c.mt * W8_BM;
                const int bn = c.nt * BN;
                for (int kb = 0; kb < nkb; kb += 2) {
                    const int halves = min(2, nkb - kb);
                    if (!fast_wait(smem_addr(&empty[stage]), phase ^ 1, abort_flag)) { ok = false; break; }
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_expect_tx(fb, C::NA * C::Q_BYTES + halves * C::X_HALF);
                    uint8_t* st = raw + stage * C::RAW_BYTES;
                    // elements of X, bytes of Q: both multiples of 64, so 16-byte aligned.  A
                    // lone last half still copies the whole 128-byte Q row span; the
                    // bytes past the split are never widened.
                    const int kx = (int)(k0 + kb * W8_BK);
                    tma_load_hint(smem_addr(st), &tmX, fb, kx, bn, pol_x);
                    if (halves == 2) tma_load_hint(smem_addr(st + C::X_HALF), &tmX, fb, kx + W8_BK, bn, pol_x);
                    tma_load_hint(smem_addr(st + C::X_BYTES), &tmQ, fb, kx, am, pol_w);
                    if (DUAL) tma_load_hint(smem_addr(st + C::X_BYTES + C::Q_BYTES), &tmQ2, fb, kx, am, pol_w);
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
            constexpr uint32_t idesc = make_idesc(W8_BM, BN);
            int stage = 0, cst = 0;
            uint32_t phase = 0, cph = 0;
            bool ok = true;
            int it = 0;
            for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++it) {
                const TileCoord c = tile_coord(p, t);
                int64_t k0;
                int nkb;
                split_range(p, c.sp, k0, nkb);
                const int acc = it % C::NACC;
                const uint32_t acc_phase = (it / C::NACC) & 1;
                if (!fast_wait(smem_addr(&acc_empty[acc]), acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * C::ACC_COLS;
                for (int kb = 0; kb < nkb && ok; kb += 2) {
                    const int halves = min(2, nkb - kb);
                    for (int hh = 0; hh < halves; ++hh) {
                        // widened weights in TMEM (the converters saw the stage land);
                        // the token tiles' own barrier is already complete by then and
                        // is observed once per stage
                        if (!fast_wait(smem_addr(&cfull[cst]), cph, abort_flag) ||
                            (hh == 0 && !fast_wait(smem_addr(&full[stage]), phase, abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a = tmem_base + C::A_BASE + cst * C::A_COLS;
                        // descriptor of the token tile; each 16-wide K slice starts 32 bytes
                        // further, i.e. 2 in the descriptor's address field
                        const uint64_t bdesc = sw128_desc(smem_addr(raw + stage * C::RAW_BYTES + hh * C::X_HALF));
#pragma unroll
                        for (int kk = 0; kk < W8_BK / 16; ++kk) {
                            // K slice kk goes to chain kk % NCHAIN; each chain starts from zero
                            const int j = kk % C::NCHAIN;
                            const uint32_t accum = (kb == 0 && hh == 0 && kk < C::NCHAIN) ? 0u : 1u;
                            const uint32_t dj = d + j * C::ACC1;
                            // K = 16 bf16 per instruction: 8 TMEM columns of A, 32 bytes of the B row
                            mma_bf16_ta(dj, a + kk * 8, bdesc + 2 * kk, idesc, accum);
                            if (DUAL) mma_bf16_ta(dj + BN, a + W8_BK / 2 + kk * 8, bdesc + 2 * kk, idesc, accum);
                        }
                        mma_commit(smem_addr(&cempty[cst]));
                        if (++cst == C::CSTAGES) { cst = 0; cph ^= 1; }
                    }
                    if (!ok) break;
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
    } else if (warp < 6) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int it = 0;
        for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const TileCoord c = tile_coord(p, t);
            const int acc = it % C::NACC;
            const uint32_t acc_phase = (it / C::NACC) & 1;
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&acc_full[acc]), acc_phase, abort_flag));
            if (!ok) { if (lane == 0) fail(); break; }
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
            const int64_t f = (int64_t)c.mt * W8_BM + row;            // weight row = output feature
            const int grp = p.groups > 1 ? c.sp / p.ks.sub : 0;       // the shard this split lies in
            float sc = 0.0f, sc2 = 0.0f;
            if (f < p.M) {
                sc = p.scale[f * p.groups + grp];
                if (DUAL) sc2 = p.scale2[f * p.groups + grp];
            }
            constexpr int CH = BN >= 32 ? 32 : 16;
            float v[32], u[32], t2[32];
            auto ld = [&](uint32_t addr, float (&dst)[32]) {
                if (CH == 32) tmem_ld32(addr, dst); else tmem_ld16(addr, dst);
            };
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += CH) {
                // the chains' sums, added in chain order
                ld(tbase + c0, v);
#pragma unroll 1
                for (int j = 1; j < C::NCHAIN; ++j) {
                    ld(tbase + j * C::ACC1 + c0, t2);
#pragma unroll
                    for (int e = 0; e < CH; ++e) v[e] += t2[e];
                }
                if (DUAL) {
                    ld(tbase + BN + c0, u);
#pragma unroll 1
                    for (int j = 1; j < C::NCHAIN; ++j) {
                        ld(tbase + j * C::ACC1 + BN + c0, t2);
#pragma unroll
                        for (int e = 0; e < CH; ++e) u[e] += t2[e];
                    }
                }
                if (f < p.M) {
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const int64_t tok = (int64_t)c.nt * BN + c0 + j;
                        if (tok < p.NB) {
                            if (DUAL) store_pair(p.epi, c.sp, tok, f, v[j] * sc, u[j] * sc2);
                            else store_value(p.epi, c.sp, tok, f, v[j] * sc);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&acc_empty[acc]));
        }
    } else {
        // ---------------------------------------------------------- converters
        const int q = warp & 3;                 // TMEM lane quarter this warp may write
        const int kq = (warp - 6) >> 2;         // which 32 of a half's 64 K elements
        const int r = q * 32 + lane;            // weight row within the tile = TMEM lane
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + C::A_BASE + kq * 16;
        int stage = 0, cst = 0;
        uint32_t phase = 0, cph = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            const TileCoord c = tile_coord(p, t);
            int64_t k0;
            int nkb;
            split_range(p, c.sp, k0, nkb);
            for (int kb = 0; kb < nkb && ok; kb += 2) {
                const int halves = min(2, nkb - kb);
                if (!__all_sync(0xFFFFFFFFu, fast_wait(smem_addr(&full[stage]), phase, abort_flag))) {
                    ok = false;
                    break;
                }
                const uint8_t* src = raw + stage * C::RAW_BYTES + C::X_BYTES + r * W8_RK;
                for (int hh = 0; hh < halves; ++hh) {
                    uint32_t wa[16], wb[16];
                    widen(src, r, hh, kq, wa);
                    if (DUAL) widen(src + C::Q_BYTES, r, hh, kq, wb);
                    if (!__all_sync(0xFFFFFFFFu, fast_wait(smem_addr(&cempty[cst]), cph ^ 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dst = lane_base + cst * C::A_COLS;
                    tmem_st16(dst, wa);
                    if (DUAL) tmem_st16(dst + W8_BK / 2, wb);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&cfull[cst]));
                    if (++cst == C::CSTAGES) { cst = 0; cph ^= 1; }
                }
                if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok && lane == 0) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, W8_TMEM_COLS);
    }
}

// One warp per (row, group): the group's amax, s = amax / 127, then the codes.
__global__ void __launch_bounds__(256)
quantize_w8_kernel(const __nv_bfloat16* __restrict__ W, int64_t rows, int64_t cols, int groups, int8_t* Q,
                   float* scale) {
    const int64_t gid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gid >= rows * groups) return;
    const int64_t r = gid / groups;
    const int g = (int)(gid - r * groups);
    const int64_t gw = cols / groups;
    const __nv_bfloat16* src = W + r * cols + g * gw;
    int8_t* dst = Q + r * cols + g * gw;
    float amax = 0.0f;
    for (int64_t i = (int64_t)lane * 8; i < gw; i += 256) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + i);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&w);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(__bfloat162float(e[j])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 127.0f);
    for (int64_t i = (int64_t)lane * 8; i < gw; i += 256) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + i);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&w);
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int qv = 0;
            if (s > 0.0f) qv = max(-127, min(127, __float2int_rn(__fdiv_rn(__bfloat162float(e[j]), s))));
            packed[j >> 2] |= (uint32_t)(qv & 0xFF) << (8 * (j & 3));
        }
        *reinterpret_cast<uint2*>(dst + i) = make_uint2(packed[0], packed[1]);
    }
    if (lane == 0) scale[gid] = s;
}

// ------------------------------------------------ CUDA-core int8 row-dot
// For one or two tokens the tensor-core kernel above is the wrong tool: its
// MMA warp issues eight MMAs plus barrier checks per 64-wide K half, which
// holds it near the bf16 weight rate, so int8 gains little there.  This kernel streams the
// codes with 16-byte loads, widens them with the same exact trick and does
// fp32 FMAs: about three instructions per weight and token.  Measured on the
// Llama-3.1-70B-shaped MLP: 181 us at one token against 229 us for bf16; at
// four tokens its FMAs and registers make it slower than the tensor cores.
//
// Each warp owns RW output features (rows of Q; with DUAL the same rows of Q
// and Q2) over one K split; lanes stride over K in 16-weight vectors, U vectors
// per lane in flight per row; the warp's sums are reduced with shuffles,
// scaled, and stored by distinct lanes.
constexpr int W8R_WARPS = 8;

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 16 int8 codes -> 16 exact floats (see widen).
__device__ __forceinline__ void codes_to_f32(const uint4& v, float (&f)[16]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t b = w[i] ^ 0x80808080u;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            f[4 * i + e] = __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7540 + e)) - 8388736.0f;
    }
}

struct W8RowdotArgs {
    const int8_t* Q; const int8_t* Q2;
    const float* scale; const float* scale2;
    int groups;
    int64_t M, K;
    const __nv_bfloat16* X; int64_t ldx; int nb;
    KSplit ks;
    Epilogue epi;
};

template <int NB, int RW, bool DUAL>
__global__ void __launch_bounds__(W8R_WARPS * 32) w8_rowdot_kernel(const W8RowdotArgs a) {
    constexpr int R = DUAL ? 2 * RW : RW;
    constexpr int U = 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t f0 = ((int64_t)blockIdx.x * W8R_WARPS + warp) * RW;
    if (f0 >= a.M) return;
    const int split = blockIdx.y;
    const int sh = split / a.ks.sub, j = split - sh * a.ks.sub;
    const int64_t kbeg = sh * a.ks.k_shard + (int64_t)j * a.ks.k_chunk;
    const int64_t kend = min(kbeg + a.ks.k_chunk, (int64_t)(sh + 1) * a.ks.k_shard);

    const int8_t* wp[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = min(f0 + (r % RW), a.M - 1);
        wp[r] = ((DUAL && r >= RW) ? a.Q2 : a.Q) + row * a.K;
    }
    float acc[R][NB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;

    for (int64_t k = kbeg + lane * 16; k < kend; k += 32 * 16 * U) {
        uint4 wv[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t kk = k + u * 32 * 16;
#pragma unroll
            for (int r = 0; r < R; ++r) wv[u][r] = kk < kend ? ld_stream16(wp[r] + kk) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t kk = k + u * 32 * 16;
            if (kk >= kend) break;
            float xf[NB][16];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < a.nb) {
                    const __nv_bfloat16* xp = a.X + (int64_t)b * a.ldx + kk;
                    const uint4 lo = __ldg(reinterpret_cast<const uint4*>(xp));
                    const uint4 hi = __ldg(reinterpret_cast<const uint4*>(xp + 8));
                    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xf[b][2 * i] = __uint_as_float(w[i] << 16);
                        xf[b][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) xf[b][e] = 0.f;
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float wf[16];
                codes_to_f32(wv[u][r], wf);
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[r][b] = fmaf(wf[e], xf[b][e], acc[r][b]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[r][b] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][b], o);
        }
    const int grp = a.groups > 1 ? sh : 0;
#pragma unroll
    for (int r = 0; r < RW; ++r) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int idx = r * NB + b;
            const int64_t f = f0 + r;
            if (lane == (idx & 31) && b < a.nb && f < a.M) {
                const float sc = a.scale[f * a.groups + grp];
                if (DUAL)
                    store_pair(a.epi, split, b, f, acc[r][b] * sc, acc[r + RW][b] * a.scale2[f * a.groups + grp]);
                else
                    store_value(a.epi, split, b, f, acc[r][b] * sc);
            }
        }
    }
}

template <bool DUAL>
cudaError_t launch_w8_rowdot_t(const W8RowdotArgs& a, cudaStream_t st) {
    constexpr int RW = DUAL ? 2 : 4;
    dim3 grid((unsigned)((a.M + W8R_WARPS * RW - 1) / (W8R_WARPS * RW)), (unsigned)(a.ks.tp * a.ks.sub));
    dim3 block(W8R_WARPS * 32);
    if (a.nb <= 1) w8_rowdot_kernel<1, RW, DUAL><<<grid, block, 0, st>>>(a);
    else w8_rowdot_kernel<2, RW, DUAL><<<grid, block, 0, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// int8 [rows, cols] (row pitch ld bytes), box 128 bytes x 128 rows, 128-byte
// swizzle; cached.
struct U8Key {
    const void* base; int64_t rows, cols, ld;
    bool operator==(const U8Key& o) const { return base == o.base && rows == o.rows && cols == o.cols && ld == o.ld; }
};
struct U8KeyHash {
    size_t operator()(const U8Key& k) const {
        return std::hash<const void*>()(k.base) ^ std::hash<int64_t>()(k.rows * 1000003 + k.cols * 31 + k.ld);
    }
};
bool u8_map(CUtensorMap* out, const void* base, int64_t rows, int64_t cols, int64_t ld) {
    static std::mutex mu;
    static std::unordered_map<U8Key, CUtensorMap, U8KeyHash> cache;
    const U8Key key{base, rows, cols, ld};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) { *out = it->second; return true; }
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)W8_RK, (cuuint32_t)W8_BM};
    cuuint32_t estr[2] = {1, 1};
    if (enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, *out);
    return true;
}

template <int BN, bool DUAL>
cudaError_t launch_cfg(const W8GemmArgs& a, cudaStream_t st) {
    using C = W8Cfg<BN, DUAL>;
    const DeviceCtx* ctx = device_ctx();
    if (!ctx) return cudaErrorNoDevice;
    static bool attr_set[64] = {};
    if (ctx->device < 64 && !attr_set[ctx->device]) {
        const cudaError_t e = cudaFuncSetAttribute(w8_gemm_kernel<BN, DUAL>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[ctx->device] = true;
    }
    CUtensorMap mQ, mQ2, mX;
    if (!u8_map(&mQ, a.Q, a.M, a.K, a.K)) return cudaErrorInvalidValue;
    mQ2 = mQ;
    if (DUAL && !u8_map(&mQ2, a.Q2, a.M, a.K, a.K)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(&mX, a.X, a.N, a.K, a.ldx, BN)) return cudaErrorInvalidValue;
    W8Params p{};
    p.M = a.M;
    p.NB = a.N;
    p.m_tiles = (int)((a.M + W8_BM - 1) / W8_BM);
    p.n_tiles = (int)((a.N + BN - 1) / BN);
    p.splits = a.ks.tp * a.ks.sub;
    p.total_tiles = (int64_t)p.m_tiles * p.n_tiles * p.splits;
    p.ks = a.ks;
    p.epi = a.epi;
    p.scale = a.scale;
    p.scale2 = a.scale2;
    p.groups = a.groups;
    p.err = ctx->err_word;
    const int64_t grid = std::min<int64_t>(p.total_tiles, ctx->num_sms);
    w8_gemm_kernel<BN, DUAL><<<(unsigned)grid, W8_THREADS, C::SMEM_BYTES, st>>>(mQ, mQ2, mX, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_w8_gemm(const W8GemmArgs& a, cudaStream_t st) {
    const bool dual = a.epi.mode == EPI_SWIGLU || a.epi.mode == EPI_PARTIAL2;
    if (a.N <= 16) return dual ? launch_cfg<16, true>(a, st) : launch_cfg<16, false>(a, st);
    if (a.N <= 32) return dual ? launch_cfg<32, true>(a, st) : launch_cfg<32, false>(a, st);
    if (a.N <= 64) return dual ? launch_cfg<64, true>(a, st) : launch_cfg<64, false>(a, st);
    return dual ? launch_cfg<128, true>(a, st) : launch_cfg<128, false>(a, st);
}

cudaError_t launch_w8_rowdot(const W8GemmArgs& g, cudaStream_t st) {
    if (g.N > kW8RowdotMaxTokens) return cudaErrorInvalidValue;
    W8RowdotArgs a{};
    a.Q = g.Q; a.Q2 = g.Q2; a.scale = g.scale; a.scale2 = g.scale2; a.groups = g.groups;
    a.M = g.M; a.K = g.K;
    a.X = static_cast<const __nv_bfloat16*>(g.X); a.ldx = g.ldx; a.nb = (int)g.N;
    a.ks = g.ks;
    a.epi = g.epi;
    const bool dual = g.epi.mode == EPI_SWIGLU || g.epi.mode == EPI_PARTIAL2;
    return dual ? launch_w8_rowdot_t<true>(a, st) : launch_w8_rowdot_t<false>(a, st);
}

cudaError_t launch_quantize_w8(const void* W, int64_t rows, int64_t cols, int groups, int8_t* Q, float* scale,
                               cudaStream_t st) {
    const int64_t warps = rows * groups;
    const int64_t blocks = (warps + 7) / 8;
    quantize_w8_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(W), rows, cols, groups,
                                                         Q, scale);
    return cudaGetLastError();
}

}  // namespace tpl
