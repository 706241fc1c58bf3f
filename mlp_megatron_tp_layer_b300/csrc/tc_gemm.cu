// Tensor-core GEMM for sm_103a: TMA loads into 128B-swizzled shared memory,
// tcgen05.mma (kind::f16, bf16 in, fp32 accumulate) issued by one thread into
// a double-buffered TMEM accumulator, tcgen05.ld epilogue.  Persistent: one
// CTA per SM walks a static tile list, so the load pipeline keeps streaming
// across tile boundaries and the epilogue of tile i overlaps the MMAs of i+1.
//
//   D[M, N] = A[M, K] . B[N, K]^T     (both operands K-major, bf16)
//
// Normal orientation: A = activations (M = tokens), B = [out, in] weights.
// Swapped orientation (decode, few tokens): A = weights (M = features, 128 per
// tile), B = tokens (N = 16..128), so weights stream as the M=128 operand.
// DUAL (SwiGLU): normal -> the B tile is [128 gate rows; 128 up rows] and one
// N=256 MMA produces both; swapped -> two A tiles (gate, up) and two MMAs into
// adjacent TMEM column ranges.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA
// issuer, warps 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA sets
// the sticky device error word, drains what it started, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tpl {
namespace {

constexpr int BM = 128;             // rows of A per tile (TMEM lanes)
constexpr int BK = 64;              // K elements per stage (128 bytes of bf16: one swizzle row)
constexpr int kThreads = 192;

struct TcParams {
    int64_t M;            // valid rows of A (tokens, or features when swapped)
    int64_t NB;           // valid rows of each B operand (features, hidden units, or tokens)
    int m_tiles, n_tiles, splits;
    int64_t total_tiles;
    KSplit ks;
    Epilogue epi;
    unsigned int* err;
    // split last wave: tiles [main_tiles, total_tiles) are cut into tail_s
    // K-chunks each; CTA b < tail tiles x tail_s computes chunk b % tail_s of
    // tail tile b / tail_s after its whole tiles and writes an fp32 partial
    // (column-major [OUT_COLS][BM]) to slot b of tail_ws
    int64_t main_tiles;
    int tail_s;
    float* tail_ws;
    // normal orientation with few m-tiles: A (tokens, reused by every n-tile)
    // is loaded evict_last and B (weights, read by the few CTAs of one wave)
    // evict_first, so the streamed weights do not push A out of L2
    int hint_ab;
};

template <int BN, bool SWAP, bool DUAL>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;                          // 16 KB
    static constexpr int A2_BYTES = (SWAP && DUAL) ? A_BYTES : 0;
    static constexpr int B_BYTES = BN * BK * 2;                          // includes gate+up when normal DUAL
    static constexpr int STAGE_BYTES = A_BYTES + A2_BYTES + B_BYTES;
    static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 10 ? 10 : STAGES_RAW;
    static constexpr int B_ROWS = (!SWAP && DUAL) ? BN / 2 : BN;         // rows per B TMA box
    static constexpr int ACC_COLS = (SWAP && DUAL) ? 2 * BN : BN;        // TMEM columns per accumulator
    static constexpr int TMEM_COLS = (2 * ACC_COLS <= 32) ? 32 : (2 * ACC_COLS <= 64) ? 64
                                   : (2 * ACC_COLS <= 128) ? 128 : (2 * ACC_COLS <= 256) ? 256 : 512;
    static constexpr int OUT_COLS = (!SWAP && DUAL) ? BN / 2 : BN;       // output columns per tile
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
    static_assert(2 * ACC_COLS <= 512, "TMEM holds 512 fp32 columns");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "M=128 MMA needs N in 16..256 step 16");
};

struct TileCoord { int sp, mt, nt; };
__device__ __forceinline__ TileCoord tile_coord(const TcParams& p, int64_t t) {
    const int64_t per_split = (int64_t)p.m_tiles * p.n_tiles;
    TileCoord c;
    c.sp = (int)(t / per_split);
    const int64_t r = t - (int64_t)c.sp * per_split;
    c.mt = (int)(r % p.m_tiles);      // m fastest: concurrent CTAs share the B (weight) tile
    c.nt = (int)(r / p.m_tiles);
    return c;
}
__device__ __forceinline__ void split_range(const TcParams& p, int sp, int64_t& k0, int& nkb) {
    const int sh = sp / p.ks.sub, j = sp - sh * p.ks.sub;
    k0 = sh * p.ks.k_shard + (int64_t)j * p.ks.k_chunk;
    const int64_t k1 = min(k0 + p.ks.k_chunk, (int64_t)(sh + 1) * p.ks.k_shard);
    nkb = (int)((k1 - k0 + BK - 1) / BK);
}

// Work item `it` of this CTA: its whole tiles (blockIdx.x, + gridDim.x, ...)
// below main_tiles, then at most one K-chunk of a tail tile.  slot < 0: a
// whole tile; else the chunk's partial slot.
struct Item { TileCoord c; int64_t k0; int nkb; int slot; };
__device__ __forceinline__ bool item_of(const TcParams& p, int it, Item& w) {
    const int b = blockIdx.x;
    const int64_t n_main = p.main_tiles > b ? (p.main_tiles - 1 - b) / gridDim.x + 1 : 0;
    if (it < n_main) {
        w.c = tile_coord(p, b + (int64_t)it * gridDim.x);
        split_range(p, w.c.sp, w.k0, w.nkb);
        w.slot = -1;
        return true;
    }
    if (it > n_main || p.tail_s == 0 || b >= (p.total_tiles - p.main_tiles) * p.tail_s) return false;
    const int i = b / p.tail_s, j = b - i * p.tail_s;
    w.c = tile_coord(p, p.main_tiles + i);
    int64_t k0;
    int nkb;
    split_range(p, w.c.sp, k0, nkb);
    const int kb0 = (int)((int64_t)nkb * j / p.tail_s), kb1 = (int)((int64_t)nkb * (j + 1) / p.tail_s);
    w.k0 = k0 + (int64_t)kb0 * BK;
    w.nkb = kb1 - kb0;
    w.slot = b;
    return true;
}

template <int BN, bool SWAP, bool DUAL>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
               const TcParams p) {
    using C = Cfg<BN, SWAP, DUAL>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* acc_full = bars + 2 * C::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // zero the row accumulators of the reduction that will consume this output
    if (p.epi.zero_words && blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.epi.zero_count; i += blockDim.x) p.epi.zero_words[i] = 0u;

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
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (DUAL) { if (SWAP) prefetch_tmap(&tmA2); else prefetch_tmap(&tmB2); }
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        if (p.err) atomicOr(p.err, TPL_DEVERR_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int issued_tail = 0;   // stages loaded but not yet known to be consumed (abort drain)
            bool ok = true;
            Item w;
            for (int it = 0; ok && item_of(p, it, w); ++it) {
                const TileCoord c = w.c;
                const int64_t k0 = w.k0;
                const int nkb = w.nkb;
                const int am = c.mt * BM;
                const int bn = c.nt * C::B_ROWS;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(smem_addr(&empty[stage]), phase ^ 1, abort_flag)) { ok = false; break; }
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_expect_tx(fb, C::STAGE_BYTES);
                    uint8_t* st = smem + stage * C::STAGE_BYTES;
                    const int kx = (int)(k0 + kb * BK);
                    if (SWAP) {
                        tma_load_hint(smem_addr(st), &tmA, fb, kx, am, pol_w);
                        if (DUAL) tma_load_hint(smem_addr(st + C::A_BYTES), &tmA2, fb, kx, am, pol_w);
                        tma_load_hint(smem_addr(st + C::A_BYTES + C::A2_BYTES), &tmB, fb, kx, bn, pol_x);
                    } else if (p.hint_ab) {
                        tma_load_hint(smem_addr(st), &tmA, fb, kx, am, pol_x);
                        tma_load_hint(smem_addr(st + C::A_BYTES), &tmB, fb, kx, bn, pol_w);
                        if (DUAL) tma_load_hint(smem_addr(st + C::A_BYTES + C::B_BYTES / 2), &tmB2, fb, kx, bn, pol_w);
                    } else {
                        tma_load(smem_addr(st), &tmA, fb, kx, am);
                        tma_load(smem_addr(st + C::A_BYTES), &tmB, fb, kx, bn);
                        if (DUAL) tma_load(smem_addr(st + C::A_BYTES + C::B_BYTES / 2), &tmB2, fb, kx, bn);
                    }
                    issued_tail = min(issued_tail + 1, C::STAGES);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                fail();
                // Let the copies already issued land before the CTA exits: wait
                // (bounded) on the full barrier of each in-flight stage.
                for (int i = 0; i < issued_tail; ++i) {
                    if (--stage < 0) { stage = C::STAGES - 1; phase ^= 1; }
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_addr(&full[stage]), phase) && globaltimer() - t0 < kWaitLimitNs) {}
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(BM, (SWAP || !DUAL) ? BN : BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            Item w;
            for (int it = 0; ok && item_of(p, it, w); ++it) {
                const int nkb = w.nkb;
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(smem_addr(&acc_empty[acc]), acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * C::ACC_COLS;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(smem_addr(&full[stage]), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + C::A_BYTES + C::A2_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t accum = (kb | kk) ? 1u : 0u;
                        mma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), idesc, accum);
                        if (SWAP && DUAL)
                            mma_bf16(d + BN, sw128_desc(sa + C::A_BYTES + kk * 32), sw128_desc(sb + kk * 32),
                                     idesc, accum);
                    }
                    mma_commit(smem_addr(&empty[stage]));
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_addr(&acc_full[acc]));
            }
            if (!ok) fail();
            // Wait (bounded) until every MMA issued above has completed, so TMEM
            // can be released safely.
            mma_commit(smem_addr(drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_addr(drain), 0) && globaltimer() - t0 < kWaitLimitNs) {}
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        Item w;
        for (int it = 0; item_of(p, it, w); ++it) {
            const TileCoord c = w.c;
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // every lane polls; the vote keeps the warp converged for the
            // .sync.aligned TMEM loads even when a wait gives up
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&acc_full[acc]), acc_phase, abort_flag));
            if (!ok) { if (lane == 0) fail(); break; }
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
            const int64_t a_row = (int64_t)c.mt * BM + row;         // token (normal) or feature (swapped)
            constexpr int CH = C::OUT_COLS >= 32 ? 32 : 16;
            float v[32], u[32];
#pragma unroll 1
            for (int c0 = 0; c0 < C::OUT_COLS; c0 += CH) {
                if (CH == 32) tmem_ld32(tbase + c0, v); else tmem_ld16(tbase + c0, v);
                if (DUAL) {
                    const int up_off = SWAP ? BN : BN / 2;
                    if (CH == 32) tmem_ld32(tbase + up_off + c0, u); else tmem_ld16(tbase + up_off + c0, u);
                }
                if (w.slot >= 0) {
                    // tail chunk: the whole fp32 tile, column-major (lanes = rows: coalesced)
                    float* dst = p.tail_ws + (size_t)w.slot * C::OUT_COLS * BM + row;
#pragma unroll
                    for (int j = 0; j < CH; ++j) dst[(size_t)(c0 + j) * BM] = v[j];
                } else if (a_row < p.M) {
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const int64_t b_row = (int64_t)c.nt * C::OUT_COLS + c0 + j;
                        if (b_row < p.NB) {
                            const int64_t tok = SWAP ? b_row : a_row;
                            const int64_t feat = SWAP ? a_row : b_row;
                            if (DUAL) store_pair(p.epi, c.sp, tok, feat, v[j], u[j]);
                            else store_value(p.epi, c.sp, tok, feat, v[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&acc_empty[acc]));
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

// Tail tiles of a split last wave: element (row, col) of tail tile i is the
// sum of its tail_s chunk partials in ascending k order (a fixed order), then
// stored through the launch's epilogue.  Column-major within a tile, so the
// threads of a warp read consecutive rows.
template <int OUT_COLS>
__global__ void __launch_bounds__(256) tail_reduce_kernel(const TcParams p) {
    const int64_t per = (int64_t)OUT_COLS * BM;
    const int64_t n = (p.total_tiles - p.main_tiles) * per;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n; g += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(g / per);
        const int64_t e = g - (int64_t)i * per;
        const int col = (int)(e / BM), row = (int)(e - (int64_t)col * BM);
        const float* src = p.tail_ws + (size_t)i * p.tail_s * per + e;
        float v = 0.f;
#pragma unroll 8
        for (int j = 0; j < p.tail_s; ++j) v += __ldcs(src + (size_t)j * per);
        const TileCoord c = tile_coord(p, p.main_tiles + i);
        const int64_t tok = (int64_t)c.mt * BM + row, feat = (int64_t)c.nt * OUT_COLS + col;
        if (tok < p.M && feat < p.NB) store_value(p.epi, 0, tok, feat, v);
    }
}

// Split of the last wave (see TcParams): tail tiles and chunks per tile, for
// a plain-store GEMM of M x N output with N-tiles of 256 and K-depth K.
struct TailPlan { int64_t tail_tiles; int s; size_t bytes; };
TailPlan tail_plan(int64_t M, int64_t N, int64_t K, int sms) {
    TailPlan t{0, 0, 0};
    const int64_t total = ((M + BM - 1) / BM) * ((N + 255) / 256);
    const int64_t nkb = (K + BK - 1) / BK;
    if (sms <= 0 || total <= sms || total >= 8LL * sms) return t;   // one partial wave, or a negligible tail
    const int64_t tail = total % sms;
    if (tail == 0) return t;
    const int64_t s = std::min<int64_t>(sms / tail, nkb);
    if (s < 2) return t;
    t.tail_tiles = tail;
    t.s = (int)s;
    t.bytes = (size_t)tail * s * 256 * BM * 4;
    return t;
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

// 2-D bf16 tensor [rows, cols] with row pitch ld (elements); box = 64 x box_rows.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor maps are pure functions of (pointer, shape, box); cache them so a
// decode step does not re-encode the same weights on every call.
struct MapKey {
    const void* base; int64_t rows, cols, ld; int box;
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && cols == o.cols && ld == o.ld && box == o.box;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.base);
        h ^= std::hash<int64_t>()(k.rows * 1000003 + k.cols * 31 + k.ld * 7 + k.box) + 0x9e3779b97f4a7c15ull + (h << 6);
        return h;
    }
};
bool cached_map(CUtensorMap* out, const void* base, int64_t rows, int64_t cols, int64_t ld, int box) {
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    MapKey k{base, rows, cols, ld, box};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(k);
    if (it != cache.end()) { *out = it->second; return true; }
    if (!make_map(out, base, rows, cols, ld, box)) return false;
    if (cache.size() > 4096) cache.clear();
    cache.emplace(k, *out);
    return true;
}

template <int BN, bool SWAP, bool DUAL>
cudaError_t launch_cfg(const TcGemmArgs& a, cudaStream_t st) {
    using C = Cfg<BN, SWAP, DUAL>;
    const DeviceCtx* ctx = device_ctx();
    if (!ctx) return cudaErrorNoDevice;
    static bool attr_set[64] = {};
    const int dev = ctx->device;
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, SWAP, DUAL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    CUtensorMap mA, mA2, mB, mB2;
    const int a_box = BM;
    const int b_box = C::B_ROWS;
    if (!cached_map(&mA, a.A, a.M, a.K, a.lda, a_box)) return cudaErrorInvalidValue;
    if (!cached_map(&mB, a.B, a.N, a.K, a.ldb, b_box)) return cudaErrorInvalidValue;
    mA2 = mA;
    mB2 = mB;
    if (DUAL && SWAP && !cached_map(&mA2, a.A2, a.M, a.K, a.lda, a_box)) return cudaErrorInvalidValue;
    if (DUAL && !SWAP && !cached_map(&mB2, a.B2, a.N, a.K, a.ldb, b_box)) return cudaErrorInvalidValue;

    TcParams p;
    p.M = a.M;
    p.NB = a.N;
    p.m_tiles = (int)((a.M + BM - 1) / BM);
    p.n_tiles = (int)((a.N + C::OUT_COLS - 1) / C::OUT_COLS);
    p.splits = a.ks.tp * a.ks.sub;
    p.total_tiles = (int64_t)p.m_tiles * p.n_tiles * p.splits;
    p.ks = a.ks;
    p.epi = a.epi;
    p.err = ctx->err_word;
    p.main_tiles = p.total_tiles;
    p.tail_s = 0;
    p.tail_ws = nullptr;
    // (measured: the sharded-matmul cases, 4 m-tiles, 834-839 -> 864-866 TFLOP/s;
    // the 4096-token prefill, 32 m-tiles, is slower with it: its weights are
    // read by 32 CTAs and evict_first loses them between readers)
    p.hint_ab = (!SWAP && p.m_tiles <= 8) ? 1 : 0;
    if (!SWAP && !DUAL && C::OUT_COLS == 256 && a.epi.mode == EPI_STORE && p.splits == 1 && a.tail_ws) {
        const TailPlan t = tail_plan(a.M, a.N, a.K, ctx->num_sms);
        if (t.s > 0 && t.bytes <= a.tail_ws_bytes) {
            p.main_tiles = p.total_tiles - t.tail_tiles;
            p.tail_s = t.s;
            p.tail_ws = a.tail_ws;
        }
    }
    const int64_t grid = std::min<int64_t>(p.total_tiles, ctx->num_sms);
    tc_gemm_kernel<BN, SWAP, DUAL><<<(unsigned)grid, kThreads, C::SMEM_BYTES, st>>>(mA, mA2, mB, mB2, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.tail_s == 0) return e;
    const int64_t n = (p.total_tiles - p.main_tiles) * C::OUT_COLS * BM;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)ctx->num_sms * 8);
    tail_reduce_kernel<C::OUT_COLS><<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t tc_tail_ws_bytes(int64_t M, int64_t N, int64_t K, int sms) { return tail_plan(M, N, K, sms).bytes; }

bool tma_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    return cached_map(m, base, rows, cols, ld, box_rows);
}

bool tc_gemm_supported() {
    const DeviceCtx* ctx = device_ctx();
    if (!ctx) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, ctx->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
    return major == 10 && minor == 3 && get_encoder() != nullptr;
}

cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st) {
    const bool dual = a.epi.mode == EPI_SWIGLU || a.epi.mode == EPI_PARTIAL2;
    if (!a.swap) {
        return dual ? launch_cfg<256, false, true>(a, st) : launch_cfg<256, false, false>(a, st);
    }
    // swapped: tile N covers the tokens
    if (a.N <= 16) return dual ? launch_cfg<16, true, true>(a, st) : launch_cfg<16, true, false>(a, st);
    if (a.N <= 32) return dual ? launch_cfg<32, true, true>(a, st) : launch_cfg<32, true, false>(a, st);
    if (a.N <= 64) return dual ? launch_cfg<64, true, true>(a, st) : launch_cfg<64, true, false>(a, st);
    return dual ? launch_cfg<128, true, true>(a, st) : launch_cfg<128, true, false>(a, st);
}

}  // namespace tpl
