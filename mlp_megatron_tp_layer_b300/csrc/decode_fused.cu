// Fused decode stack: ONE persistent launch runs every layer of a serial
// pre-norm decoder stack (h = x + Attn(RMSNorm(x)); y = h + MLP(RMSNorm(h)))
// for a small batch of tokens (B <= 128), with the tensor-parallel shards as
// logical weight partitions.
//
// Each layer is four projections, each a "phase" of the launch:
//   QKV    [n_qkv, D] . RMSNorm(x)      -> packed QKV (shard blocks) and the
//                                          context-1 attention output O
//   OPROJ  [D, n_q hd] . O  (row-par.)  -> h = x + sum over shards
//   GATEUP [F, D] x2 . RMSNorm(h)       -> H = silu(gate) * up
//   DOWN   [D, F] . H       (row-par.)  -> y = h + sum over shards
// Weights are the M = 128 operand of tcgen05.mma (kind::f16), tokens the N
// operand (padded to NP by TMA's zero fill), accumulators in TMEM.
//
// Work split: a phase's work is the flattened list of (m-tile, 64-wide
// k-block) pairs; CTA c of g takes the contiguous range [c T/g, (c+1) T/g),
// with g = m_tiles x s (every tile exactly s segments) when that still uses
// at least 94% of the G CTAs, else g = G.
// A range may cover parts of several m-tiles ("units"); each unit leaves an
// fp32 partial tile in global memory.  In the 32- to 128-column
// instantiations it then counts itself on the tile's ticket (a release
// increment), and a finalizing CTA waits for the count before it loads the
// partials.  In the 16-column one (up to 16 tokens, where a phase is short
// and that fence and ticket round trip are a large part of it) each partial
// value is stored with a 32-bit tag (layer + 1) in one 8-byte word, which a
// reader sees whole or not at all: the finalizer polls the words themselves
// until every one carries this layer's tag, with no fence or counter in
// between.  Once all of a tile's units have arrived, the CTAs that hold them
// each finalize a share of the tile's tokens: they add the tile's partials in
// k order (the order of the shards for the row-parallel phases) and apply the
// phase's epilogue.  The sum is therefore the same whatever order the CTAs
// ran in, and the same in both exchanges.
//
// There is no grid-wide barrier between phases.  Each output tile of a phase
// has a ready counter (tokens finalized, monotone over the layers of the
// launch); a unit's activation loads wait only for the tiles of the previous
// phase that its k-blocks read, so a phase starts wherever its inputs are
// final.  Each phase also has a done counter (tokens finalized over all its
// tiles), and a phase finalizes no tile before the previous finalizing phase
// is done.  By induction every earlier phase is then complete, which is what
// makes it safe to overwrite the buffers the layers share: a phase's partial
// slots (one region per projection kind), its output tile, and the RMSNorm
// tile sums are rewritten only after every reader of the previous contents
// has finished.  The launch is cooperative, so every CTA is resident and these
// waits (all bounded in time) can be met.  Weight tiles do not depend on the
// activations, so the weight producer keeps loading the next phases' weights
// into the shared-memory ring while their inputs are pending.
//
// RMSNorm: the producer of a residual-stream value also writes, per 128-column
// tile and token, the sum of squares of the rounded values; the consumer's
// epilogue turns the tile sums into 1/rms and multiplies its fp32 products by
// it (RMSNorm(x) W^T = diag(1/rms(x)) x W^T).
//
// Warp roles (256 threads): 0 weight TMA producer, 1 TMEM owner + MMA issuer,
// 2..5 epilogue (warp w reads TMEM lanes 32 (w % 4) ..), 6 activation TMA
// producer, 7 phase watcher (polls the done counters ahead of the epilogue
// and posts, in shared memory, which phases may finalize).  Every wait is
// bounded in time; on expiry the CTA sets the grid abort flag and the sticky
// device error word, and every role winds down.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tpl {

// Phase trace (instrumented builds only, -DTPL_FUSED_TRACE): per CTA and
// phase of the last launch, %globaltimer stamps of kFusedTraceEvents events
// (see tpl_fused_trace_read).  In normal builds the stamps compile to nothing.
#ifdef TPL_FUSED_TRACE
constexpr int kFusedTracePhases = 1 + 4 * kFusedMaxLayers;
__device__ unsigned long long g_fused_trace[kFusedGridCap * kFusedTracePhases * kFusedTraceEvents];
#define TPL_TRACE(k, e) \
    (g_fused_trace[((size_t)cta * kFusedTracePhases + (k)) * kFusedTraceEvents + (e)] = globaltimer())
#else
#define TPL_TRACE(k, e) ((void)0)
#endif

namespace {

constexpr int kFThreads = 256;
constexpr int kSmemLimit = 227 * 1024;     // dynamic shared memory of one CTA
constexpr int kWarpW = 0, kWarpMma = 1, kWarpAct = 6, kWarpWatch = 7;
constexpr int kTmemCols = 512;     // two accumulators of up to 256 columns
// Instantiations up to this width exchange tagged partial words.  (At 32
// columns, twice the words per unit and the longer polls lost 5-10%.)
constexpr int kTaggedNP = 16;
constexpr int kAccStride = 256;
enum Kind { K_QKV = 0, K_OPROJ = 1, K_GATEUP = 2, K_DOWN = 3 };
enum ActMap { A_X = 0, A_R0 = 1, A_R1 = 2, A_QKV = 3, A_H = 4, A_HID = 5, A_COUNT = 6 };
enum WMap { W_QKV = 0, W_O = 1, W_G = 2, W_U = 3, W_D = 4, W_COUNT = 5 };

// Tensor maps travel as a __grid_constant__ kernel parameter (about 21 KB).
struct FusedMaps {
    CUtensorMap act[A_COUNT];                      // [B rows, cols] bf16, box NP x 64
    CUtensorMap w[kFusedMaxLayers][W_COUNT];       // [rows, K] bf16, box 128 x 64
};

struct FusedParams {
    int B, D, F, L, G;
    int parallel;              // 1: parallel block ([L4] S5.5), 0: serial pre-norm block
    int n_qkv, ko;             // packed QKV rows, o_proj input width n_q hd
    int max_mt;                // length of a ticket / ready row
    float eps;
    QkvMap qkv;                // packed-QKV layout (qkv_out = shard blocks [tp, B, w_s])
    const __nv_bfloat16* x_in;
    __nv_bfloat16 *y_out, *R0, *R1, *h, *H;
    float* slots_y;            // [ceil(D/128)][B] sums of squares of the layer input / output
    float* slots_h;            // [ceil(D/128)][B] sums of squares of h
    float* part;               // partial tiles, [4 kinds][G + max_mt][2][NP][128] fp32
    unsigned* tickets;         // [4][max_mt] units arrived per tile (monotone over the layers)
    unsigned* ready;           // [4][max_mt] tokens finalized per output tile (monotone)
    unsigned* done;            // [1 + 4 L] tokens finalized per phase (phase 0: input tile sums)
    int* gabort;               // grid abort flag (zero at launch)
    unsigned* err;
    uint64_t wait_ns;          // time limit of every wait between CTAs and roles
    int skip_cta, skip_phase;  // test hook: that CTA does not deliver its first unit of that phase (-1: off)
    int s_cap[4];              // most segments a tile of each projection kind is split into
};

template <int NP>
struct FCfg {
    static constexpr int W_BYTES = 128 * 64 * 2;                 // one 128 x 64 weight tile
    static constexpr int X_BYTES = NP * 64 * 2;                  // the NP x 64 activation tile
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int CTRL = 1024;                            // mbarriers and flags
    static constexpr int EPI = (2 * kFusedGridCap + 8) * 4;     // two segment lists and their counts
    static constexpr int FIN_ITEMS = NP == 32 ? 10 : 12;   // float4 rows (of 32 lanes) a finalizing warp stages
    static constexpr int FIN = 4 * FIN_ITEMS * 32 * 16;          // finalize staging, all epilogue warps
    static constexpr int STAGES_RAW = (kSmemLimit - 1024 - CTRL - EPI - FIN) / STAGE;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    static constexpr int SMEM = 1024 + STAGES * STAGE + CTRL + EPI + FIN;
    static constexpr int PART_FLOATS = 2 * NP * 128;             // one partial slot
    static constexpr int CH = NP >= 32 ? 32 : 16;                // TMEM columns per load
    static_assert(NP % 16 == 0 && NP >= 16 && NP <= 128, "N of an M=128 MMA: 16..256, step 16");
    static_assert(STAGE % 1024 == 0, "128B-swizzled tiles need 1024-byte alignment");
    static_assert(3 * STAGES + 5 <= 120, "mbarriers must fit the control block");
    static_assert(STAGES >= 4, "too few ring stages");
};

struct Phase {
    int kind, layer, m_tiles, nkb, M;
    int gw;                    // CTAs holding units of the phase: 0 .. gw-1
    int whole;                 // tiles 0 .. whole-1 go whole to CTAs 0 .. whole-1 (0: none)
    int rev;                   // 1: a CTA takes its units last tile first (see phase_of)
    int prev_fin;              // phase whose completion this phase's finalize waits for (-1: none)
    int src_kind;              // kind whose output tiles the activation loads wait for (-1: launch input)
    unsigned src_target;       // ready count of such a tile once this layer's input is final
    int total;                 // m_tiles x nkb (the shape check keeps total x G below 2^31)
    const CUtensorMap* wa;
    const CUtensorMap* wb;
    const CUtensorMap* act;
};

// Phase k >= 1 of the launch: layer (k-1)/4, projection (k-1)%4.  Serial
// block: QKV, o_proj, gate/up, down.  Parallel block: QKV and gate/up (both
// on RMSNorm(x)), then o_proj and down, whose partials are summed together
// into y by down's finalize (o_proj finalizes nothing of its own).
template <bool WH = false>
__device__ __forceinline__ Phase phase_of(const FusedMaps& mp, const FusedParams& p, int k) {
    Phase ph;
    ph.layer = (k - 1) >> 2;
    const int pos = (k - 1) & 3;
    const int l = ph.layer;
    const unsigned B = (unsigned)p.B;
    if (p.parallel) {
        constexpr int order[4] = {K_QKV, K_GATEUP, K_OPROJ, K_DOWN};
        ph.kind = order[pos];
        ph.prev_fin = ph.kind == K_OPROJ ? -1 : (ph.kind == K_DOWN ? k - 2 : k - 1);
    } else {
        ph.kind = pos;
        ph.prev_fin = k - 1;
    }
    // the layer input y(l-1) is tile-ready once down of layer l-1 finalized it
    const bool from_x = ph.kind == K_QKV || (p.parallel && ph.kind == K_GATEUP);
    int K, wa, wb = -1;
    switch (ph.kind) {
    case K_QKV:
        ph.M = p.n_qkv; K = p.D; wa = W_QKV;
        break;
    case K_OPROJ:
        ph.M = p.D; K = p.ko; wa = W_O; ph.act = &mp.act[A_QKV];
        ph.src_kind = K_QKV; ph.src_target = B * (unsigned)(l + 1);
        break;
    case K_GATEUP:
        ph.M = p.F; K = p.D; wa = W_G; wb = W_U;
        if (!p.parallel) { ph.act = &mp.act[A_H]; ph.src_kind = K_OPROJ; ph.src_target = B * (unsigned)(l + 1); }
        break;
    default:
        ph.M = p.D; K = p.F; wa = W_D; ph.act = &mp.act[A_HID];
        ph.src_kind = K_GATEUP; ph.src_target = B * (unsigned)(l + 1);
        break;
    }
    if (from_x) {
        ph.act = &mp.act[l == 0 ? A_X : (((l - 1) & 1) ? A_R1 : A_R0)];
        ph.src_kind = l == 0 ? -1 : K_DOWN;
        ph.src_target = B * (unsigned)l;
    }
    ph.wa = &mp.w[l][wa];
    ph.wb = wb < 0 ? nullptr : &mp.w[l][wb];
    ph.m_tiles = (ph.M + 127) / 128;
    ph.nkb = (K + 63) / 64;
    ph.total = ph.m_tiles * ph.nkb;
    // every tile split into exactly s segments when m_tiles x s CTAs still
    // cover at least 94% of the grid (fewer, aligned segments: less partial
    // traffic per tile; the CTAs left over stream no weights in this phase)
    ph.gw = p.G;
    // gate/up with at least one tile per CTA: CTA c first takes tile c whole
    // (its SwiGLU comes straight from TMEM, no partials), then its share of
    // the remaining tiles, split as below
    // (only the 128-column instantiation carries this path: it pays at 65-128
    // tokens, where the gate/up finalize is long)
    ph.whole = (WH && ph.kind == K_GATEUP && ph.m_tiles >= p.G) ? p.G : 0;
    // down after whole gate/up tiles: H tiles 0 .. G-1 are final long before
    // the split ones, so a CTA whose range starts among the split tiles' k-blocks
    // and runs into the next m-tile takes that next tile's unit first (units
    // are separate partials: their order changes no sum)
    ph.rev = (WH && ph.kind == K_DOWN && (p.F + 127) / 128 >= p.G) ? 1 : 0;
    if (ph.whole) return ph;
    const int s = min(p.G / ph.m_tiles, ph.nkb);
    if (s > p.s_cap[ph.kind]) ph.gw = ph.m_tiles * p.s_cap[ph.kind];
    else if (s >= 1 && ph.m_tiles * s * 100 >= p.G * 94) ph.gw = ph.m_tiles * s;
    return ph;
}

// Tokens a phase has finalized once it is complete (phase 0: the tile sums
// of squares of the launch input, B per 128-column tile).
__device__ __forceinline__ unsigned done_target(const FusedMaps& mp, const FusedParams& p, int k) {
    if (k == 0) return (unsigned)((p.D + 127) / 128) * (unsigned)p.B;
    return (unsigned)phase_of(mp, p, k).m_tiles * (unsigned)p.B;
}

// The output tile of phase ph.src_kind that k-block kb of ph's activations
// lies in.  o_proj's input O is the context-1 attention output: column block
// kb belongs to Q head h = 64 kb / hd, whose value is V of KV group
// g = h / (n_q / n_kv), i.e. packed-QKV rows (n_q + n_kv + g) hd + (64 kb mod hd)
// (a 64-wide block never straddles two heads: hd % 64 == 0).  Every other
// input is the previous phase's output read in place: 128-wide tile kb / 2.
__device__ __forceinline__ int src_tile(const FusedParams& p, const Phase& ph, int kb);

// Coordinates (x = column, y = first row) of k-block kb's activation tile.
// o_proj's input is the context-1 attention output O, whose column block kb
// (Q head h = 64 kb / hd) equals V of KV group g = h / (n_q / n_kv): it is
// read in place from the shard-blocked QKV output [tp B, w_s], at the V
// columns of the first shard holding group g (the TMA box's rows past that
// shard's B tokens are other shards' rows, or zero fill past the end: they
// only reach accumulator columns of padding tokens, which are never stored).
// Every other input is [B, K] read at column 64 kb.
__device__ __forceinline__ void act_coord(const FusedParams& p, const Phase& ph, int kb, int& x, int& y) {
    if (ph.kind != K_OPROJ) { x = kb * 64; y = 0; return; }
    const QkvMap& q = p.qkv;
    const int col = kb * 64;
    const int head = col / q.head_dim;
    const int g = head / (q.n_q / q.n_kv);
    const int s = q.tp <= q.n_kv ? g / q.kv_s : g * (q.tp / q.n_kv);
    const int c = q.tp <= q.n_kv ? g - s * q.kv_s : 0;
    x = (q.nq_s + q.kv_s + c) * q.head_dim + (col - head * q.head_dim);
    y = s * p.B;
}

__device__ __forceinline__ int src_tile(const FusedParams& p, const Phase& ph, int kb) {
    if (ph.kind != K_OPROJ) return kb >> 1;
    const int hd = p.qkv.head_dim;
    const int col = kb * 64;
    const int head = col / hd;
    const int g = head / (p.qkv.n_q / p.qkv.n_kv);
    return ((p.qkv.n_q + p.qkv.n_kv + g) * hd + (col - head * hd)) >> 7;
}

// The CTA owning flattened index a: the largest c with floor(c T / G) <= a.
__device__ __forceinline__ int owner_of(int a, int total, int G) {
    return (int)((unsigned)((a + 1) * G - 1) / (unsigned)total);
}

// Whether CTA c's range is non-empty (always, unless the phase has fewer
// (m-tile, k-block) pairs than CTAs).
__device__ __forceinline__ bool has_work(int total, int G, int c) {
    return (unsigned)(total * (c + 1)) / (unsigned)G > (unsigned)(total * c) / (unsigned)G;
}

// The split part of a phase: the flattened (m-tile, k-block) pairs from
// index seg_base on (the tiles after the whole ones), seg_total of them,
// split over CTAs 0 .. gw-1.
__device__ __forceinline__ int seg_base(const Phase& ph) { return ph.whole * ph.nkb; }
__device__ __forceinline__ int seg_total(const Phase& ph) { return ph.total - seg_base(ph); }

// The units (m-tile, k-block range) of CTA c in a phase, in k order: its
// whole tile if it has one (WH), then its range [idx2, hi2) of the split part.
template <bool WH>
struct Units {
    int idx, hi, idx2, hi2;
    int nkb;
    bool rev;
    __device__ __forceinline__ Units() : idx(0), hi(0), idx2(0), hi2(0), nkb(1), rev(false) {}
    __device__ __forceinline__ Units(const Phase& ph, int c) : nkb(ph.nkb), rev(WH && ph.rev) {
        const unsigned gw = (unsigned)ph.gw;
        if constexpr (WH) {
            const int b = seg_base(ph);
            const unsigned t = (unsigned)seg_total(ph);
            idx = c < ph.whole ? c * ph.nkb : 0;
            hi = c < ph.whole ? idx + ph.nkb : 0;
            idx2 = c < ph.gw ? b + (int)(t * c / gw) : 0;
            hi2 = c < ph.gw ? b + (int)(t * (c + 1) / gw) : 0;
        } else {
            idx = c < ph.gw ? (int)((unsigned)ph.total * c / gw) : 0;
            hi = c < ph.gw ? (int)((unsigned)ph.total * (c + 1) / gw) : 0;
            idx2 = hi2 = 0;
        }
    }
    __device__ __forceinline__ bool next(int& mt, int& kb0, int& kb1) {
        if (idx >= hi) {
            if (!WH || idx2 >= hi2) return false;
            idx = idx2;
            hi = hi2;
            idx2 = hi2 = 0;
        }
        if (WH && rev) {                    // the range's last m-tile first
            mt = (int)((unsigned)(hi - 1) / (unsigned)nkb);
            const int start = max(idx, mt * nkb);
            kb0 = start - mt * nkb;
            kb1 = hi - mt * nkb;
            hi = start;
            return true;
        }
        mt = (int)((unsigned)idx / (unsigned)nkb);
        kb0 = idx - mt * nkb;
        kb1 = min(nkb, kb0 + (hi - idx));
        idx += kb1 - kb0;
        return true;
    }
};

// Walks the weight tiles this CTA loads, in load order, across phases and
// layers (a gate/up k-block is two tiles: gate, then up).
template <bool WH>
struct TileCursor {
    int k;
    Phase ph;
    Units<WH> u;
    int mt, kb, kb1, hf;
    __device__ __forceinline__ bool next(const FusedMaps& mp, const FusedParams& p, int G, int cta, int n_phases,
                                         const CUtensorMap*& map, int& x, int& y) {
        for (;;) {
            if (kb < kb1) {
                map = hf ? ph.wb : ph.wa;
                x = kb * 64;
                y = mt * 128;
                if (++hf == (ph.kind == K_GATEUP ? 2 : 1)) { hf = 0; ++kb; }
                return true;
            }
            int kb0;
            if (k >= 1 && u.next(mt, kb0, kb1)) { kb = kb0; hf = 0; continue; }
            if (++k >= n_phases) return false;
            ph = phase_of<WH>(mp, p, k);
            u = Units<WH>(ph, cta);
            kb = kb1 = 0;
        }
    }
};

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ float warp_sum32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Counter increment with release semantics: everything this thread (and,
// through a preceding barrier, its CTA) wrote is visible before the count.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until a counter in global memory reaches target (acquire).
__device__ __noinline__ bool grid_wait(const unsigned* bar, unsigned target, volatile int* labort,
                                       volatile int* gabort, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
        if (v >= target) return true;
        if ((i & 15u) == 15u) {
            if (*labort || *gabort) return false;
            if (globaltimer() - t0 > limit_ns) return false;
        }
        if (i > 64) __nanosleep(32);
    }
}

// Tagged partial words (the 16-column instantiation): an fp32 partial and a
// 32-bit tag (layer + 1) stored as one aligned 8-byte word, which a reader
// sees whole or not at all, so a finalizer polls the data itself and the
// writer needs neither a fence nor a ticket.
__device__ __forceinline__ void st_tagged(uint64_t* a, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_tagged2(const uint64_t* a) {
    ulonglong2 r;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(a) : "memory");
    return r;
}

// 16-byte global -> shared copy through L2 only (cp.async, no registers held
// while it is in flight), and the wait for every copy this thread issued.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// This lane's share of token t's RMSNorm tile sums (tiles lane, lane+32, ...,
// added in that order).  The first two loads are issued together, so the
// usual D <= 8192 costs one round trip, not one per tile.
__device__ __forceinline__ float tile_sums(const float* sl, int Dt, int B, int t, int lane) {
    const float a0 = lane < Dt ? __ldcg(sl + lane * B + t) : 0.f;
    const float a1 = lane + 32 < Dt ? __ldcg(sl + (lane + 32) * B + t) : 0.f;
    float s = 0.f;
    s += a0;
    s += a1;
    for (int m2 = lane + 64; m2 < Dt; m2 += 32) s += __ldcg(sl + m2 * B + t);
    return s;
}

// Packed-QKV rows r0 .. r0+3 (one head: hd % 64 == 0) of token t, rounded
// to bf16, stored as one 8-byte word into every shard block that holds the
// head (KV groups are replicated over shards when tp > n_kv).
__device__ __forceinline__ void store_qkv4(const QkvMap& q, int t, int r0, float v0, float v1, float v2, float v3) {
    const int hd = q.head_dim;
    const int head = r0 / hd, d = r0 - head * hd;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v0, v1), hi = __floats2bfloat162_rn(v2, v3);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(q.qkv_out);
    if (head < q.n_q) {
        const int s = head / q.nq_s, j = head - s * q.nq_s;
        *reinterpret_cast<uint2*>(out + s * q.shard_stride + (int64_t)t * q.w_s + (int64_t)j * hd + d) = w;
        return;
    }
    const bool is_v = head >= q.n_q + q.n_kv;
    const int g = head - q.n_q - (is_v ? q.n_kv : 0);
    const int64_t col = (int64_t)(q.nq_s + (is_v ? q.kv_s : 0)) * hd + d;
    if (q.tp <= q.n_kv) {
        const int s = g / q.kv_s, c = g - s * q.kv_s;
        *reinterpret_cast<uint2*>(out + s * q.shard_stride + (int64_t)t * q.w_s + col + (int64_t)c * hd) = w;
    } else {
        const int copies = q.tp / q.n_kv;
        for (int s = g * copies; s < (g + 1) * copies; ++s)
            *reinterpret_cast<uint2*>(out + s * q.shard_stride + (int64_t)t * q.w_s + col) = w;
    }
}

// Release-publish two counter increments: every write this thread (and,
// through a preceding barrier, its CTA) made is visible before either count.
__device__ __forceinline__ void publish2(unsigned* a, unsigned* b, unsigned v) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(b), "r"(v) : "memory");
}

// Warp-collective: how many of this CTA's (m-tile, k-block) pairs idx, idx+1,
// .. < hi of phase ph (at most 32, flattened m-major like Units) lead with
// the source tiles of their k-blocks final, waiting until at least one is.
// Lane j polls the ready counter of pair idx+j (acquire; pairs of different
// m-tiles with the same k-block read the same counter), so one round trip
// usually covers a CTA's whole share of a phase.  The count returned is the
// same in every lane; 0: the wait gave up (time limit or abort).  Every lane
// then fences the async proxy, so the TMA loads issued after the warp
// barrier see the tiles' contents.
__device__ __forceinline__ int ready_prefix(const FusedParams& p, const Phase& ph, int idx, int hi,
                                            int lane, volatile int* labort, volatile int* gabort) {
    const int want = min(hi - idx, 32);
    const unsigned* ctr = nullptr;
    if (lane < want) {
        const int kb = (int)((unsigned)(idx + lane) % (unsigned)ph.nkb);
        ctr = p.ready + ph.src_kind * p.max_mt + src_tile(p, ph, kb);
    }
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        bool r = true;
        if (ctr) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            r = v >= ph.src_target;
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, r);
        const int lead = __ffs(~m) == 0 ? 32 : __ffs(~m) - 1;     // leading ready pairs
        const int n = min(want, lead);
        if (n > 0) {
            fence_proxy_async_global();
            __syncwarp();
            return n;
        }
        if ((i & 15u) == 15u) {
            const bool stop = *labort || *gabort || globaltimer() - t0 > p.wait_ns;
            if (__any_sync(0xFFFFFFFFu, stop)) return 0;
        }
        if (i > 64) __nanosleep(32);
    }
}

template <int NP, bool WHT>
__global__ void __launch_bounds__(kFThreads, 1)
fused_stack_kernel(const __grid_constant__ FusedMaps mp, const FusedParams p) {
    using C = FCfg<NP>;
    // gate/up tiles taken whole (the launch picks this build when gate/up has
    // at least one 128-row tile per CTA: at 32 and 128 columns, where the
    // gate/up finalize is long; built without it, the other shapes skip its
    // extra unit ranges, which cost them about 1%)
    constexpr bool WH = WHT;
    constexpr bool LL = NP <= kTaggedNP;  // tagged partial words instead of tile tickets
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ctrl = smem + C::STAGES * C::STAGE;
    uint64_t* full_w = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* full_x = full_w + C::STAGES;
    uint64_t* empty = full_x + C::STAGES;
    uint64_t* acc_full = empty + C::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 1000);
    volatile int* labort = reinterpret_cast<volatile int*>(ctrl + 1004);
    int* fin_ok = reinterpret_cast<int*>(ctrl + 1008);         // latest phase whose previous finalizing phase is complete
    int* seg = reinterpret_cast<int*>(ctrl + C::CTRL);          // partial slots of the tile being finalized
    float4* fin_buf = reinterpret_cast<float4*>(ctrl + C::CTRL + C::EPI);   // [4 warps][FIN_ITEMS][32 lanes]
    int* seg2 = seg + kFusedGridCap;                            // ... of its o_proj part (parallel block)
    volatile int* seg_info = seg2 + kFusedGridCap;              // [nseg, -, nseg2, -]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, cta = blockIdx.x;
    const int n_phases = 1 + 4 * p.L;
    volatile int* gabort = p.gabort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_addr(&full_w[s]), 1);
            mbar_init(smem_addr(&full_x[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&acc_full[a]), 1);
            mbar_init(smem_addr(&acc_empty[a]), 4);
        }
        mbar_init(smem_addr(drain), 1);
        *labort = 0;
        *fin_ok = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == kWarpMma) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        *labort = 1;
        atomicExch(p.gabort, 1);
        if (p.err) atomicOr(p.err, TPL_DEVERR_TIMEOUT);
    };

    if (warp == kWarpW) {
        // ---------------------------------------------------- weight producer
        // Loads every weight tile of this CTA into the ring, across phase and
        // layer boundaries (weights never depend on activations).
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            TileCursor<WH> ld{};
            int stage = 0;
            uint32_t par = 0;
            int last_par[C::STAGES];           // parity of the latest copy issued into each stage, -1: none
            for (int s = 0; s < C::STAGES; ++s) last_par[s] = -1;
            const CUtensorMap* map;
            int x, y;
            bool ok = true;
            int traced_k = -1;
            while (ok && ld.next(mp, p, G, cta, n_phases, map, x, y)) {
                if (ld.k != traced_k) { traced_k = ld.k; TPL_TRACE(ld.k, 6); }
                if (!mbar_wait(smem_addr(&empty[stage]), par ^ 1, labort, gabort, p.wait_ns)) { ok = false; break; }
                const uint32_t fb = smem_addr(&full_w[stage]);
                mbar_expect_tx(fb, C::W_BYTES);
                tma_load_hint(smem_addr(smem + stage * C::STAGE), map, fb, x, y, pol);
                TPL_TRACE(ld.k, 9);
                last_par[stage] = (int)par;
                if (++stage == C::STAGES) { stage = 0; par ^= 1; }
            }
            if (!ok) {
                fail();
                // let the copies already issued land before the CTA exits
                for (int s = 0; s < C::STAGES; ++s) {
                    if (last_par[s] < 0) continue;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_addr(&full_w[s]), (uint32_t)last_par[s]) &&
                           globaltimer() - t0 < kWaitLimitNs) {}
                }
            }
        }
    } else if (warp == kWarpAct) {
        // ---------------------------------------------------- activation producer
        // Fills the activation half of each stage once the source tiles of its
        // k-block are final (the whole warp polls their ready counters, lane 0
        // issues the copies).  The second stage of a gate/up k-block reuses the
        // first one's activations: its activation barrier still completes a
        // phase (a plain arrive), so every barrier of the ring advances once
        // per round, and the MMA issuer waits for that arrive too, so no
        // producer falls a round behind the releases it waits for.
        const uint64_t pol = policy_evict_last();
        int stage = 0;
        uint32_t par = 0;
        int last_par[C::STAGES];
        for (int s = 0; s < C::STAGES; ++s) last_par[s] = -1;
        bool ok = true;
        for (int k = 1; k < n_phases && ok; ++k) {
            const Phase ph = phase_of<WH>(mp, p, k);
            const int halves = ph.kind == K_GATEUP ? 2 : 1;
            const Units<WH> u(ph, cta);        // this CTA's pairs: [u.idx, u.hi) then [u.idx2, u.hi2)
            // the pairs [r_lo, r_hi) in order: ready polls of up to 32 at a time,
            // then one copy per k-block
            auto feed = [&](int r_lo, int r_hi, bool first_range) {
                for (int idx = r_lo; ok && idx < r_hi;) {
                    int n = min(r_hi - idx, 32);
                    const bool first_k = first_range && idx == r_lo;
                    if (first_k && lane == 0) TPL_TRACE(k, 7);
                    if (ph.src_kind >= 0) {
                        n = ready_prefix(p, ph, idx, r_hi, lane, labort, gabort);
                        if (n == 0) { ok = false; break; }
                    }
                    if (first_k && lane == 0) TPL_TRACE(k, 0);
                    if (lane == 0) {
                        int kb = (int)((unsigned)idx % (unsigned)ph.nkb);
                        for (int j = 0; j < n && ok; ++j, kb = kb + 1 == ph.nkb ? 0 : kb + 1) {
                            for (int hf = 0; hf < halves; ++hf) {
                                if (!mbar_wait(smem_addr(&empty[stage]), par ^ 1, labort, gabort, p.wait_ns)) { ok = false; break; }
                                const uint32_t fb = smem_addr(&full_x[stage]);
                                if (hf == 0) {
                                    mbar_expect_tx(fb, C::X_BYTES);
                                    int ax, ay;
                                    act_coord(p, ph, kb, ax, ay);
                                    tma_load_hint(smem_addr(smem + stage * C::STAGE + C::W_BYTES), ph.act, fb, ax, ay, pol);
                                    TPL_TRACE(k, 11);
                                } else {
                                    mbar_arrive(fb);
                                }
                                last_par[stage] = (int)par;
                                if (++stage == C::STAGES) { stage = 0; par ^= 1; }
                            }
                        }
                    }
                    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
                    idx += n;
                }
            };
            if (WH && ph.rev) {
                // unit by unit, in the order the MMA issuer takes them
                Units<WH> uu(ph, cta);
                int mt_u, kb0_u, kb1_u;
                bool first_u = true;
                while (ok && uu.next(mt_u, kb0_u, kb1_u)) {
                    feed(mt_u * ph.nkb + kb0_u, mt_u * ph.nkb + kb1_u, first_u);
                    first_u = false;
                }
            } else {
                for (int range = 0; range < (WH ? 2 : 1) && ok; ++range)
                    feed(range ? u.idx2 : u.idx, range ? u.hi2 : u.hi, range == 0 ? u.idx < u.hi : u.idx >= u.hi);
            }
        }
        if (!ok && lane == 0) {
            fail();
            for (int s = 0; s < C::STAGES; ++s) {
                if (last_par[s] < 0) continue;
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_addr(&full_x[s]), (uint32_t)last_par[s]) &&
                       globaltimer() - t0 < kWaitLimitNs) {}
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(128, NP);
            int stage = 0;
            uint32_t par = 0;
            int uc = 0;
            bool ok = true;
            for (int k = 1; k < n_phases && ok; ++k) {
                const Phase ph = phase_of<WH>(mp, p, k);
                const bool dual = ph.kind == K_GATEUP;
                Units<WH> u(ph, cta);
                int mt, kb0, kb1;
                const int uc_phase0 = uc;
                while (ok && u.next(mt, kb0, kb1)) {
                    const int a = uc & 1;
                    if (!mbar_wait(smem_addr(&acc_empty[a]), ((uc >> 1) & 1) ^ 1, labort, gabort, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem + a * kAccStride;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(smem_addr(&full_w[stage]), par, labort, gabort, p.wait_ns) ||
                            !mbar_wait(smem_addr(&full_x[stage]), par, labort, gabort, p.wait_ns)) { ok = false; break; }
                        tc_fence_after();
                        if (kb == kb0 && uc == uc_phase0) TPL_TRACE(k, 1);
                        const uint32_t sw = smem_addr(smem + stage * C::STAGE);
                        const uint32_t sx = sw + C::W_BYTES;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16(d, sw128_desc(sw + kk * 32), sw128_desc(sx + kk * 32), idesc,
                                     (kb > kb0 || kk > 0) ? 1u : 0u);
                        int s2 = stage + 1;
                        uint32_t p2 = par;
                        if (s2 == C::STAGES) { s2 = 0; p2 ^= 1; }
                        if (dual) {
                            // the up half's stage: its weights, and the activation
                            // producer's plain arrive (waited for so that the MMA
                            // never releases the stage a round before the producer
                            // has waited for it: the parity waits would alias)
                            if (!mbar_wait(smem_addr(&full_w[s2]), p2, labort, gabort, p.wait_ns) ||
                                !mbar_wait(smem_addr(&full_x[s2]), p2, labort, gabort, p.wait_ns)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t sw2 = smem_addr(smem + s2 * C::STAGE);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16(d + NP, sw128_desc(sw2 + kk * 32), sw128_desc(sx + kk * 32), idesc,
                                         (kb > kb0 || kk > 0) ? 1u : 0u);
                            mma_commit(smem_addr(&empty[stage]));
                            mma_commit(smem_addr(&empty[s2]));
                            stage = s2 + 1;
                            par = p2;
                            if (stage == C::STAGES) { stage = 0; par ^= 1; }
                        } else {
                            mma_commit(smem_addr(&empty[stage]));
                            stage = s2;
                            par = p2;
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_addr(&acc_full[a]));
                    if (uc == uc_phase0) TPL_TRACE(k, 8);
                    ++uc;
                }
            }
            if (!ok) fail();
            // every MMA issued above must complete before TMEM is released
            mma_commit(smem_addr(drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_addr(drain), 0) && globaltimer() - t0 < kWaitLimitNs) {}
        }
    } else if (warp == kWarpWatch) {
        // ---------------------------------------------------- phase watcher
        // Waits, phase after phase, until the phase that phase k's finalize
        // follows is complete, and posts k in shared memory, so the finalizing
        // warps find the answer there instead of polling global memory
        // on their critical path.
        if (lane == 0) {
            for (int k = 1; k < n_phases; ++k) {
                const Phase ph = phase_of<WH>(mp, p, k);
                if (ph.prev_fin >= 0 &&
                    !grid_wait(p.done + ph.prev_fin, done_target(mp, p, ph.prev_fin), labort, gabort, p.wait_ns)) {
                    fail();
                    break;
                }
                asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(fin_ok)), "r"(k) : "memory");
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2..5)
        // (warps 0, 1 and 6 have their own roles above)
        // Control flow is identical in all four warps, so the named barriers
        // (bar 1, 128 threads) always match; after an abort the waits return
        // at once and the memory work is skipped.
        const int q = warp & 3;
        const int row = q * 32 + lane;                 // drain: row of the tile (TMEM lane)
        const bool leader = warp == 2 && lane == 0;
        const bool helper = warp == 3 && lane == 0;    // waits for the previous phase beside the leader
        // bounded wait until the watcher has posted phase k (acquire)
        auto posted = [&](int k) {
            const uint64_t t0 = globaltimer();
            for (uint32_t i = 0;; ++i) {
                int v;
                asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(fin_ok)) : "memory");
                if (v >= k) return true;
                if ((i & 15u) == 15u && (*labort || *gabort || globaltimer() - t0 > p.wait_ns)) return false;
            }
        };
        const int B = p.B, D = p.D;
        const int Dt = (D + 127) / 128;
        bool dead = false;

        // phase 0: tile sums of squares of the launch input (warp per token)
        unsigned n0 = 0;
        for (int mt = cta; mt < Dt; mt += G) {
            for (int t = q; t < B; t += 4) {
                float ss = 0.f;
                const int f = mt * 128 + lane * 4;
                if (f < D) {
                    const uint2 v = __ldcg(reinterpret_cast<const uint2*>(p.x_in + (int64_t)t * D + f));
                    const float a0 = __uint_as_float(v.x << 16), a1 = __uint_as_float(v.x & 0xFFFF0000u);
                    const float a2 = __uint_as_float(v.y << 16), a3 = __uint_as_float(v.y & 0xFFFF0000u);
                    ss = a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
                }
                ss = warp_sum32(ss);
                if (lane == 0) p.slots_y[mt * B + t] = ss;
            }
            n0 += (unsigned)B;
        }
        epi_sync();
        if (leader && n0) red_release_add(p.done, n0);

        const size_t region = (size_t)(kFusedGridCap + p.max_mt);    // partial slots per projection kind
        int uc = 0;
        for (int k = 1; k < n_phases; ++k) {
            const Phase ph = phase_of<WH>(mp, p, k);
            const bool dual = ph.kind == K_GATEUP;
            const int planes = dual ? 2 : 1;
            const int l = ph.layer;
            // parallel block: o_proj and down partials of a tile are added
            // together (one reduction for both sublayers), so they share the
            // down tile's ticket and its finalize
            const bool merged = p.parallel && ph.kind == K_DOWN;
            const int tk_kind = (p.parallel && ph.kind == K_OPROJ) ? K_DOWN : ph.kind;
            Units<WH> u(ph, cta);
            int mt, kb0, kb1;
            const int first_uc = uc;
            // the serial block's MLP normalises h, everything else the layer input
            const float* sl = (ph.kind == K_GATEUP && !p.parallel) ? p.slots_h : p.slots_y;
            // pass 1: drain every unit into its partial slot and count it on
            // its tile's ticket (no waiting here, so tiles never wait on one
            // another through a CTA that holds pieces of two of them); a whole
            // gate/up tile is finished here instead
            while (u.next(mt, kb0, kb1)) {
                const int a = uc & 1;
                dead = dead || *labort || *gabort;
                const bool got = dead ? false : mbar_wait(smem_addr(&acc_full[a]), (uc >> 1) & 1, labort, gabort, p.wait_ns);
                dead = !__all_sync(0xFFFFFFFFu, got);
                if (dead && lane == 0) fail();
                if (leader && uc == first_uc) TPL_TRACE(k, 10);
                float* slot = p.part + ((size_t)ph.kind * region + cta + mt) * C::PART_FLOATS;
                const bool whole = WH && mt < ph.whole;  // the same in every epilogue warp
                if (whole) {
                    // h = SwiGLU of the RMSNorm-scaled accumulators, as a finalize
                    // computes it.  Every tile sum of the norm's input is final
                    // once the phase before this one has finished.
                    if (helper && !dead && ph.prev_fin >= 0 && !posted(k)) fail();
                    epi_sync();
                    dead = dead || *labort;
                    float* scl = reinterpret_cast<float*>(seg);     // per-token scales (the segment lists are idle)
                    if (!dead) {
                        for (int t = q; t < B; t += 4) {
                            const float ss = warp_sum32(tile_sums(sl, Dt, B, t, lane));
                            if (lane == 0) scl[t] = 1.0f / sqrtf(ss / (float)D + p.eps);
                        }
                    }
                    epi_sync();
                    if (!dead) {
                        tc_fence_after();
                        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + a * kAccStride;
                        const int r0 = mt * 128 + row;
#pragma unroll 1
                        for (int c0 = 0; c0 < NP && c0 < B; c0 += 16) {
                            float g[32], up[32];            // (16 columns used)
                            tmem_ld16(tb + c0, g);
                            tmem_ld16(tb + NP + c0, up);
                            if (r0 < p.F) {
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const int t = c0 + j;
                                    if (t < B) {
                                        const float sc = scl[t];
                                        p.H[(int64_t)t * p.F + r0] = __float2bfloat16_rn(silu_f(g[j] * sc) * (up[j] * sc));
                                    }
                                }
                            }
                        }
                    }
                } else if (LL && !dead) {
                    // [plane][token][row] tagged words; the test hook leaves one unit unwritten
                    tc_fence_after();
                    const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + a * kAccStride;
                    const bool skip_w = cta == p.skip_cta && k == p.skip_phase && uc == first_uc;
                    uint64_t* s64 = reinterpret_cast<uint64_t*>(p.part) +
                                    ((size_t)ph.kind * region + cta + mt) * (size_t)(2 * B * 128);
                    const uint64_t tag = (uint64_t)(l + 1) << 32;
                    for (int pl = 0; pl < planes; ++pl) {
#pragma unroll 1
                        for (int c0 = 0; c0 < NP && c0 < B; c0 += C::CH) {
                            float v[32];
                            if (C::CH == 32) tmem_ld32(tb + pl * NP + c0, v); else tmem_ld16(tb + pl * NP + c0, v);
#pragma unroll
                            for (int j = 0; j < C::CH; ++j)
                                if (c0 + j < B && !skip_w)
                                    st_tagged(s64 + (size_t)(pl * B + c0 + j) * 128 + row, tag | __float_as_uint(v[j]));
                        }
                    }
                } else if (!dead) {
                    tc_fence_after();
                    const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + a * kAccStride;
                    for (int pl = 0; pl < planes; ++pl) {
#pragma unroll 1
                        for (int c0 = 0; c0 < NP && c0 < B; c0 += C::CH) {
                            float v[32];
                            if (C::CH == 32) tmem_ld32(tb + pl * NP + c0, v); else tmem_ld16(tb + pl * NP + c0, v);
#pragma unroll
                            for (int j = 0; j < C::CH; ++j)
                                if (c0 + j < B) slot[(pl * NP + c0 + j) * 128 + row] = v[j];
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&acc_empty[a]));
                ++uc;
                epi_sync();                     // this CTA's partial of the tile (or the whole tile) is written
                const bool skip = cta == p.skip_cta && k == p.skip_phase && uc == first_uc + 1;
                if (whole) {
                    if (leader && !dead && !skip) publish2(p.ready + ph.kind * p.max_mt + mt, p.done + k, (unsigned)B);
                } else if (!LL && leader && !dead && !skip) {
                    red_release_add(p.tickets + tk_kind * p.max_mt + mt, 1u);
                }
                if (leader && uc == first_uc + 1) TPL_TRACE(k, 2);
            }
            if (leader) TPL_TRACE(k, 3);
            if (p.parallel && ph.kind == K_OPROJ) continue;    // finalized with down
            // pass 2: the phase's (tile, token) pairs, m_tiles x B in
            // tile-major order, are split evenly over the CTAs; CTA c
            // finalizes pairs [c W / G, (c+1) W / G), a tile at a time, once
            // all of the tile's units have arrived (a tile ticket counts
            // arrivals monotonically over the layers of the launch).  Any CTA
            // can finalize any tile: its partials are added in k order, so the
            // sum does not depend on which CTA adds them.
            // segments of tile mt of phase phx in k order: the CTAs from the
            // owner of its first k-block to the owner of its last one, all of
            // which hold work unless the phase has fewer pairs than CTAs (then
            // warp 2 lists the ones that do into list / seg_info[info])
            auto seg_list = [&](const Phase& phx, int mt_, int* list, int info, int& cf_, bool& every_) {
                const int sb = seg_base(phx), st = seg_total(phx);
                every_ = st >= phx.gw;
                cf_ = owner_of(mt_ * phx.nkb - sb, st, phx.gw);
                const int cl_ = owner_of(mt_ * phx.nkb + phx.nkb - 1 - sb, st, phx.gw);
                if (!every_ && warp == 2) {
                    int n = 0;
                    for (int base = cf_; base <= cl_; base += 32) {
                        const int cc = base + lane;
                        const bool w = cc <= cl_ && has_work(st, phx.gw, cc);
                        const unsigned m = __ballot_sync(0xFFFFFFFFu, w);
                        if (w) list[n + __popc(m & ((1u << lane) - 1u))] = cc + mt_;
                        n += __popc(m);
                    }
                    if (lane == 0) seg_info[info] = n;
                }
                return cl_;
            };
            const Phase ph_o = merged ? phase_of<WH>(mp, p, k - 1) : ph;   // the o_proj phase of the layer
            const bool normed = ph.kind == K_QKV || ph.kind == K_GATEUP;
            bool prev_done = ph.prev_fin < 0;
            // (tiles before ph.whole were finished whole in pass 1)
            // 128 columns, QKV: the tiles holding V rows first, spread over every
            // CTA, then the Q and K tiles.  o_proj reads only V, so its stream
            // starts while the rest is being finalized (which CTA adds which
            // pair changes no sum).  (Measured: +2% on the Llama-3.1-70B shape at
            // 128 tokens, where a CTA finalizes ~70 pairs; at a few pairs a CTA
            // it moved V's finalizers away from V's segments and cost up to 7%.)
            const int nsplit = ph.m_tiles - ph.whole;
            const int pt0 = (NP == 128 && ph.kind == K_QKV)
                ? min(nsplit, (p.qkv.n_q + p.qkv.n_kv) * p.qkv.head_dim / 128) : nsplit;
            for (int rg = 0; rg < 2; ++rg) {
            const unsigned ntr = (unsigned)(rg == 0 ? nsplit - pt0 : pt0);   // split tiles in this range
            const unsigned npairs = ntr * (unsigned)B;
            const int fbase = rg == 0 ? pt0 * B : 0;
            int f0, f1;
            if (NP <= 64 && npairs > (unsigned)G && ntr <= (unsigned)G) {
                // more (tile, token) pairs than CTAs, but no more tiles: each tile
                // gets a contiguous group of CTAs that divides its tokens, so no
                // CTA finalizes parts of two tiles one after the other (two polls
                // and two epilogues in series: the last such CTA held up the next
                // phase by about 3 us at 8 tokens).  (Measured at 128 columns,
                // where a CTA finalizes ~60 pairs, it cost 3%, so that build keeps
                // the even split.)
                const unsigned i = (unsigned)cta * ntr / (unsigned)G;
                const unsigned c0 = (i * (unsigned)G + ntr - 1) / ntr, c1 = ((i + 1) * (unsigned)G + ntr - 1) / ntr;
                const unsigned j = (unsigned)cta - c0, g = c1 - c0;
                f0 = fbase + (int)(i * (unsigned)B + (unsigned)B * j / g);
                f1 = fbase + (int)(i * (unsigned)B + (unsigned)B * (j + 1) / g);
            } else {
                f0 = fbase + (int)(npairs * cta / (unsigned)G);
                f1 = fbase + (int)(npairs * (cta + 1) / (unsigned)G);
            }
            for (int f = f0; f < f1;) {
                const int fm = (int)((unsigned)f / (unsigned)B);   // tile index among the split tiles
                mt = ph.whole + (int)fm;
                // this CTA's tokens of tile mt
                const int t_lo = (int)(f - fm * B);
                const int t_hi = min(B, f1 - fm * B);
                f = fm * B + t_hi;
                int cf, cf_o = 0;
                bool every, every_o = true;
                const int cl = seg_list(ph, mt, seg, 0, cf, every);
                int cl_o = -1;
                if (merged) cl_o = seg_list(ph_o, mt, seg2, 2, cf_o, every_o);
                epi_sync();
                const int nseg_d = every ? cl - cf + 1 : seg_info[0];
                const int nseg_o = !merged ? 0 : (every_o ? cl_o - cf_o + 1 : seg_info[2]);
                const int nseg = nseg_o + nseg_d;
                // slot of segment j: the o_proj segments first, then this
                // phase's own, each in k order
                auto slot_of = [&](int j) -> size_t {
                    if (j < nseg_o) return (size_t)K_OPROJ * region + (size_t)(every_o ? cf_o + j + mt : seg2[j]);
                    const int jd = j - nseg_o;
                    return (size_t)ph.kind * region + (size_t)(every ? cf + jd + mt : seg[jd]);
                };

                // every unit of the tile has arrived, and the phase finalized
                // before this one is complete (so are all earlier ones: each
                // waited likewise); two threads wait side by side
                if (!LL && leader && !dead &&
                    !grid_wait(p.tickets + tk_kind * p.max_mt + mt, (unsigned)nseg * (unsigned)(l + 1), labort, gabort, p.wait_ns))
                    fail();
                if (helper && !dead && !prev_done && !posted(k)) fail();
                if (leader && !prev_done) TPL_TRACE(k, 4);
                prev_done = true;
                epi_sync();                     // every segment of the tile is visible
                if (dead || *labort) { epi_sync(); continue; }

                // warp per token, lane per 4 consecutive rows; segments added
                // in k order, all loads of a token issued before the sum
                const int r0 = mt * 128 + lane * 4;
                const __nv_bfloat16* resid = (ph.kind == K_OPROJ || merged)
                    ? (l == 0 ? p.x_in : (((l - 1) & 1) ? p.R1 : p.R0)) : p.h;
                __nv_bfloat16* dst = ph.kind == K_OPROJ ? p.h : (l == p.L - 1 ? p.y_out : ((l & 1) ? p.R1 : p.R0));
                const float* pbase = p.part + lane * 4;     // + slot * PART_FLOATS
                const bool has_resid = ph.kind == K_OPROJ || ph.kind == K_DOWN;
                auto emit = [&](int t, const float4& acc, const float4& acc2, const uint2& rv, float s) {
                    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
                    if (ph.kind == K_QKV) {
                        if (r0 < p.n_qkv) store_qkv4(p.qkv, t, r0, av[0] * s, av[1] * s, av[2] * s, av[3] * s);
                    } else if (ph.kind == K_GATEUP) {
                        if (r0 < p.F) {
                            const float uv[4] = {acc2.x, acc2.y, acc2.z, acc2.w};
                            __nv_bfloat16 hb[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) hb[e] = __float2bfloat16_rn(silu_f(av[e] * s) * (uv[e] * s));
                            uint2 w;
                            w.x = (uint32_t)__bfloat16_as_ushort(hb[0]) | ((uint32_t)__bfloat16_as_ushort(hb[1]) << 16);
                            w.y = (uint32_t)__bfloat16_as_ushort(hb[2]) | ((uint32_t)__bfloat16_as_ushort(hb[3]) << 16);
                            *reinterpret_cast<uint2*>(p.H + (int64_t)t * p.F + r0) = w;
                        }
                    } else {
                        // residual add; the rounded values also feed the next RMSNorm
                        float ss = 0.f;
                        if (r0 < D) {
                            const float rr[4] = {__uint_as_float(rv.x << 16), __uint_as_float(rv.x & 0xFFFF0000u),
                                                 __uint_as_float(rv.y << 16), __uint_as_float(rv.y & 0xFFFF0000u)};
                            __nv_bfloat16 hb[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                hb[e] = __float2bfloat16_rn(rr[e] + av[e]);
                                const float hv = __bfloat162float(hb[e]);
                                ss = fmaf(hv, hv, ss);
                            }
                            uint2 w;
                            w.x = (uint32_t)__bfloat16_as_ushort(hb[0]) | ((uint32_t)__bfloat16_as_ushort(hb[1]) << 16);
                            w.y = (uint32_t)__bfloat16_as_ushort(hb[2]) | ((uint32_t)__bfloat16_as_ushort(hb[3]) << 16);
                            *reinterpret_cast<uint2*>(dst + (int64_t)t * D + r0) = w;
                        }
                        ss = warp_sum32(ss);
                        if (lane == 0) (ph.kind == K_OPROJ ? p.slots_h : p.slots_y)[mt * B + t] = ss;
                    }
                };
                auto add4 = [](float4& a, const float4& b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; };
                // A warp takes TB of its tokens at a time (TB = 2, or 3 in the
                // 128-column instantiation, when their segments fit its staging
                // rows, else 1).  Each lane copies
                // its own 16 bytes (4 rows) of every partial segment of the
                // batch's tokens (both planes for gate/up) into the warp's
                // staging rows with cp.async, up to SB segments per token and
                // batch, all in flight at once, and adds them from shared
                // memory in k order; the residuals, or the tokens' RMSNorm
                // tile sums (lanes over the tiles, summed lane-strided then by
                // a butterfly: a fixed order), load alongside.
                const uint32_t fb_s = smem_addr(fin_buf + q * (C::FIN_ITEMS * 32) + lane);
                const float4* fb = fin_buf + q * (C::FIN_ITEMS * 32) + lane;
                auto share_tb = [&](auto tb_c, auto dual_c, auto norm_c) {
                    constexpr int TB = decltype(tb_c)::value;
                    constexpr bool DU = decltype(dual_c)::value, NO = decltype(norm_c)::value;
                    constexpr int PL = DU ? 2 : 1;
                    constexpr int SB = C::FIN_ITEMS / (PL * TB);
                    for (int t0 = t_lo + q; t0 < t_hi; t0 += 4 * TB) {
                        float4 acc[TB], acc2[TB];
                        uint2 rv[TB];
                        float ssq[TB];
#pragma unroll
                        for (int j = 0; j < TB; ++j) {
                            acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                            acc2[j] = acc[j];
                            rv[j] = make_uint2(0u, 0u);
                            ssq[j] = 0.f;
                            const int t = t0 + 4 * j;
                            if (t < t_hi) {
                                if (has_resid && r0 < D)
                                    rv[j] = __ldcg(reinterpret_cast<const uint2*>(resid + (int64_t)t * D + r0));
                                if constexpr (NO) ssq[j] = tile_sums(sl, Dt, B, t, lane);
                            }
                        }
                        {
                        for (int s0 = 0; s0 < nseg; s0 += SB) {
                            const int nb = min(SB, nseg - s0);
#pragma unroll
                            for (int j = 0; j < TB; ++j) {
#pragma unroll
                                for (int k2 = 0; k2 < SB; ++k2) {
                                    const int t = t0 + 4 * j;
                                    if (t < t_hi && k2 < nb) {
                                        const float* sp = pbase + (size_t)slot_of(s0 + k2) * C::PART_FLOATS + t * 128;
                                        const uint32_t it = (uint32_t)((j * SB + k2) * PL);
                                        cp_async16(fb_s + it * 512u, sp);
                                        if constexpr (DU) cp_async16(fb_s + (it + 1) * 512u, sp + NP * 128);
                                    }
                                }
                            }
                            cp_async_wait_all();
#pragma unroll
                            for (int j = 0; j < TB; ++j) {
#pragma unroll
                                for (int k2 = 0; k2 < SB; ++k2) {
                                    if (t0 + 4 * j < t_hi && k2 < nb) {
                                        const int it = (j * SB + k2) * PL;
                                        add4(acc[j], fb[it * 32]);
                                        if constexpr (DU) add4(acc2[j], fb[(it + 1) * 32]);
                                    }
                                }
                            }
                        }
                        }
#pragma unroll
                        for (int j = 0; j < TB; ++j) {
                            float sc = 1.f;
                            if constexpr (NO) sc = 1.0f / sqrtf(warp_sum32(ssq[j]) / (float)D + p.eps);
                            if (t0 + 4 * j < t_hi) emit(t0 + 4 * j, acc[j], acc2[j], rv[j], sc);
                        }
                    }
                };
                // 16 columns: the tile's tagged partial words are polled by all
                // four warps at once (item i = token j x segment; warp i % 4 holds
                // it in registers), checked, staged in shared memory, and added
                // in k order by the token's warp (warp j of the round).  A round
                // takes as many whole tokens as the staging holds (at most 4),
                // or one token in chunks of segments.
                auto share_ll = [&](auto dual_c, auto norm_c) {
                    constexpr bool DU = decltype(dual_c)::value, NO = decltype(norm_c)::value;
                    constexpr int PL = DU ? 2 : 1;
                    constexpr int SLOTS = 6 / PL;                  // items a warp holds
                    constexpr int CAP = 4 * SLOTS;                 // items a round stages
                    static_assert(CAP * PL <= 4 * C::FIN_ITEMS, "staging rows");
                    const int tr = nseg >= CAP ? 1 : min(4, CAP / nseg);
                    const uint64_t* pb = reinterpret_cast<const uint64_t*>(p.part) + lane * 4;
                    const size_t sw = (size_t)2 * B * 128;
                    const uint32_t want = (uint32_t)(l + 1);
                    float4* stg = fin_buf;             // the whole staging area, [item][plane][lane]
                    for (int tb = t_lo; tb < t_hi; tb += tr) {
                        const int ntr = min(tr, t_hi - tb);
                        const int t = tb + q;                      // the token this warp adds up (q < ntr)
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), acc2 = acc;
                        uint2 rv = make_uint2(0u, 0u);
                        float ssq = 0.f;
                        if (q < ntr) {
                            if (has_resid && r0 < D) rv = __ldcg(reinterpret_cast<const uint2*>(resid + (int64_t)t * D + r0));
                            if constexpr (NO) ssq = tile_sums(sl, Dt, B, t, lane);
                        }
                        const int step = ntr == 1 ? CAP : nseg;
                        for (int c0 = 0; c0 < nseg; c0 += step) {
                            const int cn = min(step, nseg - c0);
                            const int nit = ntr * cn;
                            ulonglong2 w[SLOTS][PL][2];
                            auto item_ptr = [&](int i) {
                                const int j = (int)((unsigned)i / (unsigned)cn);
                                return pb + (size_t)slot_of(c0 + (i - j * cn)) * sw + (size_t)(tb + j) * 128;
                            };
#pragma unroll
                            for (int s2 = 0; s2 < SLOTS; ++s2) {
                                const int i = q + 4 * s2;
                                if (i < nit) {
                                    const uint64_t* ip = item_ptr(i);
#pragma unroll
                                    for (int pl = 0; pl < PL; ++pl) {
                                        w[s2][pl][0] = ld_tagged2(ip + (size_t)pl * B * 128);
                                        w[s2][pl][1] = ld_tagged2(ip + (size_t)pl * B * 128 + 2);
                                    }
                                }
                            }
                            const uint64_t t_start = globaltimer();
                            for (uint32_t it = 0;; ++it) {
                                bool all = true;
#pragma unroll
                                for (int s2 = 0; s2 < SLOTS; ++s2) {
                                    const int i = q + 4 * s2;
                                    bool ok = true;
#pragma unroll
                                    for (int pl = 0; pl < PL; ++pl) {
#pragma unroll
                                        for (int h2 = 0; h2 < 2; ++h2)
                                            ok = ok && (uint32_t)(w[s2][pl][h2].x >> 32) == want &&
                                                 (uint32_t)(w[s2][pl][h2].y >> 32) == want;
                                    }
                                    if (i < nit && !ok) {
                                        all = false;
                                        const uint64_t* ip = item_ptr(i);
#pragma unroll
                                        for (int pl = 0; pl < PL; ++pl) {
                                            w[s2][pl][0] = ld_tagged2(ip + (size_t)pl * B * 128);
                                            w[s2][pl][1] = ld_tagged2(ip + (size_t)pl * B * 128 + 2);
                                        }
                                    }
                                }
                                if (__all_sync(0xFFFFFFFFu, all)) break;
                                if ((it & 15u) == 15u &&
                                    __any_sync(0xFFFFFFFFu, *labort || *gabort || globaltimer() - t_start > p.wait_ns)) {
                                    if (lane == 0) fail();
                                    break;
                                }
                            }
#pragma unroll
                            for (int s2 = 0; s2 < SLOTS; ++s2) {
                                const int i = q + 4 * s2;
                                if (i < nit) {
#pragma unroll
                                    for (int pl = 0; pl < PL; ++pl)
                                        stg[(i * PL + pl) * 32 + lane] =
                                            make_float4(__uint_as_float((uint32_t)w[s2][pl][0].x), __uint_as_float((uint32_t)w[s2][pl][0].y),
                                                        __uint_as_float((uint32_t)w[s2][pl][1].x), __uint_as_float((uint32_t)w[s2][pl][1].y));
                                }
                            }
                            epi_sync();
                            if (q < ntr) {
                                for (int k2 = 0; k2 < cn; ++k2) {
                                    const int i = q * cn + k2;
                                    add4(acc, stg[(i * PL) * 32 + lane]);
                                    if constexpr (DU) add4(acc2, stg[(i * PL + 1) * 32 + lane]);
                                }
                            }
                            epi_sync();
                        }
                        if (q < ntr) {
                            float sc = 1.f;
                            if constexpr (NO) sc = 1.0f / sqrtf(warp_sum32(ssq) / (float)D + p.eps);
                            emit(t, acc, acc2, rv, sc);
                        }
                    }
                };
                using I1 = std::integral_constant<int, 1>;
                using I2 = std::integral_constant<int, 2>;
                auto share = [&](auto dual_c, auto norm_c) {
                    constexpr int PL = decltype(dual_c)::value ? 2 : 1;
                    // three tokens a batch at 128 columns, where a CTA finalizes ~60-200 pairs
                    if constexpr (NP == 128) {
                        if (3 * PL * nseg <= C::FIN_ITEMS) {
                            share_tb(std::integral_constant<int, 3>{}, dual_c, norm_c);
                            return;
                        }
                    }
                    if constexpr (NP > 32) {
                        if (2 * PL * nseg <= C::FIN_ITEMS) {
                            share_tb(I2{}, dual_c, norm_c);
                            return;
                        }
                    }
                    share_tb(I1{}, dual_c, norm_c);
                };
                using T = std::true_type;
                using Fa = std::false_type;
                if constexpr (LL) {
                    if (dual) share_ll(T{}, T{});
                    else if (normed) share_ll(Fa{}, T{});
                    else share_ll(Fa{}, Fa{});
                } else {
                    if (dual) share(T{}, T{});
                    else if (normed) share(Fa{}, T{});
                    else share(Fa{}, Fa{});
                }
                // this CTA's share of the tile is written: count it on the
                // tile (the next phase's activation loads wait for that) and
                // on the phase
                epi_sync();
                if (leader && !dead && !*labort)
                    publish2(p.ready + ph.kind * p.max_mt + mt, p.done + k, (unsigned)(t_hi - t_lo));
                if (leader) TPL_TRACE(k, 5);
            }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int np_for(int64_t B) { return B <= 16 ? 16 : B <= 32 ? 32 : B <= 64 ? 64 : 128; }

// Most segments per tile, per projection kind.  A tile split over s CTAs
// streams its weights s times faster but leaves s fp32 partials per token to
// add up, and the finalize is spread over the whole grid.  With one CTA's
// weight stream at about 44 GB/s and its finalize at R GB/s, a phase of W
// weight bytes and m tiles takes about
//     W / (m s 44) + m B s 512 PL / (G R)
// and the best s is the square root of the ratio of the two coefficients.
// The finalize is latency-bound (each batch of staged loads is one round
// trip, and a batch carries more tokens as B grows): R = 10 sqrt(B / 32)
// fits the Qwen2.5-1.5B-shaped stack at 32 and 64 tokens.  Phases with many
// weight bytes per tile (every phase below ~16 tokens, every Llama-3.1-70B-
// shaped phase) get a cap above the grid's own split, which then stands.
void segment_caps(const FusedShape& sh, int G, int (&cap)[4]) {
    const double B = (double)sh.B, D = (double)sh.D, F = (double)sh.F;
    const double n_qkv = (double)(sh.n_q + 2 * sh.n_kv) * sh.hd, ko = (double)sh.n_q * sh.hd;
    const double W[4] = {n_qkv * D * 2, D * ko * 2, 2 * F * D * 2, D * F * 2};
    const double M[4] = {n_qkv, D, F, D};
    const double PL[4] = {1, 1, 2, 1};
    for (int k = 0; k < 4; ++k) {
        const double m = std::ceil(M[k] / 128);
        const double R = 10.0 * std::sqrt(B / 32.0);
        const double best = std::sqrt(W[k] * G * R / (m * m * B * 512 * PL[k] * 44.0));
        cap[k] = (int)std::max(1.0, std::min(1e6, std::floor(best + 0.5)));
    }
}

// Test hook state (set by tpl_test_fused_fault): the next launches' wait
// limit and the CTA / phase whose first unit is not delivered (no ticket,
// or no tagged words).
std::atomic<int> g_skip_cta{-1}, g_skip_phase{-1};
std::atomic<long long> g_wait_ns{0};

template <int NP>
int fused_smem() { return FCfg<NP>::SMEM; }

int smem_for(int np) {
    switch (np) {
    case 16: return fused_smem<16>();
    case 32: return fused_smem<32>();
    case 64: return fused_smem<64>();
    default: return fused_smem<128>();
    }
}

struct FusedPlan {
    int np, max_mt;
    size_t ctrl_off, tick_off, ready_off, done_off, sy_off, sh_off, r0_off, r1_off, h_off, hid_off, qkv_off,
        part_off, total;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

FusedPlan plan_fused(const FusedShape& s) {
    FusedPlan f{};
    f.np = np_for(s.B);
    const int64_t n_qkv = (int64_t)(s.n_q + 2 * s.n_kv) * s.hd;
    const int64_t mts[4] = {(n_qkv + 127) / 128, (s.D + 127) / 128, (s.F + 127) / 128, (s.D + 127) / 128};
    f.max_mt = (int)*std::max_element(mts, mts + 4);
    const int64_t Dt = (s.D + 127) / 128;
    const int kv_s = s.tp <= s.n_kv ? s.n_kv / s.tp : 1;
    const int64_t w_s = (int64_t)(s.n_q / s.tp + 2 * kv_s) * s.hd;
    size_t o = 0;
    // control words, tickets, ready and done counters: zeroed before each launch
    f.ctrl_off = o; o += 256;
    f.tick_off = o; o += up256((size_t)4 * f.max_mt * 4);
    f.ready_off = o; o += up256((size_t)4 * f.max_mt * 4);
    f.done_off = o; o += up256((size_t)(1 + 4 * kFusedMaxLayers) * 4);
    // narrow instantiations: tagged partial words [4 kinds][slots][2][B][128] u64, zeroed
    // with the counters before each launch (a stale word never carries a live tag)
    const bool tagged = f.np <= kTaggedNP;
    if (tagged) { f.part_off = o; o += up256((size_t)4 * (kFusedGridCap + f.max_mt) * 2 * s.B * 128 * 8); }
    f.sy_off = o; o += up256((size_t)Dt * s.B * 4);
    f.sh_off = o; o += up256((size_t)Dt * s.B * 4);
    f.r0_off = o; o += up256((size_t)s.B * s.D * 2);
    f.r1_off = o; o += up256((size_t)s.B * s.D * 2);
    f.h_off = o; o += up256((size_t)s.B * s.D * 2);
    f.hid_off = o; o += up256((size_t)s.B * s.F * 2);
    f.qkv_off = o; o += up256((size_t)s.tp * s.B * w_s * 2);
    // one region of partial slots per projection kind
    if (!tagged) { f.part_off = o; o += up256((size_t)4 * (kFusedGridCap + f.max_mt) * 2 * f.np * 128 * 4); }
    f.total = o;
    return f;
}

// Shared-memory limit of one build, and how many of its CTAs fit an SM.
template <int NP, bool WHT>
cudaError_t prep_np(int smem, int& per_sm) {
    cudaError_t e = cudaFuncSetAttribute(fused_stack_kernel<NP, WHT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_stack_kernel<NP, WHT>, kFThreads, smem);
    return e;
}

template <int NP, bool WHT>
cudaError_t launch_np(const FusedMaps& maps, const FusedParams& prm, cudaStream_t st) {
    using C = FCfg<NP>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)prm.G);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_stack_kernel<NP, WHT>, maps, prm);
}

}  // namespace

bool fused_trace_read(void* host, size_t bytes) {
#ifdef TPL_FUSED_TRACE
    return bytes <= sizeof(g_fused_trace) && cudaMemcpyFromSymbol(host, g_fused_trace, bytes) == cudaSuccess;
#else
    (void)host;
    (void)bytes;
    return false;
#endif
}

void fused_test_fault(int cta, int phase, long long wait_ns) {
    g_skip_cta = cta;
    g_skip_phase = phase;
    g_wait_ns = wait_ns;
}

bool fused_stack_shape_ok(const FusedShape& s) {
    if (s.B < 1 || s.B > 128) return false;
    if (s.D % 64 || s.F % 64 || s.hd % 64) return false;
    const int64_t n_qkv = (int64_t)(s.n_q + 2 * s.n_kv) * s.hd, ko = (int64_t)s.n_q * s.hd;
    if (s.D > (1 << 20) || s.F > (1 << 20) || n_qkv > (1 << 20)) return false;
    // the work split indexes (m-tile, k-block) pairs in 32 bits: pairs x G < 2^31
    const int64_t MK[4][2] = {{n_qkv, s.D}, {s.D, ko}, {s.F, s.D}, {s.D, s.F}};
    for (const auto& mk : MK)
        if ((mk[0] + 127) / 128 * (mk[1] / 64) * kFusedGridCap >= (int64_t(1) << 31)) return false;
    return true;
}

size_t fused_stack_ws_bytes(const FusedShape& s) { return plan_fused(s).total; }

cudaError_t launch_fused_stack(const FusedShape& s, const void* x, void* y, const void* const* Wqkv,
                               const void* const* Wo, const void* const* Wg, const void* const* Wu,
                               const void* const* Wd, int n_layers, bool parallel, void* ws, cudaStream_t st) {
    const FusedPlan f = plan_fused(s);
    const DeviceCtx* ctx = device_ctx();
    if (!ctx) return cudaErrorNoDevice;
    char* w = static_cast<char*>(ws);
    const int64_t n_qkv = (int64_t)(s.n_q + 2 * s.n_kv) * s.hd;
    const int64_t ko = (int64_t)s.n_q * s.hd;

    int G = std::min(ctx->num_sms, kFusedGridCap);
    bool wh = false;       // the build with whole gate/up tiles
    {
        int per_sm = 0;
        const int smem = smem_for(f.np);
        cudaError_t e = cudaSuccess;
        switch (f.np) {
        case 16: e = prep_np<16, false>(smem, per_sm); break;
        case 32: e = prep_np<32, false>(smem, per_sm); break;
        case 64: e = prep_np<64, false>(smem, per_sm); break;
        default: e = prep_np<128, false>(smem, per_sm); break;
        }
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        G = std::min(G, per_sm * ctx->num_sms);
        wh = (f.np == 32 || f.np == 128) && (s.F + 127) / 128 >= G;
        if (wh) {
            int per_sm_wh = 0;
            e = f.np == 32 ? prep_np<32, true>(smem, per_sm_wh) : prep_np<128, true>(smem, per_sm_wh);
            if (e != cudaSuccess) return e;
            if (per_sm_wh < per_sm) return cudaErrorInvalidConfiguration;
        }
    }

    FusedParams prm{};
    prm.B = (int)s.B; prm.D = (int)s.D; prm.F = (int)s.F; prm.G = G;
    prm.parallel = parallel ? 1 : 0;
    prm.n_qkv = (int)n_qkv; prm.ko = (int)ko; prm.max_mt = f.max_mt; prm.eps = kRmsEpsilon;
    const int kv_s = s.tp <= s.n_kv ? s.n_kv / s.tp : 1;
    prm.qkv.n_q = s.n_q; prm.qkv.n_kv = s.n_kv; prm.qkv.head_dim = s.hd; prm.qkv.tp = s.tp;
    prm.qkv.nq_s = s.n_q / s.tp; prm.qkv.kv_s = kv_s;
    prm.qkv.w_s = (int64_t)(prm.qkv.nq_s + 2 * kv_s) * s.hd;
    prm.qkv.shard_stride = s.B * prm.qkv.w_s;
    prm.qkv.qkv_out = w + f.qkv_off;
    prm.qkv.o_out = nullptr;
    prm.qkv.ldo_o = 0;
    prm.R0 = reinterpret_cast<__nv_bfloat16*>(w + f.r0_off);
    prm.R1 = reinterpret_cast<__nv_bfloat16*>(w + f.r1_off);
    prm.h = reinterpret_cast<__nv_bfloat16*>(w + f.h_off);
    prm.H = reinterpret_cast<__nv_bfloat16*>(w + f.hid_off);
    prm.slots_y = reinterpret_cast<float*>(w + f.sy_off);
    prm.slots_h = reinterpret_cast<float*>(w + f.sh_off);
    prm.part = reinterpret_cast<float*>(w + f.part_off);
    prm.tickets = reinterpret_cast<unsigned*>(w + f.tick_off);
    prm.ready = reinterpret_cast<unsigned*>(w + f.ready_off);
    prm.done = reinterpret_cast<unsigned*>(w + f.done_off);
    prm.gabort = reinterpret_cast<int*>(w + f.ctrl_off);
    prm.err = ctx->err_word;
    prm.wait_ns = g_wait_ns > 0 ? (uint64_t)g_wait_ns : kWaitLimitNs;
    prm.skip_cta = g_skip_cta;
    prm.skip_phase = g_skip_phase;
    segment_caps(s, G, prm.s_cap);
    prm.y_out = static_cast<__nv_bfloat16*>(y);

    FusedMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const int np = f.np;
    if (!tma_map_bf16(&maps.act[A_R0], prm.R0, s.B, s.D, s.D, np) ||
        !tma_map_bf16(&maps.act[A_R1], prm.R1, s.B, s.D, s.D, np) ||
        !tma_map_bf16(&maps.act[A_QKV], prm.qkv.qkv_out, (int64_t)s.tp * s.B, prm.qkv.w_s, prm.qkv.w_s, np) ||
        !tma_map_bf16(&maps.act[A_H], prm.h, s.B, s.D, s.D, np) ||
        !tma_map_bf16(&maps.act[A_HID], prm.H, s.B, s.F, s.F, np))
        return cudaErrorInvalidValue;

    for (int l0 = 0; l0 < n_layers; l0 += kFusedMaxLayers) {
        const int L = std::min(kFusedMaxLayers, n_layers - l0);
        const void* xin = l0 == 0 ? x : y;
        prm.x_in = static_cast<const __nv_bfloat16*>(xin);
        prm.L = L;
        if (!tma_map_bf16(&maps.act[A_X], xin, s.B, s.D, s.D, np)) return cudaErrorInvalidValue;
        for (int l = 0; l < L; ++l) {
            if (!tma_map_bf16(&maps.w[l][W_QKV], Wqkv[l0 + l], n_qkv, s.D, s.D, 128) ||
                !tma_map_bf16(&maps.w[l][W_O], Wo[l0 + l], s.D, ko, ko, 128) ||
                !tma_map_bf16(&maps.w[l][W_G], Wg[l0 + l], s.F, s.D, s.D, 128) ||
                !tma_map_bf16(&maps.w[l][W_U], Wu[l0 + l], s.F, s.D, s.D, 128) ||
                !tma_map_bf16(&maps.w[l][W_D], Wd[l0 + l], s.D, s.F, s.F, 128))
                return cudaErrorInvalidValue;
        }
        // abort flag, tickets, ready and done counters start at zero
        cudaError_t e = cudaMemsetAsync(w + f.ctrl_off, 0, f.sy_off - f.ctrl_off, st);
        if (e != cudaSuccess) return e;
        switch (np) {
        case 16: e = launch_np<16, false>(maps, prm, st); break;
        case 32: e = wh ? launch_np<32, true>(maps, prm, st) : launch_np<32, false>(maps, prm, st); break;
        case 64: e = launch_np<64, false>(maps, prm, st); break;
        default: e = wh ? launch_np<128, true>(maps, prm, st) : launch_np<128, false>(maps, prm, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace tpl
