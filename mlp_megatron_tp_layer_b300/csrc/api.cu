// C-ABI entry points: argument validation, workspace layout, kernel choice.
//
// Kernel choice for bf16 (token count T of the call):
//   T == 1   : CUDA-core weight-streaming row-dot kernel
//   T <= 128 : tensor-core GEMM, swapped (weights are the M=128 operand)
//   T >  128 : tensor-core GEMM, tokens as the M operand
// fp32 calls always use the CUDA-core kernel (fp32 FMA, no TF32), in launches
// of at most kSimtMaxTokens tokens.  Measured on the Llama-3.1-70B-shaped MLP:
// at T = 1 both kernels stream 6.2 TB/s; at T = 2, 4, 8 the row-dot kernel
// falls to 4.6, 3.2, 1.9 TB/s (its fp32 FMAs per weight grow with T) while the
// swapped GEMM holds 5.9 TB/s.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "w8.h"

namespace tpl {

__device__ unsigned int g_device_error_word = 0;

namespace {

constexpr int kSimtMaxTokens = 8;     // tokens per row-dot launch
constexpr int kSimtMaxTokensBf16 = 1; // bf16 calls with more tokens take the tensor cores
constexpr int kDesignSMs = 148;       // split-K sizing target (B300); shapes only, so queries match launches
constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlap(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || !an || !bn) return false;
    const char* x = static_cast<const char*>(a);
    const char* y = static_cast<const char*>(b);
    return x < y + bn && y < x + an;
}
size_t esize(int dt) { return dt == TPL_BF16 ? 2 : 4; }
cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
tpl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TPL_OK : TPL_ERR_CUDA; }
bool out_dtype_ok(int dt, int out_dt) {
    return out_dt == TPL_F32 || (out_dt == TPL_BF16 && dt == TPL_BF16);
}

std::mutex g_ctx_mu;
DeviceCtx g_ctx[64];

// ------------------------------------------------- launch timing (optional)
// While enabled, every kernel launch is bracketed by a pair of CUDA events on
// its stream and tagged with the layer step it implements.
struct ProfSlot { cudaEvent_t start, stop; const char* tag; };
std::mutex g_prof_mu;
std::vector<ProfSlot> g_prof;
int g_prof_next = 0;
bool g_prof_on = false;

struct ProfScope {
    ProfSlot* slot = nullptr;
    cudaStream_t st;
    ProfScope(const char* tag, cudaStream_t s) : st(s) {
        if (!g_prof_on) return;
        std::lock_guard<std::mutex> lock(g_prof_mu);
        if (g_prof_next >= (int)g_prof.size()) return;
        slot = &g_prof[g_prof_next++];
        slot->tag = tag;
        record(slot->start);
    }
    ~ProfScope() {
        if (slot) record(slot->stop);
    }
    // Under stream capture the record becomes an event-record node of the
    // graph, so every replay re-times the launch.
    void record(cudaEvent_t e) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(st, &cs);
        if (cs == cudaStreamCaptureStatusActive)
            cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
        else
            cudaEventRecord(e, st);
    }
};

}  // namespace

const DeviceCtx* device_ctx() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_ctx_mu);
    DeviceCtx& c = g_ctx[dev];
    if (c.device < 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
        c.num_sms = sms;
        c.err_word = static_cast<unsigned int*>(p);
        c.device = dev;
    }
    return &c;
}

namespace {

// ------------------------------------------------------------ split sizing
// Split a contracting dimension of tp shards (k_shard each) into sub chunks per
// shard so that units * tp * sub work items fill the machine in whole waves.
KSplit choose_split(int64_t units, int64_t k_shard, int tp, int64_t min_chunk, int64_t granule) {
    KSplit ks;
    ks.tp = tp;
    ks.k_shard = k_shard;
    int best_sub = 1;
    double best = 1e30;
    const int64_t max_sub = std::max<int64_t>(1, std::min<int64_t>(32, k_shard / std::max<int64_t>(min_chunk, 1)));
    for (int64_t sub = 1; sub <= max_sub; ++sub) {
        const int64_t items = units * tp * sub;
        const int64_t waves = (items + kDesignSMs - 1) / kDesignSMs;
        // cost: idle fraction of the last wave, plus a mild penalty per extra split
        const double eff = (double)items / (double)(waves * kDesignSMs);
        const double cost = (1.0 - eff) + 0.01 * (double)sub;
        if (cost < best - 1e-9) { best = cost; best_sub = (int)sub; }
    }
    ks.sub = best_sub;
    int64_t chunk = (k_shard + best_sub - 1) / best_sub;
    chunk = (chunk + granule - 1) / granule * granule;
    ks.k_chunk = chunk;
    ks.sub = (int)((k_shard + chunk - 1) / chunk);
    return ks;
}

KSplit whole(int64_t K) { KSplit ks; ks.tp = 1; ks.sub = 1; ks.k_shard = K; ks.k_chunk = K; return ks; }

enum Path { PATH_SIMT, PATH_TC_SWAP, PATH_TC };
Path pick_path(int dt, int64_t tokens) {
    if (dt != TPL_BF16 || tokens <= kSimtMaxTokensBf16) return PATH_SIMT;
    return tokens <= 128 ? PATH_TC_SWAP : PATH_TC;
}

// Tensor-core splits move whole 64-element K blocks: every split boundary
// must fall on a multiple of 64 (one split may end on the K tail instead).
bool tc_split_ok(const KSplit& ks) {
    return ks.tp * ks.sub == 1 || (ks.k_shard % 64 == 0 && ks.k_chunk % 64 == 0);
}

// The split used for a row-parallel projection with `out_features` outputs.
KSplit rowpar_split(int dt, int64_t tokens, int64_t out_features, int64_t K, int tp) {
    Path p = pick_path(dt, tokens);
    const int64_t k_shard = K / tp;
    if (p != PATH_SIMT && k_shard % 64 != 0) p = PATH_SIMT;   // project() then runs the CUDA-core kernel
    if (p == PATH_SIMT) {
        const int64_t blocks = (out_features + 31) / 32;   // row-dot: 32 features per block
        return choose_split(std::max<int64_t>(1, blocks / 4), k_shard, tp, 512, dt == TPL_BF16 ? 8 : 4);
    }
    if (p == PATH_TC_SWAP) {
        const int64_t mt = (out_features + 127) / 128;
        return choose_split(mt, k_shard, tp, 256, 64);
    }
    KSplit ks;   // prefill: one split per shard
    ks.tp = tp; ks.sub = 1; ks.k_shard = k_shard; ks.k_chunk = k_shard;
    return ks;
}

// ------------------------------------------------ generic projection launch
// out(tokens x features) = X[tokens, K] . W[features, K]^T with the given
// epilogue; W1 is the second weight for SwiGLU.  Chooses the kernel by tokens.
cudaError_t project(const char* tag, int dt, const void* X, int64_t ldx, int64_t tokens, const void* W,
                    const void* W1, int64_t ldw, int64_t features, int64_t K, const KSplit& ks, const Epilogue& epi,
                    cudaStream_t st, float* tail_ws = nullptr, size_t tail_ws_bytes = 0) {
    Path p = pick_path(dt, tokens);
    if (p != PATH_SIMT && !tc_split_ok(ks)) p = PATH_SIMT;
    if (p == PATH_SIMT) {
        RowdotArgs a{};
        a.ldx = ldx;
        a.W = W;
        a.W1 = W1;
        a.ldw = ldw;
        a.N = features;
        a.K = K;
        a.ks = ks;
        a.epi = epi;
        for (int64_t t0 = 0; t0 < tokens; t0 += kSimtMaxTokens) {
            a.X = static_cast<const char*>(X) + t0 * ldx * esize(dt);
            a.nb = (int)std::min<int64_t>(kSimtMaxTokens, tokens - t0);
            a.tok0 = t0;
            ProfScope prof(tag, st);
            cudaError_t e = launch_rowdot(a, dt == TPL_BF16, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    TcGemmArgs g{};
    g.K = K;
    g.ks = ks;
    g.epi = epi;
    g.tail_ws = tail_ws;
    g.tail_ws_bytes = tail_ws_bytes;
    if (p == PATH_TC_SWAP) {
        g.swap = true;
        g.A = W; g.A2 = W1; g.lda = ldw; g.M = features;
        g.B = X; g.B2 = nullptr; g.ldb = ldx; g.N = tokens;
    } else {
        g.swap = false;
        g.A = X; g.A2 = nullptr; g.lda = ldx; g.M = tokens;
        g.B = W; g.B2 = W1; g.ldb = ldw; g.N = features;
    }
    ProfScope prof(tag, st);
    return launch_tc_gemm(g, st);
}

Epilogue epi_store(void* out, int bf16, int64_t ldo) {
    Epilogue e{};
    e.mode = EPI_STORE; e.out = out; e.out_bf16 = bf16; e.ldo = ldo;
    return e;
}
// rowacc (optional): the consuming row-normalising reduction's tickets ([rows]
// words at its start), zeroed by this launch.
Epilogue epi_partial(float* out32, int64_t ldo, int64_t split_stride, unsigned int* rowacc = nullptr,
                     int64_t rows = 0) {
    Epilogue e{};
    e.mode = EPI_PARTIAL; e.out32 = out32; e.ldo = ldo; e.split_stride = split_stride;
    e.zero_words = rowacc;
    e.zero_count = rowacc ? (int)rows : 0;
    return e;
}

// ------------------------------------------------------ MLP workspace plan
struct MlpPlan {
    KSplit ks;
    bool fused_tc;        // prefill with no partials requested: one split, TMEM holds the sum
    size_t h_off, part_off, total;
};
MlpPlan plan_mlp(int64_t B, int64_t D, int64_t F, int tp, int dt, bool want_partials) {
    MlpPlan p{};
    const Path path = pick_path(dt, B);
    p.fused_tc = (path == PATH_TC) && !want_partials;
    p.ks = p.fused_tc ? whole(F) : rowpar_split(dt, B, D, F, tp);
    p.h_off = 0;
    p.part_off = up((size_t)B * F * esize(dt));
    size_t part = up((size_t)B * D * 4);   // fused: one fp32 plane when a residual is added
    if (!p.fused_tc) {
        // tc prefill writes the user's partials directly (one split per shard)
        const bool direct = (path == PATH_TC) && want_partials && p.ks.sub == 1 && tc_split_ok(p.ks);
        part = direct ? 0 : up((size_t)p.ks.tp * p.ks.sub * B * D * 4);
    }
    p.total = p.part_off + part;
    return p;
}
size_t mlp_ws_bytes(int64_t B, int64_t D, int64_t F, int tp, int dt) {
    return std::max(plan_mlp(B, D, F, tp, dt, true).total, plan_mlp(B, D, F, tp, dt, false).total);
}

}  // namespace

size_t mlp_plan_bytes(int64_t B, int64_t D, int64_t F, int tp, int dt, bool want_partials) {
    return plan_mlp(B, D, F, tp, dt, want_partials).total;
}
bool mlp_out_dtype_ok(int dt, int out_dt) { return out_dtype_ok(dt, out_dt); }

namespace {

tpl_status check_mlp_shape(int64_t B, int64_t D, int64_t F, int tp, int dt) {
    if (dt != TPL_F32 && dt != TPL_BF16) return TPL_ERR_DTYPE;
    if (B <= 0 || D <= 0 || F <= 0 || tp <= 0) return TPL_ERR_SHAPE;
    if (F % tp != 0) return TPL_ERR_SHAPE;
    const int64_t vec = 16 / (int64_t)esize(dt);
    if (D % vec != 0 || F % vec != 0 || (F / tp) % vec != 0) return TPL_ERR_ALIGN;
    return TPL_OK;
}

// Reduce split partials into y (+residual); optionally emit per-shard partials.
cudaError_t reduce_into(const float* ws, int64_t rows, int64_t cols, const KSplit& ks, float* shard_out,
                        void* y, int y_bf16, int mode, const void* residual, float* scale_out, unsigned int* rowacc,
                        cudaStream_t st) {
    ReduceArgs r{};
    r.ws = ws;
    r.rows = rows;
    r.cols = cols;
    r.tp = ks.tp;
    r.sub = ks.sub;
    r.shard_out = shard_out;
    r.y = y;
    r.y_bf16 = y_bf16;
    r.mode = mode;
    r.residual = residual;
    r.scale_out = scale_out;
    r.eps = kRmsEpsilon;
    r.ws_up = nullptr;
    r.row_cnt = rowacc;
    r.row_slots = rowacc ? reinterpret_cast<float*>(rowacc + rows) : nullptr;
    ProfScope prof(scale_out ? "reduce_norm" : "reduce", st);
    return launch_reduce(r, st);
}

// MLP body shared by tp_mlp_forward and the decoder layer.  Decoder layer
// only: row_scale (the input's RMSNorm scales, applied to the gate/up
// products), residual (added to the reduced sum) and scale_out (the output's
// RMSNorm scales).
cudaError_t run_mlp(const void* X, const void* Wg, const void* Wu, const void* Wd, void* Y, float* partials,
                    int64_t B, int64_t D, int64_t F, int tp, int dt, int out_dt, char* ws, const float* row_scale,
                    const void* residual, float* scale_out, unsigned int* rowacc, cudaStream_t st) {
    const MlpPlan p = plan_mlp(B, D, F, tp, dt, partials != nullptr);
    void* H = ws + p.h_off;
    const int bf = dt == TPL_BF16;
    const int ybf = out_dt == TPL_BF16;
    Epilogue e{};
    e.mode = EPI_SWIGLU; e.out = H; e.out_bf16 = bf; e.ldo = F;
    e.row_scale = row_scale;
    cudaError_t err = project("gateup", dt, X, D, B, Wg, Wu, D, F, D, whole(D), e, st);
    if (err != cudaSuccess) return err;
    const Path path = pick_path(dt, B);
    if (p.fused_tc) {
        // Shard partials accumulate in TMEM in ascending shard order (the K
        // blocks of shard 0 first): the reduction happens inside the GEMM.
        if (!residual && !scale_out)
            return project("down", dt, H, F, B, Wd, nullptr, F, D, F, whole(F), epi_store(Y, ybf, D), st);
        // decoder layer: the fused sum goes through one fp32 plane so the
        // residual add and the next RMSNorm can follow
        float* sum = reinterpret_cast<float*>(ws + p.part_off);
        err = project("down", dt, H, F, B, Wd, nullptr, F, D, F, whole(F), epi_partial(sum, D, B * D, rowacc, B), st);
        if (err != cudaSuccess) return err;
        return reduce_into(sum, B, D, whole(D), nullptr, Y, ybf, TPL_ALLREDUCE, residual, scale_out, rowacc, st);
    }
    if (path == PATH_TC && partials && p.ks.sub == 1 && tc_split_ok(p.ks)) {
        err = project("down", dt, H, F, B, Wd, nullptr, F, D, F, p.ks, epi_partial(partials, D, B * D, rowacc, B),
                      st);
        if (err != cudaSuccess) return err;
        KSplit one = p.ks;
        one.sub = 1;
        return reduce_into(partials, B, D, one, nullptr, Y, ybf, TPL_ALLREDUCE, residual, scale_out, rowacc, st);
    }
    float* part = reinterpret_cast<float*>(ws + p.part_off);
    err = project("down", dt, H, F, B, Wd, nullptr, F, D, F, p.ks, epi_partial(part, D, B * D, rowacc, B), st);
    if (err != cudaSuccess) return err;
    return reduce_into(part, B, D, p.ks, partials, Y, ybf, TPL_ALLREDUCE, residual, scale_out, rowacc, st);
}

// ------------------------------------------------- attention projections
struct AttnPlan {
    int nq_s, kv_s;
    int64_t w_s, nqkv;
    KSplit ks;
    size_t qkv_off, o_off, part_off, total;
};
tpl_status check_attn_shape(int64_t B, int64_t D, int n_q, int n_kv, int hd, int tp, int dt) {
    if (dt != TPL_F32 && dt != TPL_BF16) return TPL_ERR_DTYPE;
    if (B <= 0 || D <= 0 || n_q <= 0 || n_kv <= 0 || hd <= 0 || tp <= 0) return TPL_ERR_SHAPE;
    if (n_q % tp != 0 || n_q % n_kv != 0) return TPL_ERR_SHAPE;
    if (tp <= n_kv ? (n_kv % tp != 0) : (tp % n_kv != 0)) return TPL_ERR_SHAPE;
    const int64_t vec = 16 / (int64_t)esize(dt);
    if (D % vec != 0 || hd % vec != 0) return TPL_ERR_ALIGN;
    return TPL_OK;
}
AttnPlan plan_attn(int64_t B, int64_t D, int n_q, int n_kv, int hd, int tp, int dt) {
    AttnPlan p{};
    p.nq_s = n_q / tp;
    p.kv_s = tp <= n_kv ? n_kv / tp : 1;
    p.w_s = (int64_t)(p.nq_s + 2 * p.kv_s) * hd;
    p.nqkv = (int64_t)(n_q + 2 * n_kv) * hd;
    const int64_t K = (int64_t)n_q * hd;
    p.ks = rowpar_split(dt, B, D, K, tp);
    const Path path = pick_path(dt, B);
    if (path == PATH_TC) { p.ks.sub = 1; p.ks.k_chunk = p.ks.k_shard; }
    const size_t es = esize(dt);
    p.qkv_off = 0;
    p.o_off = up((size_t)tp * B * p.w_s * es);
    p.part_off = p.o_off + up((size_t)B * K * es);
    p.total = p.part_off + up((size_t)p.ks.tp * p.ks.sub * B * D * 4);
    return p;
}

// Decoder-layer arguments as in run_mlp (row_scale applies to the QKV products).
cudaError_t run_attn(const void* X, const void* Wqkv, const void* Wo, void* qkv_out, void* Y, float* partials,
                     int64_t B, int64_t D, int n_q, int n_kv, int hd, int tp, int dt, int out_dt, char* ws,
                     const float* row_scale, const void* residual, float* scale_out, unsigned int* rowacc,
                     cudaStream_t st) {
    const AttnPlan p = plan_attn(B, D, n_q, n_kv, hd, tp, dt);
    const int bf = dt == TPL_BF16;
    void* qkv = qkv_out ? qkv_out : ws + p.qkv_off;
    void* O = ws + p.o_off;
    Epilogue e{};
    e.mode = EPI_QKV;
    e.out_bf16 = bf;
    e.qkv.n_q = n_q; e.qkv.n_kv = n_kv; e.qkv.head_dim = hd; e.qkv.tp = tp;
    e.qkv.nq_s = p.nq_s; e.qkv.kv_s = p.kv_s;
    e.qkv.w_s = p.w_s; e.qkv.shard_stride = B * p.w_s;
    e.qkv.qkv_out = qkv; e.qkv.o_out = O; e.qkv.ldo_o = (int64_t)n_q * hd;
    e.row_scale = row_scale;
    cudaError_t err = project("qkv", dt, X, D, B, Wqkv, nullptr, D, p.nqkv, D, whole(D), e, st);
    if (err != cudaSuccess) return err;
    const int64_t K = (int64_t)n_q * hd;
    float* part = reinterpret_cast<float*>(ws + p.part_off);
    err = project("oproj", dt, O, K, B, Wo, nullptr, K, D, K, p.ks, epi_partial(part, D, B * D, rowacc, B), st);
    if (err != cudaSuccess) return err;
    return reduce_into(part, B, D, p.ks, partials, Y, out_dt == TPL_BF16, TPL_ALLREDUCE, residual, scale_out,
                       rowacc, st);
}

// ------------------------------------------------------- decoder layer
struct LayerPlan {
    size_t sx_off, h_off, sh_off, acc_off, attn_off, mlp_off, total;
};
LayerPlan plan_layer(int64_t B, int64_t D, int64_t F, int n_q, int n_kv, int hd, int tp) {
    LayerPlan p{};
    const size_t act = up((size_t)B * D * 2);
    const size_t scl = up((size_t)B * 4);
    p.sx_off = 0;                                   // RMSNorm scales of the layer input
    p.h_off = scl;
    p.sh_off = scl + act;                           // RMSNorm scales of h
    p.acc_off = 2 * scl + act;                      // row accumulators of the norm reductions
    p.attn_off = p.acc_off + up(rowacc_bytes(B, D));
    const size_t attn = plan_attn(B, D, n_q, n_kv, hd, tp, TPL_BF16).total;
    p.mlp_off = p.attn_off + up(attn);
    p.total = p.mlp_off + up(plan_mlp(B, D, F, tp, TPL_BF16, false).total);
    return p;
}

cudaError_t run_layer(const void* x, void* y, const void* Wqkv, const void* Wo, const void* Wg, const void* Wu,
                      const void* Wd, int64_t B, int64_t D, int64_t F, int n_q, int n_kv, int hd, int tp,
                      char* ws, bool x_scale_ready, cudaStream_t st) {
    const LayerPlan p = plan_layer(B, D, F, n_q, n_kv, hd, tp);
    float* sx = reinterpret_cast<float*>(ws + p.sx_off);
    void* h = ws + p.h_off;
    float* sh = reinterpret_cast<float*>(ws + p.sh_off);
    unsigned int* rowacc = reinterpret_cast<unsigned int*>(ws + p.acc_off);
    cudaError_t err;
    if (!x_scale_ready) {
        ProfScope prof("rmsnorm", st);
        err = launch_rmsnorm(x, sx, B, D, kRmsEpsilon, rowacc, st);
        if (err != cudaSuccess) return err;
    }
    // attention sublayer on RMSNorm(x) = diag(sx) x: h = x + sum_s P_s, and h's scales
    err = run_attn(x, Wqkv, Wo, nullptr, h, nullptr, B, D, n_q, n_kv, hd, tp, TPL_BF16, TPL_BF16, ws + p.attn_off, sx,
                   x, sh, rowacc, st);
    if (err != cudaSuccess) return err;
    // MLP sublayer on RMSNorm(h): y = h + sum_s P_s, and y's scales (the next layer's sx)
    return run_mlp(h, Wg, Wu, Wd, y, nullptr, B, D, F, tp, TPL_BF16, TPL_BF16, ws + p.mlp_off, sh, h, sx, rowacc, st);
}

}  // namespace
}  // namespace tpl

using namespace tpl;

// ======================================================================= ABI

extern "C" const char* tpl_status_string(int s) {
    switch (s) {
    case TPL_OK: return "ok";
    case TPL_ERR_NULL: return "null pointer";
    case TPL_ERR_SHAPE: return "invalid shape (non-positive or not divisible by the shard count)";
    case TPL_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case TPL_ERR_DTYPE: return "unsupported dtype";
    case TPL_ERR_WORKSPACE: return "workspace missing or too small";
    case TPL_ERR_UNSUPPORTED: return "unsupported argument combination";
    case TPL_ERR_CUDA: return "CUDA runtime error";
    case TPL_ERR_TIMEOUT: return "device-side wait timed out";
    case TPL_ERR_ALIAS: return "output overlaps an input";
    case TPL_ERR_STATIC_LIMIT: return "problem needs more scratch than the library's static device area holds";
    default: return "unknown status";
    }
}

extern "C" int tpl_version(void) { return (1 << 16) | 0; }

extern "C" tpl_status tpl_device_status(unsigned int* flags, void* stream) {
    if (!flags) return TPL_ERR_NULL;
    if (!device_ctx()) return TPL_ERR_CUDA;
    if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return TPL_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof(v)) != cudaSuccess) return TPL_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero)) != cudaSuccess) return TPL_ERR_CUDA;
    *flags = v;
    return v ? TPL_ERR_TIMEOUT : TPL_OK;
}

extern "C" tpl_status tpl_shard_reduce(const float* partials, void* out, int64_t rows, int64_t cols, int tp,
                                       int mode, int out_dtype, void* stream) {
    TPL_NVTX_RANGE("tpl_shard_reduce");
    if (!partials || !out) return TPL_ERR_NULL;
    if (out_dtype != TPL_F32 && out_dtype != TPL_BF16) return TPL_ERR_DTYPE;
    if (rows <= 0 || cols <= 0 || tp <= 0) return TPL_ERR_SHAPE;
    if (mode != TPL_ALLREDUCE && mode != TPL_REDUCE_SCATTER) return TPL_ERR_UNSUPPORTED;
    if (mode == TPL_REDUCE_SCATTER && cols % tp != 0) return TPL_ERR_SHAPE;
    const int64_t out_cols = mode == TPL_REDUCE_SCATTER ? cols / tp : cols;
    if (!al16(partials) || !al16(out) || cols % 4 != 0 || (out_cols * (int64_t)esize(out_dtype)) % 16 != 0)
        return TPL_ERR_ALIGN;
    if (overlap(partials, (size_t)tp * rows * cols * 4, out, (size_t)rows * cols * esize(out_dtype)))
        return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    KSplit ks = whole(cols);
    ks.tp = tp;
    return cuda_status(reduce_into(partials, rows, cols, ks, nullptr, out, out_dtype == TPL_BF16, mode, nullptr,
                                   nullptr, nullptr, S(stream)));
}

extern "C" tpl_status tpl_tp_mlp_forward_workspace(int64_t B, int64_t D, int64_t F, int tp, int dtype,
                                                   size_t* bytes) {
    if (!bytes) return TPL_ERR_NULL;
    tpl_status s = check_mlp_shape(B, D, F, tp, dtype);
    if (s != TPL_OK) return s;
    *bytes = mlp_ws_bytes(B, D, F, tp, dtype);
    return TPL_OK;
}

extern "C" tpl_status tpl_tp_mlp_forward(const void* X, const void* Wg, const void* Wu, const void* Wd, void* Y,
                                         float* partials, int64_t B, int64_t D, int64_t F, int tp, int dtype,
                                         int out_dtype, void* ws, size_t ws_bytes, void* stream) {
    TPL_NVTX_RANGE("tpl_tp_mlp_forward");
    if (!X || !Wg || !Wu || !Wd || !Y) return TPL_ERR_NULL;
    tpl_status s = check_mlp_shape(B, D, F, tp, dtype);
    if (s != TPL_OK) return s;
    if (!out_dtype_ok(dtype, out_dtype)) return TPL_ERR_DTYPE;
    if (!al16(X) || !al16(Wg) || !al16(Wu) || !al16(Wd) || !al16(Y) || (partials && !al16(partials)) ||
        (ws && !al16(ws)))
        return TPL_ERR_ALIGN;
    const size_t es = esize(dtype);
    const size_t ybytes = (size_t)B * D * esize(out_dtype);
    if (overlap(Y, ybytes, X, (size_t)B * D * es) || overlap(Y, ybytes, Wg, (size_t)F * D * es) ||
        overlap(Y, ybytes, Wu, (size_t)F * D * es) || overlap(Y, ybytes, Wd, (size_t)F * D * es) ||
        (partials && overlap(partials, (size_t)tp * B * D * 4, Y, ybytes)) ||
        (partials && overlap(partials, (size_t)tp * B * D * 4, X, (size_t)B * D * es)))
        return TPL_ERR_ALIAS;
    const size_t need = plan_mlp(B, D, F, tp, dtype, partials != nullptr).total;
    if (!ws || ws_bytes < need) return TPL_ERR_WORKSPACE;
    if (overlap(ws, need, X, (size_t)B * D * es) || overlap(ws, need, Y, ybytes)) return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    return cuda_status(run_mlp(X, Wg, Wu, Wd, Y, partials, B, D, F, tp, dtype, out_dtype, static_cast<char*>(ws),
                               nullptr, nullptr, nullptr, nullptr, S(stream)));
}

extern "C" tpl_status tpl_tp_attn_proj_workspace(int64_t B, int64_t D, int n_q, int n_kv, int head_dim, int tp,
                                                 int dtype, size_t* bytes) {
    if (!bytes) return TPL_ERR_NULL;
    tpl_status s = check_attn_shape(B, D, n_q, n_kv, head_dim, tp, dtype);
    if (s != TPL_OK) return s;
    *bytes = plan_attn(B, D, n_q, n_kv, head_dim, tp, dtype).total;
    return TPL_OK;
}

extern "C" tpl_status tpl_tp_attn_proj(const void* X, const void* Wqkv, const void* Wo, void* qkv_out, void* Y,
                                       float* partials, int64_t B, int64_t D, int n_q, int n_kv, int head_dim,
                                       int tp, int dtype, int out_dtype, void* ws, size_t ws_bytes, void* stream) {
    TPL_NVTX_RANGE("tpl_tp_attn_proj");
    if (!X || !Wqkv || !Wo || !Y) return TPL_ERR_NULL;
    tpl_status s = check_attn_shape(B, D, n_q, n_kv, head_dim, tp, dtype);
    if (s != TPL_OK) return s;
    if (!out_dtype_ok(dtype, out_dtype)) return TPL_ERR_DTYPE;
    if (!al16(X) || !al16(Wqkv) || !al16(Wo) || !al16(Y) || (qkv_out && !al16(qkv_out)) ||
        (partials && !al16(partials)) || (ws && !al16(ws)))
        return TPL_ERR_ALIGN;
    const AttnPlan p = plan_attn(B, D, n_q, n_kv, head_dim, tp, dtype);
    const size_t es = esize(dtype);
    const size_t ybytes = (size_t)B * D * esize(out_dtype);
    const size_t qkv_bytes = (size_t)tp * B * p.w_s * es;
    if (overlap(Y, ybytes, X, (size_t)B * D * es) || overlap(Y, ybytes, Wqkv, (size_t)p.nqkv * D * es) ||
        overlap(Y, ybytes, Wo, (size_t)D * n_q * head_dim * es) ||
        (qkv_out && (overlap(qkv_out, qkv_bytes, X, (size_t)B * D * es) || overlap(qkv_out, qkv_bytes, Y, ybytes))) ||
        (partials && overlap(partials, (size_t)tp * B * D * 4, Y, ybytes)))
        return TPL_ERR_ALIAS;
    if (!ws || ws_bytes < p.total) return TPL_ERR_WORKSPACE;
    if (overlap(ws, p.total, X, (size_t)B * D * es) || overlap(ws, p.total, Y, ybytes)) return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    return cuda_status(run_attn(X, Wqkv, Wo, qkv_out, Y, partials, B, D, n_q, n_kv, head_dim, tp, dtype, out_dtype,
                                static_cast<char*>(ws), nullptr, nullptr, nullptr, nullptr, S(stream)));
}

// ------------------------------------------------------------ four cases
namespace tpl {
namespace {
struct CasePlan { KSplit ks; bool partial_path; size_t total; };
CasePlan plan_case(int case_id, int64_t I, int64_t J, int64_t K, int X, int dt, bool want_partials) {
    CasePlan c{};
    c.ks = whole(J);
    c.partial_path = false;
    // the direct GEMM's split last wave (the same shape rule the launch applies)
    c.total = pick_path(dt, I) == PATH_TC ? up(tc_tail_ws_bytes(I, K, J, kDesignSMs)) : 0;
    if (case_id == 3) {
        const Path path = pick_path(dt, I);
        if (want_partials || path != PATH_TC) {
            c.partial_path = true;
            c.total = 0;
            if (want_partials && path == PATH_TC && (J / X) % 64 == 0) {
                c.ks.tp = X; c.ks.sub = 1; c.ks.k_shard = J / X; c.ks.k_chunk = J / X;
            } else {
                c.ks = rowpar_split(dt, I, K, J, X);
                c.total = up((size_t)c.ks.tp * c.ks.sub * I * K * 4);
            }
        }
    }
    return c;
}
tpl_status check_case(int case_id, int mode, int gather, int64_t I, int64_t J, int64_t K, int X, int dt) {
    if (dt != TPL_F32 && dt != TPL_BF16) return TPL_ERR_DTYPE;
    if (case_id < 1 || case_id > 4) return TPL_ERR_UNSUPPORTED;
    if (mode != TPL_ALLREDUCE && mode != TPL_REDUCE_SCATTER) return TPL_ERR_UNSUPPORTED;
    if (gather != TPL_GATHER_A && gather != TPL_GATHER_B) return TPL_ERR_UNSUPPORTED;
    if (I <= 0 || J <= 0 || K <= 0 || X <= 0) return TPL_ERR_SHAPE;
    const int64_t vec = 16 / (int64_t)esize(dt);
    if (J % vec != 0 || K % vec != 0) return TPL_ERR_ALIGN;
    switch (case_id) {
    case 1: if (I % X) return TPL_ERR_SHAPE; break;
    case 2: if (J % X) return TPL_ERR_SHAPE; break;
    case 3:
        if (J % X) return TPL_ERR_SHAPE;
        if ((J / X) % vec) return TPL_ERR_ALIGN;
        if (mode == TPL_REDUCE_SCATTER && (K % X || ((K / X) % vec))) return TPL_ERR_SHAPE;
        break;
    case 4:
        if (I % X || K % X) return TPL_ERR_SHAPE;
        if (gather == TPL_GATHER_A && (K / X) % vec) return TPL_ERR_ALIGN;
        break;
    }
    return TPL_OK;
}
}  // namespace
}  // namespace tpl

extern "C" tpl_status tpl_sharded_matmul_workspace(int case_id, int mode, int64_t I, int64_t J, int64_t K, int X,
                                                   int dtype, size_t* bytes) {
    if (!bytes) return TPL_ERR_NULL;
    tpl_status s = check_case(case_id, mode, TPL_GATHER_B, I, J, K, X, dtype);
    if (s != TPL_OK) return s;
    *bytes = std::max(plan_case(case_id, I, J, K, X, dtype, true).total,
                      plan_case(case_id, I, J, K, X, dtype, false).total);
    return TPL_OK;
}

extern "C" tpl_status tpl_sharded_matmul(int case_id, int mode, int gather, const void* A, const void* Bt, void* C,
                                         float* partials, int64_t I, int64_t J, int64_t K, int X, int dtype,
                                         int out_dtype, void* ws, size_t ws_bytes, void* stream) {
    TPL_NVTX_RANGE("tpl_sharded_matmul");
    if (!A || !Bt || !C) return TPL_ERR_NULL;
    tpl_status s = check_case(case_id, mode, gather, I, J, K, X, dtype);
    if (s != TPL_OK) return s;
    if (!out_dtype_ok(dtype, out_dtype)) return TPL_ERR_DTYPE;
    if ((case_id == 3 && mode == TPL_REDUCE_SCATTER) || (case_id == 4 && gather == TPL_GATHER_A)) {
        if (((K / X) * (int64_t)esize(out_dtype)) % 16 != 0) return TPL_ERR_ALIGN;
    }
    if (partials && case_id != 3) return TPL_ERR_UNSUPPORTED;
    if (!al16(A) || !al16(Bt) || !al16(C) || (partials && !al16(partials)) || (ws && !al16(ws)))
        return TPL_ERR_ALIGN;
    const size_t es = esize(dtype);
    const size_t cbytes = (size_t)I * K * esize(out_dtype);
    if (overlap(C, cbytes, A, (size_t)I * J * es) || overlap(C, cbytes, Bt, (size_t)K * J * es) ||
        (partials && (overlap(partials, (size_t)X * I * K * 4, C, cbytes) ||
                      overlap(partials, (size_t)X * I * K * 4, A, (size_t)I * J * es))))
        return TPL_ERR_ALIAS;
    const CasePlan p = plan_case(case_id, I, J, K, X, dtype, partials != nullptr);
    if (p.total > 0 && (!ws || ws_bytes < p.total)) return TPL_ERR_WORKSPACE;
    if (p.total > 0 && (overlap(ws, p.total, C, cbytes) || overlap(ws, p.total, A, (size_t)I * J * es)))
        return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    const int bf = out_dtype == TPL_BF16;
    cudaStream_t st = S(stream);
    // Output layout: C[I, K] row-major, or shard-blocked [X, I, K/X] when the
    // result is sharded along K (case 3 reduce-scatter, case 4 gather-A).
    Epilogue e = epi_store(C, bf, K);
    const bool k_sharded = (case_id == 3 && mode == TPL_REDUCE_SCATTER) || (case_id == 4 && gather == TPL_GATHER_A);
    if (k_sharded) {
        e.ldo = K / X;
        e.col_block = K / X;
        e.block_stride = I * (K / X);
    }
    cudaError_t err;
    if (case_id != 3 || !p.partial_path) {
        // cases 1, 2, 4: the gathered operand is a view of the shards already
        // resident in this GPU's memory; case 3 fused: partial sums over the J
        // shards accumulate in ascending shard order inside the GEMM.
        err = project("matmul", dtype, A, J, I, Bt, nullptr, J, K, J, whole(J), e, st, reinterpret_cast<float*>(ws),
                      ws ? ws_bytes : 0);
        return cuda_status(err);
    }
    float* part = partials;
    const bool direct = partials && pick_path(dtype, I) == PATH_TC && (J / X) % 64 == 0;
    if (!direct) part = reinterpret_cast<float*>(ws);
    err = project("matmul", dtype, A, J, I, Bt, nullptr, J, K, J, p.ks, epi_partial(part, K, I * K), st);
    if (err != cudaSuccess) return cuda_status(err);
    KSplit ks = p.ks;
    float* shard_out = direct ? nullptr : partials;
    if (direct) ks.sub = 1;
    return cuda_status(reduce_into(part, I, K, ks, shard_out, C, bf, mode, nullptr, nullptr, nullptr, st));
}

// --------------------------------------------------------------- decoder
extern "C" tpl_status tpl_tp_decoder_workspace(int64_t B, int64_t D, int64_t F, int n_q, int n_kv, int head_dim,
                                               int tp, size_t* bytes) {
    if (!bytes) return TPL_ERR_NULL;
    tpl_status s = check_mlp_shape(B, D, F, tp, TPL_BF16);
    if (s != TPL_OK) return s;
    s = check_attn_shape(B, D, n_q, n_kv, head_dim, tp, TPL_BF16);
    if (s != TPL_OK) return s;
    size_t need = plan_layer(B, D, F, n_q, n_kv, head_dim, tp).total;
    const FusedShape fs{B, D, F, n_q, n_kv, head_dim, tp};
    if (fused_stack_shape_ok(fs)) need = std::max(need, fused_stack_ws_bytes(fs));
    *bytes = need;
    return TPL_OK;
}

static tpl_status check_layer_args(const void* x, const void* y, const void* Wqkv, const void* Wo, const void* Wg,
                                   const void* Wu, const void* Wd) {
    if (!x || !y || !Wqkv || !Wo || !Wg || !Wu || !Wd) return TPL_ERR_NULL;
    if (!al16(x) || !al16(y) || !al16(Wqkv) || !al16(Wo) || !al16(Wg) || !al16(Wu) || !al16(Wd))
        return TPL_ERR_ALIGN;
    return TPL_OK;
}

extern "C" tpl_status tpl_tp_decoder_stack_ex(const void* x, void* y, const void* const* Wqkv,
                                              const void* const* Wo, const void* const* Wg, const void* const* Wu,
                                              const void* const* Wd, int n_layers, int64_t B, int64_t D, int64_t F,
                                              int n_q, int n_kv, int head_dim, int tp, void* ws, size_t ws_bytes,
                                              int path, int block, void* stream) {
    TPL_NVTX_RANGE("tpl_tp_decoder_stack_ex");
    if (!Wqkv || !Wo || !Wg || !Wu || !Wd || !ws) return TPL_ERR_NULL;
    if (path != TPL_PATH_AUTO && path != TPL_PATH_UNFUSED && path != TPL_PATH_FUSED) return TPL_ERR_UNSUPPORTED;
    if (block != TPL_BLOCK_SERIAL && block != TPL_BLOCK_PARALLEL) return TPL_ERR_UNSUPPORTED;
    if (block == TPL_BLOCK_PARALLEL && path == TPL_PATH_UNFUSED) return TPL_ERR_UNSUPPORTED;
    if (n_layers <= 0) return TPL_ERR_SHAPE;
    size_t need = 0;
    tpl_status s = tpl_tp_decoder_workspace(B, D, F, n_q, n_kv, head_dim, tp, &need);
    if (s != TPL_OK) return s;
    if (ws_bytes < need) return TPL_ERR_WORKSPACE;
    if (!al16(ws)) return TPL_ERR_ALIGN;
    for (int l = 0; l < n_layers; ++l) {
        s = check_layer_args(x, y, Wqkv[l], Wo[l], Wg[l], Wu[l], Wd[l]);
        if (s != TPL_OK) return s;
    }
    const size_t act = (size_t)B * D * 2;
    if (overlap(ws, need, x, act) || overlap(ws, need, y, act)) return TPL_ERR_ALIAS;
    if (x != y && overlap(x, act, y, act)) return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    cudaStream_t st = S(stream);
    const FusedShape fs{B, D, F, n_q, n_kv, head_dim, tp};
    const bool fused_ok = fused_stack_shape_ok(fs) && tc_gemm_supported();
    if ((path == TPL_PATH_FUSED || block == TPL_BLOCK_PARALLEL) && !fused_ok) return TPL_ERR_UNSUPPORTED;
    if (path != TPL_PATH_UNFUSED && fused_ok) {
        ProfScope prof("fused_stack", st);
        return cuda_status(launch_fused_stack(fs, x, y, Wqkv, Wo, Wg, Wu, Wd, n_layers, block == TPL_BLOCK_PARALLEL,
                                              ws, st));
    }
    for (int l = 0; l < n_layers; ++l) {
        // every layer after the first finds the RMSNorm scales of its input
        // already produced by the previous layer's final reduction
        cudaError_t e = run_layer(l == 0 ? x : y, y, Wqkv[l], Wo[l], Wg[l], Wu[l], Wd[l], B, D, F, n_q, n_kv,
                                  head_dim, tp, static_cast<char*>(ws), l > 0, st);
        if (e != cudaSuccess) return TPL_ERR_CUDA;
    }
    return TPL_OK;
}

extern "C" tpl_status tpl_fused_trace_read(void* host, size_t bytes) {
    if (!host) return TPL_ERR_NULL;
    if (!device_ctx()) return TPL_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return TPL_ERR_CUDA;
    return fused_trace_read(host, bytes) ? TPL_OK : TPL_ERR_UNSUPPORTED;
}

extern "C" tpl_status tpl_test_fused_fault(int cta, int phase, int64_t wait_limit_ns) {
    if (wait_limit_ns > 2000000000LL) return TPL_ERR_UNSUPPORTED;
    if (wait_limit_ns > 0 && wait_limit_ns < 10000) return TPL_ERR_UNSUPPORTED;
    if (cta >= kFusedGridCap || (cta >= 0 && phase < 1)) return TPL_ERR_UNSUPPORTED;
    fused_test_fault(cta < 0 ? -1 : cta, cta < 0 ? -1 : phase, wait_limit_ns);
    return TPL_OK;
}

extern "C" tpl_status tpl_tp_decoder_stack_path(const void* x, void* y, const void* const* Wqkv,
                                                const void* const* Wo, const void* const* Wg, const void* const* Wu,
                                                const void* const* Wd, int n_layers, int64_t B, int64_t D, int64_t F,
                                                int n_q, int n_kv, int head_dim, int tp, void* ws, size_t ws_bytes,
                                                int path, void* stream) {
    return tpl_tp_decoder_stack_ex(x, y, Wqkv, Wo, Wg, Wu, Wd, n_layers, B, D, F, n_q, n_kv, head_dim, tp, ws,
                                   ws_bytes, path, TPL_BLOCK_SERIAL, stream);
}

extern "C" tpl_status tpl_tp_decoder_stack(const void* x, void* y, const void* const* Wqkv, const void* const* Wo,
                                           const void* const* Wg, const void* const* Wu, const void* const* Wd,
                                           int n_layers, int64_t B, int64_t D, int64_t F, int n_q, int n_kv,
                                           int head_dim, int tp, void* ws, size_t ws_bytes, void* stream) {
    return tpl_tp_decoder_stack_path(x, y, Wqkv, Wo, Wg, Wu, Wd, n_layers, B, D, F, n_q, n_kv, head_dim, tp, ws,
                                     ws_bytes, TPL_PATH_AUTO, stream);
}

extern "C" tpl_status tpl_tp_decoder_layer(const void* x, void* y, const void* Wqkv, const void* Wo, const void* Wg,
                                           const void* Wu, const void* Wd, int64_t B, int64_t D, int64_t F, int n_q,
                                           int n_kv, int head_dim, int tp, void* ws, size_t ws_bytes, void* stream) {
    const void* q[1] = {Wqkv};
    const void* o[1] = {Wo};
    const void* g[1] = {Wg};
    const void* u[1] = {Wu};
    const void* d[1] = {Wd};
    return tpl_tp_decoder_stack(x, y, q, o, g, u, d, 1, B, D, F, n_q, n_kv, head_dim, tp, ws, ws_bytes, stream);
}

// ------------------------------------------------- weight-only int8 MLP

namespace {
struct W8Plan {
    bool rowdot;    // few tokens: CUDA-core kernel (see launch_w8_rowdot), else tensor cores
    KSplit ks_gu;   // gate/up: K = D, one shard, split into chunks to fill the machine
    KSplit ks_d;    // down: K = F, tp shards, each split into chunks
    size_t h_off, gu_off, gu2_off, part_off, total;
};
W8Plan plan_mlp_w8(int64_t B, int64_t D, int64_t F, int tp) {
    W8Plan p{};
    p.rowdot = B <= kW8RowdotMaxTokens;
    if (p.rowdot) {
        // row-dot blocks cover 16 (gate/up pairs) or 32 (down) features; about
        // four blocks share an SM
        p.ks_gu = choose_split(std::max<int64_t>(1, (F + 15) / 16 / 4), D, 1, 512, 64);
        p.ks_d = choose_split(std::max<int64_t>(1, (D + 31) / 32 / 4), F / tp, tp, 512, 64);
    } else {
        const int64_t ntok = (B + 127) / 128;
        p.ks_gu = choose_split((F + 127) / 128 * ntok, D, 1, 256, 64);
        p.ks_d = choose_split((D + 127) / 128 * ntok, F / tp, tp, 256, 64);
    }
    p.h_off = 0;
    p.gu_off = up((size_t)B * F * 2);
    const size_t gu = p.ks_gu.sub > 1 ? up((size_t)p.ks_gu.sub * B * F * 4) : 0;
    p.gu2_off = p.gu_off + gu;
    p.part_off = p.gu2_off + gu;
    p.total = p.part_off + up((size_t)p.ks_d.tp * p.ks_d.sub * B * D * 4);
    return p;
}
tpl_status check_w8_shape(int64_t B, int64_t D, int64_t F, int tp) {
    if (B <= 0 || D <= 0 || F <= 0 || tp <= 0 || F % tp != 0) return TPL_ERR_SHAPE;
    if (D % 64 != 0 || (F / tp) % 64 != 0) return TPL_ERR_SHAPE;
    return TPL_OK;
}
bool al8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
}  // namespace

extern "C" tpl_status tpl_quantize_w8(const void* W, int64_t rows, int64_t cols, int groups, int8_t* Q,
                                      float* scale, void* stream) {
    TPL_NVTX_RANGE("tpl_quantize_w8");
    if (!W || !Q || !scale) return TPL_ERR_NULL;
    if (rows <= 0 || cols <= 0 || groups <= 0 || cols % groups != 0) return TPL_ERR_SHAPE;
    if ((cols / groups) % 8 != 0) return TPL_ERR_ALIGN;
    if (!al16(W) || !al8(Q) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0) return TPL_ERR_ALIGN;
    const size_t wb = (size_t)rows * cols * 2, qb = (size_t)rows * cols, sb = (size_t)rows * groups * 4;
    if (overlap(Q, qb, W, wb) || overlap(scale, sb, W, wb) || overlap(scale, sb, Q, qb)) return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    cudaStream_t st = S(stream);
    ProfScope prof("quantize_w8", st);
    return cuda_status(launch_quantize_w8(W, rows, cols, groups, Q, scale, st));
}

extern "C" tpl_status tpl_tp_mlp_forward_w8_workspace(int64_t B, int64_t D, int64_t F, int tp, size_t* bytes) {
    if (!bytes) return TPL_ERR_NULL;
    const tpl_status s = check_w8_shape(B, D, F, tp);
    if (s != TPL_OK) return s;
    *bytes = plan_mlp_w8(B, D, F, tp).total;
    return TPL_OK;
}

extern "C" tpl_status tpl_tp_mlp_forward_w8(const void* X, const int8_t* Qg, const float* sg, const int8_t* Qu,
                                            const float* su, const int8_t* Qd, const float* sd, void* Y,
                                            float* partials, int64_t B, int64_t D, int64_t F, int tp,
                                            int out_dtype, void* ws, size_t ws_bytes, void* stream) {
    TPL_NVTX_RANGE("tpl_tp_mlp_forward_w8");
    if (!X || !Qg || !sg || !Qu || !su || !Qd || !sd || !Y) return TPL_ERR_NULL;
    tpl_status s = check_w8_shape(B, D, F, tp);
    if (s != TPL_OK) return s;
    if (out_dtype != TPL_F32 && out_dtype != TPL_BF16) return TPL_ERR_DTYPE;
    if (!al16(X) || !al16(Qg) || !al16(Qu) || !al16(Qd) || !al16(Y) || (partials && !al16(partials)) ||
        (ws && !al16(ws)))
        return TPL_ERR_ALIGN;
    const void* f4[3] = {sg, su, sd};
    for (const void* q : f4)
        if ((reinterpret_cast<uintptr_t>(q) & 3u) != 0) return TPL_ERR_ALIGN;
    const W8Plan p = plan_mlp_w8(B, D, F, tp);
    if (!ws || ws_bytes < p.total) return TPL_ERR_WORKSPACE;
    const size_t ybytes = (size_t)B * D * esize(out_dtype), wq = (size_t)F * D, xb = (size_t)B * D * 2;
    const size_t pb = (size_t)tp * B * D * 4;
    const void* ins[7] = {X, Qg, Qu, Qd, sg, su, sd};
    const size_t insz[7] = {xb, wq, wq, wq, (size_t)F * 4, (size_t)F * 4, (size_t)D * tp * 4};
    for (int i = 0; i < 7; ++i) {
        if (overlap(Y, ybytes, ins[i], insz[i]) || overlap(ws, p.total, ins[i], insz[i])) return TPL_ERR_ALIAS;
        if (partials && overlap(partials, pb, ins[i], insz[i])) return TPL_ERR_ALIAS;
    }
    if (overlap(Y, ybytes, ws, p.total) || (partials && (overlap(partials, pb, ws, p.total) ||
                                                         overlap(partials, pb, Y, ybytes))))
        return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    if (!tc_gemm_supported()) return TPL_ERR_UNSUPPORTED;
    cudaStream_t st = S(stream);
    char* w = static_cast<char*>(ws);
    void* H = w + p.h_off;

    W8GemmArgs g{};
    g.Q = Qg; g.Q2 = Qu; g.scale = sg; g.scale2 = su; g.groups = 1;
    g.M = F; g.X = X; g.ldx = D; g.N = B; g.K = D; g.ks = p.ks_gu;
    float* gp = reinterpret_cast<float*>(w + p.gu_off);
    float* up_p = reinterpret_cast<float*>(w + p.gu2_off);
    if (p.ks_gu.sub == 1) {
        g.epi.mode = EPI_SWIGLU; g.epi.out = H; g.epi.out_bf16 = 1; g.epi.ldo = F;
    } else {
        g.epi.mode = EPI_PARTIAL2; g.epi.out32 = gp; g.epi.out32b = up_p; g.epi.ldo = F;
        g.epi.split_stride = B * F;
    }
    auto gemm = p.rowdot ? launch_w8_rowdot : launch_w8_gemm;
    {
        ProfScope prof("w8_gateup", st);
        if (gemm(g, st) != cudaSuccess) return TPL_ERR_CUDA;
    }
    if (p.ks_gu.sub > 1) {
        // SwiGLU of the chunk sums (chunks added in K order), stored bf16
        ReduceArgs r{};
        r.ws = gp; r.ws_up = up_p; r.rows = B; r.cols = F; r.tp = 1; r.sub = p.ks_gu.sub;
        r.y = H; r.y_bf16 = 1; r.mode = TPL_ALLREDUCE; r.eps = kRmsEpsilon;
        ProfScope prof("reduce", st);
        if (launch_reduce(r, st) != cudaSuccess) return TPL_ERR_CUDA;
    }
    W8GemmArgs d{};
    d.Q = Qd; d.scale = sd; d.groups = tp;
    d.M = D; d.X = H; d.ldx = F; d.N = B; d.K = F; d.ks = p.ks_d;
    float* part = reinterpret_cast<float*>(w + p.part_off);
    d.epi = epi_partial(part, D, B * D);
    {
        ProfScope prof("w8_down", st);
        if (gemm(d, st) != cudaSuccess) return TPL_ERR_CUDA;
    }
    return cuda_status(reduce_into(part, B, D, p.ks_d, partials, Y, out_dtype == TPL_BF16, TPL_ALLREDUCE, nullptr,
                                   nullptr, nullptr, st));
}

// ----------------------------------------------- vocabulary-parallel lm_head

namespace {
tpl_status check_vocab_shape(int64_t B, int64_t V, int tp, int k) {
    if (B < 1 || V < 1 || tp < 1 || V % tp != 0 || V >= (int64_t(1) << 31)) return TPL_ERR_SHAPE;
    if (k < 1 || k > kVocabTopkMax || k > V / tp) return TPL_ERR_SHAPE;
    if (B > 65535 * int64_t(1024)) return TPL_ERR_SHAPE;
    return TPL_OK;
}
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
}  // namespace

extern "C" tpl_status tpl_vocab_parallel_topk_workspace(int64_t B, int64_t V, int tp, int k, size_t* bytes) {
    if (!bytes) return TPL_ERR_NULL;
    const tpl_status s = check_vocab_shape(B, V, tp, k);
    if (s != TPL_OK) return s;
    *bytes = vocab_topk_ws_bytes(B, V, tp, k);
    return TPL_OK;
}

extern "C" tpl_status tpl_vocab_parallel_topk(const void* X, const void* W, int64_t B, int64_t D, int64_t V,
                                              int tp, int k, int dtype, int32_t* top_idx, float* top_val,
                                              int32_t* shard_idx, float* shard_val, void* ws, size_t ws_bytes,
                                              void* stream) {
    TPL_NVTX_RANGE("tpl_vocab_parallel_topk");
    if (!X || !W || !top_idx) return TPL_ERR_NULL;
    tpl_status s = check_vocab_shape(B, V, tp, k);
    if (s != TPL_OK) return s;
    if (D < 8 || D % 8 != 0) return TPL_ERR_SHAPE;
    if (dtype != TPL_BF16) return TPL_ERR_DTYPE;
    if (!al16(X) || !al16(W) || !al4(top_idx) || (top_val && !al4(top_val)) || (shard_idx && !al4(shard_idx)) ||
        (shard_val && !al4(shard_val)))
        return TPL_ERR_ALIGN;
    const size_t need = vocab_topk_ws_bytes(B, V, tp, k);
    if (!ws || ws_bytes < need) return TPL_ERR_WORKSPACE;
    if (!al16(ws)) return TPL_ERR_ALIGN;
    const size_t xb = (size_t)B * D * 2, wb = (size_t)V * D * 2;
    const size_t ob = (size_t)B * k * 4, sb = (size_t)tp * B * k * 4;
    const void* outs[4] = {top_idx, top_val, shard_idx, shard_val};
    const size_t osz[4] = {ob, ob, sb, sb};
    for (int i = 0; i < 4; ++i) {
        if (!outs[i]) continue;
        if (overlap(outs[i], osz[i], X, xb) || overlap(outs[i], osz[i], W, wb) || overlap(outs[i], osz[i], ws, need))
            return TPL_ERR_ALIAS;
        for (int j = 0; j < i; ++j)
            if (outs[j] && overlap(outs[i], osz[i], outs[j], osz[j])) return TPL_ERR_ALIAS;
    }
    if (overlap(ws, need, X, xb) || overlap(ws, need, W, wb)) return TPL_ERR_ALIAS;
    if (!device_ctx()) return TPL_ERR_CUDA;
    if (!tc_gemm_supported()) return TPL_ERR_UNSUPPORTED;
    VocabTopkArgs a{X, W, B, D, V, tp, k, top_idx, top_val, shard_idx, shard_val, ws};
    cudaStream_t st = S(stream);
    ProfScope prof("lm_head_topk", st);
    return cuda_status(launch_vocab_topk(a, st));
}

extern "C" tpl_status tpl_profile_enable(int max_launches) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (auto& p : g_prof) {
        cudaEventDestroy(p.start);
        cudaEventDestroy(p.stop);
    }
    g_prof.clear();
    g_prof_next = 0;
    g_prof_on = false;
    if (max_launches <= 0) return TPL_OK;
    if (!device_ctx()) return TPL_ERR_CUDA;
    g_prof.resize(max_launches);
    for (auto& p : g_prof) {
        p.tag = "";
        if (cudaEventCreate(&p.start) != cudaSuccess || cudaEventCreate(&p.stop) != cudaSuccess) return TPL_ERR_CUDA;
    }
    g_prof_on = true;
    return TPL_OK;
}

extern "C" int tpl_profile_count(void) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    return g_prof_next;
}

extern "C" tpl_status tpl_profile_read(int i, char* tag, size_t tag_len, float* ms) {
    if (!tag || !ms) return TPL_ERR_NULL;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (i < 0 || i >= g_prof_next) return TPL_ERR_SHAPE;
    if (cudaEventSynchronize(g_prof[i].stop) != cudaSuccess) return TPL_ERR_CUDA;
    if (cudaEventElapsedTime(ms, g_prof[i].start, g_prof[i].stop) != cudaSuccess) return TPL_ERR_CUDA;
    std::snprintf(tag, tag_len, "%s", g_prof[i].tag);
    return TPL_OK;
}
