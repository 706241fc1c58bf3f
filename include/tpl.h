/*
 * tpl.h -- Megatron-style tensor-parallel layer forward on one GPU (C ABI).
 *
 * The tensor-parallel (TP) shards are logical partitions of the weights held
 * in one GPU's memory.  What would be a cross-device all-reduce of per-shard
 * partial sums becomes an on-device partial-sum reduction.
 *
 * Sources (reference pages, by title and section):
 *   [L4] "Lecture 4 - Distributed Serving" (CS349E notes): S3.1 sharding
 *        notation A[I_X, J]; S3.2 the four sharded-matmul cases; S4.1 MLP
 *        column-then-row split; S4.2 attention split by head; S4.3 the
 *        sharded output equals the single-device output up to summation
 *        order; S4.4 KV groups when tp > n_kv.
 *   [V4] "vLLM model parallelism" article: S2.1 ColumnParallelLinear keeps its
 *        weight as [output_size_per_partition, input_size] and applies
 *        F.linear; RowParallelLinear splits along the input and all-reduces.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensor pointers are DEVICE pointers into the calling process's current
 *    CUDA device.  The caller owns all memory; the library keeps no pointer
 *    after a call returns and never allocates device memory on these paths.
 *  - Matrices are row-major.  Weights are stored [out, in] (the nn.Linear /
 *    [V4] layout): y = x W^T.  A dimension split over tp shards is split in
 *    tp contiguous blocks; shard s holds block s ([L4] S3.1).
 *  - A tensor sharded along its LAST dimension, e.g. C[I, K_X], is stored as
 *    the concatenation of the shard-local pieces: [X, I, K/X].  One sharded
 *    along its first dimension, C[I_X, K], is [I, K] row-major.
 *  - dtype TPL_BF16: activations and weights are bfloat16; products
 *    accumulate in fp32; partial sums are fp32; intermediates the next
 *    product consumes (SwiGLU output, packed QKV, attention output) are
 *    rounded to bf16.  The final output has element type out_dtype: TPL_BF16
 *    (rounded to nearest even) or TPL_F32 (the unrounded fp32 result).
 *    dtype TPL_F32: everything fp32 (CUDA-core fp32 FMA, no TF32); out_dtype
 *    must then be TPL_F32.
 *  - Every pointer must be 16-byte aligned and every row length (in bytes) a
 *    multiple of 16; otherwise TPL_ERR_ALIGN.  Outputs must not overlap
 *    inputs (TPL_ERR_ALIAS).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls only enqueue work; they are asynchronous and
 *    stream-ordered.  Arguments are validated before anything is launched: a
 *    call that returns an error has launched nothing.  Launch failures return
 *    TPL_ERR_CUDA.  Faults during execution surface at the caller's next
 *    synchronisation, like any CUDA kernel.
 *  - Kernels never spin without bound.  A device-side wait that gives up sets
 *    a sticky device error word, read and cleared with tpl_device_status().
 *  - `ws` is caller-provided scratch of at least the size the matching
 *    *_workspace() query returns (TPL_ERR_WORKSPACE otherwise).  Its contents
 *    on entry do not matter; calls sharing one `ws` must be stream-ordered.
 */
#ifndef TPL_H
#define TPL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tpl_status {
    TPL_OK = 0,
    TPL_ERR_NULL = 1,         /* a required pointer is NULL                        */
    TPL_ERR_SHAPE = 2,        /* size <= 0, or not divisible by the shard count     */
    TPL_ERR_ALIGN = 3,        /* pointer or row pitch not a multiple of 16 bytes    */
    TPL_ERR_DTYPE = 4,        /* dtype not supported by this call                   */
    TPL_ERR_WORKSPACE = 5,    /* ws NULL or smaller than the workspace query        */
    TPL_ERR_UNSUPPORTED = 6,  /* argument combination not supported (see the call)  */
    TPL_ERR_CUDA = 7,         /* the CUDA runtime reported an error                 */
    TPL_ERR_TIMEOUT = 8,      /* a device-side bounded wait gave up                 */
    TPL_ERR_ALIAS = 9,        /* an output buffer overlaps an input buffer          */
    TPL_ERR_STATIC_LIMIT = 10 /* the problem needs more scratch than the library's
                                 static device area (TPL_STATIC_WS_BYTES) holds    */
} tpl_status;

typedef enum tpl_dtype { TPL_F32 = 0, TPL_BF16 = 1 } tpl_dtype;

/* How a partial-sum reduction distributes its result ([L4] S3.2 case 3):
 * ALLREDUCE: every shard holds the full sum -> one [rows, cols] copy here.
 * REDUCE_SCATTER: shard s keeps columns [s cols/tp, (s+1) cols/tp), stored
 * shard-blocked as [tp, rows, cols/tp]. */
typedef enum tpl_reduce_mode { TPL_ALLREDUCE = 0, TPL_REDUCE_SCATTER = 1 } tpl_reduce_mode;

/* Case 4 of [L4] S3.2 needs one operand all-gathered first. */
typedef enum tpl_gather { TPL_GATHER_B = 0, TPL_GATHER_A = 1 } tpl_gather;

/* Device error word bits (tpl_device_status). */
#define TPL_DEVERR_TIMEOUT 0x1u   /* an mbarrier wait exceeded its time limit */

/* Human-readable name of a status code (static storage, never NULL). */
const char* tpl_status_string(int status);

/* Library ABI version: (major << 16) | minor. */
int tpl_version(void);

/* Reads and clears the sticky device error word after synchronising `stream`.
 * *flags receives TPL_DEVERR_* bits (0 = no device-side error). */
tpl_status tpl_device_status(unsigned int* flags, void* stream);

/* --------------------------------------------------------------------------
 * shard_reduce -- the all-reduce stand-in ([L4] S3.2 case 3, S4.1, S4.2).
 *
 * out = partials[0] + partials[1] + ... + partials[tp-1], added left to right
 * in fp32, for a [rows, cols] result.
 *   partials : fp32 [tp, rows, cols], shard-major.               (input)
 *   out      : [rows, cols] (ALLREDUCE) or [tp, rows, cols/tp]
 *              (REDUCE_SCATTER), element type out_dtype.          (output)
 *   tp >= 1; REDUCE_SCATTER needs cols % tp == 0.
 * ------------------------------------------------------------------------ */
tpl_status tpl_shard_reduce(const float* partials, void* out, int64_t rows, int64_t cols,
                            int tp, int mode, int out_dtype, void* stream);

/* --------------------------------------------------------------------------
 * tp_mlp_forward -- Megatron SwiGLU MLP, column then row ([L4] S4.1).
 *
 *   X  [B, D]            input tokens (replicated on every shard).
 *   Wg, Wu [F, D]        gate / up weights; shard s uses rows
 *                        [s F/tp, (s+1) F/tp) (column-parallel, case 1).
 *   Wd [D, F]            down weight; shard s uses columns
 *                        [s F/tp, (s+1) F/tp) (row-parallel, case 3).
 *   Y  [B, D]            output, sum over shards of H_s Wd_s^T.
 *   partials             optional fp32 [tp, B, D]: if non-NULL the per-shard
 *                        partials P_s = H_s Wd_s^T are written there and then
 *                        reduced by the shard_reduce kernel; if NULL the
 *                        reduction is fused into the down projection
 *                        (shard partials accumulated in ascending s order).
 * H_s = silu(X Wg_s^T) * (X Wu_s^T) with silu(z) = z / (1 + exp(-z)); for
 * TPL_BF16 H is rounded to bf16 (it is the down projection's operand).
 * F % tp == 0 and D % 8 == 0, F % 8 == 0 are required (TPL_ERR_SHAPE / ALIGN).
 * ------------------------------------------------------------------------ */
tpl_status tpl_tp_mlp_forward_workspace(int64_t B, int64_t D, int64_t F, int tp, int dtype,
                                        size_t* bytes);
tpl_status tpl_tp_mlp_forward(const void* X, const void* Wg, const void* Wu, const void* Wd,
                              void* Y, float* partials, int64_t B, int64_t D, int64_t F, int tp,
                              int dtype, int out_dtype, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * tp_mlp_forward_static_ws -- tp_mlp_forward for callers that cannot allocate
 * device memory.  The reference pages have no counterpart: this is a service
 * of this library, not a step of the method.
 *
 * Some callers have no device buffer to give as `ws`: a serving loop that has
 * handed all of HBM to its own pool (KV cache, weights), code that must not
 * call cudaMalloc because it synchronises the device or would break a stream
 * capture in progress, or a host that links this library without any
 * allocator of its own.  This entry point takes the same arguments as
 * tp_mlp_forward minus ws / ws_bytes and runs the same kernels, with scratch
 * taken from a static __device__ array inside the library of
 * TPL_STATIC_WS_BYTES (32 MiB).  Every GPU on which the library is loaded
 * holds that array until the process exits.
 *   - The caller still owns and passes X, the weights, Y and the optional
 *     partials.  No device memory is allocated or freed by this call.
 *   - The scratch this call needs (the workspace plan of tp_mlp_forward for
 *     the partials argument given) must fit in TPL_STATIC_WS_BYTES, else
 *     TPL_ERR_STATIC_LIMIT and nothing is launched.  Shape and dtype errors
 *     are reported first, with the codes tp_mlp_forward gives.  Decode-sized
 *     calls fit, e.g. D 1536, F 8960 (tp 2) up to B = 128 and D 8192,
 *     F 28672 (tp 8) up to B = 32; B = 64 of the latter and a 4096-token
 *     prefill (352 MiB of workspace) do not.
 *   - The array used is the one of the host thread's current device, so the
 *     current device must be the one that owns the stream and the tensors.
 *     A stream of another device gives TPL_ERR_UNSUPPORTED.
 *   - All calls on a device share the one array, which keeps what the last
 *     call left in it (nothing in it needs to start at zero).  Calls whose
 *     kernels overlap on the GPU -- on different streams or from different
 *     host threads without ordering -- race on it; order them on one stream.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture that includes this call.
 * ------------------------------------------------------------------------ */
#define TPL_STATIC_WS_BYTES (32u << 20)
tpl_status tpl_tp_mlp_forward_static_ws(const void* X, const void* Wg, const void* Wu,
                                        const void* Wd, void* Y, float* partials, int64_t B,
                                        int64_t D, int64_t F, int tp, int dtype, int out_dtype,
                                        void* stream);

/* --------------------------------------------------------------------------
 * tp_attn_proj -- attention projections split by head ([L4] S4.2, S4.4).
 *
 *   X     [B, D]
 *   Wqkv  [(n_q + 2 n_kv) head_dim, D], rows [Q heads | K heads | V heads],
 *         each head head_dim consecutive rows.
 *   Wo    [D, n_q head_dim]; shard s uses the columns of its Q heads.
 *   qkv_out optional: per shard s, [B, (nq_s + 2 nkv_s) head_dim] in
 *         [Q_s | K_s | V_s] order, shards concatenated ([tp, B, ...]).
 *   Y     [B, D] = sum over shards of O_s Wo_s^T.
 *   partials optional fp32 [tp, B, D] as in tp_mlp_forward.
 * Shard s owns Q heads [s n_q/tp, (s+1) n_q/tp).  If tp <= n_kv it owns KV
 * groups [s n_kv/tp, (s+1) n_kv/tp) (needs n_kv % tp == 0); if tp > n_kv it
 * holds a copy of KV group floor(s n_kv / tp) (needs tp % n_kv == 0).
 * The attention core between the projections is not part of this library:
 * O_s is the attention output for a context of one token (the token itself),
 * where softmax over one key is exactly 1, so Q head h outputs the value
 * vector of its KV group floor(h n_kv / n_q).
 * ------------------------------------------------------------------------ */
tpl_status tpl_tp_attn_proj_workspace(int64_t B, int64_t D, int n_q, int n_kv, int head_dim,
                                      int tp, int dtype, size_t* bytes);
tpl_status tpl_tp_attn_proj(const void* X, const void* Wqkv, const void* Wo, void* qkv_out,
                            void* Y, float* partials, int64_t B, int64_t D, int n_q, int n_kv,
                            int head_dim, int tp, int dtype, int out_dtype, void* ws,
                            size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * sharded_matmul -- C = A B in one of the four cases of [L4] S3.2, over X
 * logical devices.  A [I, J] row-major; B [J, K] stored transposed as
 * Bt [K, J] (the [out, in] weight layout).
 *   case 1: A[I_X, J] B[J, K]   -> C[I_X, K] stored [I, K]; no communication.
 *   case 2: A[I, J_X] B[J, K]   -> all-gather A (a view here), C[I, K].
 *   case 3: A[I, J_X] B[J_X, K] -> partial sums over J blocks, then
 *           mode ALLREDUCE: C[I, K]; REDUCE_SCATTER: C[I, K_X] ([X, I, K/X]).
 *           partials optional fp32 [X, I, K] as in tp_mlp_forward.
 *   case 4: A[I_X, J] B[J, K_X] -> gather TPL_GATHER_B: case 1, C[I, K];
 *           TPL_GATHER_A: C[I, K_X] stored [X, I, K/X].
 * The sharded dimensions must divide by X (TPL_ERR_SHAPE).
 * ------------------------------------------------------------------------ */
tpl_status tpl_sharded_matmul_workspace(int case_id, int mode, int64_t I, int64_t J, int64_t K,
                                        int X, int dtype, size_t* bytes);
tpl_status tpl_sharded_matmul(int case_id, int mode, int gather, const void* A, const void* Bt,
                              void* C, float* partials, int64_t I, int64_t J, int64_t K, int X,
                              int dtype, int out_dtype, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * tp_decoder_layer / tp_decoder_stack -- serial pre-norm decoder layer built
 * from the calls above (bf16 only):
 *   h = x + Attn(RMSNorm(x));  y = h + MLP(RMSNorm(h))
 * RMSNorm has unit gain and eps = 1e-6 and is computed on every shard
 * ([L4] S4.2: replicated).  Its per-row scale 1/rms multiplies the fp32
 * products of the projection that consumes it (RMSNorm(x) W^T =
 * diag(1/rms(x)) x W^T), so the normalised rows are never rounded to bf16.
 * Attn and MLP are tp_attn_proj and tp_mlp_forward with the shard reduction
 * fused with the residual add.  x, y [B, D] bf16;
 * y may equal x.  The stack applies n_layers layers in order; the weight
 * pointer arrays live in HOST memory, one device pointer per layer.
 * This composition goes beyond the pages' four operations; it exists to run
 * a whole decode step.
 *
 * Two implementations compute it.  FUSED (B <= 128 tokens; D, F and
 * head_dim multiples of 64): one persistent cooperative launch per up to
 * 32 layers streams every weight once through tensor-core GEMMs with the
 * weights as the M operand; split-K partial tiles are added, in k (shard)
 * order, by the CTAs that computed them, and each projection starts on the
 * tiles whose inputs are final (per-tile readiness, no grid-wide barrier).  UNFUSED: one launch per
 * projection and per shard reduction.  The two add partial sums in
 * different orders, so they agree to rounding, not bit for bit; each is
 * deterministic.  tpl_tp_decoder_stack / _layer take FUSED where it applies.
 * ------------------------------------------------------------------------ */
typedef enum tpl_decode_path {
    TPL_PATH_AUTO = 0,      /* FUSED where it applies, else UNFUSED */
    TPL_PATH_UNFUSED = 1,
    TPL_PATH_FUSED = 2      /* TPL_ERR_UNSUPPORTED where it does not apply */
} tpl_decode_path;
tpl_status tpl_tp_decoder_workspace(int64_t B, int64_t D, int64_t F, int n_q, int n_kv,
                                    int head_dim, int tp, size_t* bytes);
tpl_status tpl_tp_decoder_layer(const void* x, void* y, const void* Wqkv, const void* Wo,
                                const void* Wg, const void* Wu, const void* Wd, int64_t B,
                                int64_t D, int64_t F, int n_q, int n_kv, int head_dim, int tp,
                                void* ws, size_t ws_bytes, void* stream);
tpl_status tpl_tp_decoder_stack(const void* x, void* y, const void* const* Wqkv,
                                const void* const* Wo, const void* const* Wg,
                                const void* const* Wu, const void* const* Wd, int n_layers,
                                int64_t B, int64_t D, int64_t F, int n_q, int n_kv, int head_dim,
                                int tp, void* ws, size_t ws_bytes, void* stream);
/* Block arrangement ([L4] S5.5).  SERIAL: the pre-norm block above.  PARALLEL
 * (PaLM): y = x + Attn(RMSNorm(x)) + MLP(RMSNorm(x)); both sublayers read the
 * same normalised input and their shard partials are summed together with x in
 * one reduction (the pages' shared all-reduce), so the fused stack needs two
 * grid-wide exchanges per layer instead of four.  PARALLEL runs on the FUSED
 * implementation only (TPL_ERR_UNSUPPORTED where it does not apply). */
typedef enum tpl_block { TPL_BLOCK_SERIAL = 0, TPL_BLOCK_PARALLEL = 1 } tpl_block;

/* tp_decoder_stack with the implementation chosen by `path` (tpl_decode_path). */
tpl_status tpl_tp_decoder_stack_path(const void* x, void* y, const void* const* Wqkv,
                                     const void* const* Wo, const void* const* Wg,
                                     const void* const* Wu, const void* const* Wd, int n_layers,
                                     int64_t B, int64_t D, int64_t F, int n_q, int n_kv,
                                     int head_dim, int tp, void* ws, size_t ws_bytes, int path,
                                     void* stream);
/* tp_decoder_stack with both the implementation (`path`) and the block
 * arrangement (`block`, tpl_block) chosen. */
tpl_status tpl_tp_decoder_stack_ex(const void* x, void* y, const void* const* Wqkv,
                                   const void* const* Wo, const void* const* Wg,
                                   const void* const* Wu, const void* const* Wd, int n_layers,
                                   int64_t B, int64_t D, int64_t F, int n_q, int n_kv, int head_dim,
                                   int tp, void* ws, size_t ws_bytes, int path, int block,
                                   void* stream);

/* --------------------------------------------------------------------------
 * Weight-only int8 decode MLP ("Lecture 4 - Distributed Serving", S5.5: only
 * the weights are quantised, which cuts the time spent reading them; S6.2: the
 * cheapest configurations are those whose weights take half the bytes).
 *
 * tpl_quantize_w8: symmetric per-(row, column group) quantisation of a bf16
 * matrix W [rows, cols] (row-major, read only).  Row r is split into `groups`
 * contiguous groups of cols/groups columns; group g gets
 * scale[r * groups + g] = amax(|W[r, group g]|) / 127 (float32) and
 * Q[r, c] = clamp(round_half_even(W[r, c] / scale), -127, 127) (int8,
 * row-major), the division in IEEE float32; a group of zeros gets scale 0 and
 * codes 0.  Use groups = 1 for Wg and Wu ([F, D]) and groups = tp for Wd
 * ([D, F], row-parallel), so that every shard's codes depend only on the
 * weights that shard holds.  Requires (cols / groups) % 8 == 0 and W 16-byte,
 * Q 8-byte, scale 4-byte aligned (TPL_ERR_ALIGN), no overlap (TPL_ERR_ALIAS).
 *
 * tpl_tp_mlp_forward_w8: tp_mlp_forward with int8 weights and bf16
 * activations.  Computes exactly what tp_mlp_forward computes on the
 * dequantised weights Q * scale: H = bf16(silu(X Wg^T) * (X Wu^T)), per-shard
 * fp32 partials of H Wd^T, summed in ascending shard order into Y.
 *   X [B, D] bf16; Qg, Qu [F, D] int8 with sg, su [F]; Qd [D, F] int8 with
 *   sd [D, tp]; Y [B, D] of out_dtype (TPL_BF16 or TPL_F32); partials
 *   (optional) [tp, B, D] fp32.  Requires F % tp == 0, D % 64 == 0,
 *   (F / tp) % 64 == 0 (TPL_ERR_SHAPE); X, Y, partials, Q* and ws 16-byte
 *   aligned, scales 4-byte aligned (TPL_ERR_ALIGN); ws of at least
 *   tpl_tp_mlp_forward_w8_workspace bytes (TPL_ERR_WORKSPACE; nothing in it
 *   needs to start at zero); outputs and ws disjoint from the inputs
 *   (TPL_ERR_ALIAS); the sm_103 tensor-core path (TPL_ERR_UNSUPPORTED).
 *   One or two tokens run on CUDA cores (fp32 FMAs); more run on the tensor
 *   cores, the int8 tiles widened to bf16 on the chip.  Every int8 value is a
 *   bf16 value, so only the accumulation order differs from the bf16 call.
 *   Asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
tpl_status tpl_quantize_w8(const void* W, int64_t rows, int64_t cols, int groups, int8_t* Q,
                           float* scale, void* stream);
tpl_status tpl_tp_mlp_forward_w8_workspace(int64_t B, int64_t D, int64_t F, int tp, size_t* bytes);
tpl_status tpl_tp_mlp_forward_w8(const void* X, const int8_t* Qg, const float* sg, const int8_t* Qu,
                                 const float* su, const int8_t* Qd, const float* sd, void* Y,
                                 float* partials, int64_t B, int64_t D, int64_t F, int tp,
                                 int out_dtype, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * Vocabulary-parallel lm_head with a top-k candidate exchange
 * ("Lecture 4 - Distributed Serving", S4.5 "lm_head and sequence parallelism").
 * The lm_head is split by vocabulary: shard s owns the rows
 * [s V/tp, (s+1) V/tp) of W and scores only those entries.  Instead of
 * gathering all V logits per token, each shard keeps its k best (index, logit)
 * pairs and only those tp x k candidates per token are exchanged; the result
 * is the global top-k of the logits x . W[v].
 *   X          [B, D] bf16 row-major: final hidden states (after any final
 *              norm; a positive per-token scale does not change the ranking).
 *   W          [V, D] bf16 row-major: lm_head weight, one row per vocabulary
 *              entry ([out, in]).  Read only.
 *   top_idx    [B, k] int32 out: vocabulary indices, best first.
 *   top_val    [B, k] fp32 out, may be NULL: their logits (fp32 accumulation
 *              of the bf16 products).
 *   shard_idx, shard_val  [tp, B, k] out, each may be NULL: every shard's own
 *              top-k, i.e. the candidates that are exchanged.
 * Order: larger logit first; equal logits (-0 equals +0) by lower index, so
 * the result is unique and deterministic.  NaN logits rank above +inf.
 * Requires 1 <= B, V % tp == 0, 1 <= k <= min(8, V / tp), D % 8 == 0
 * (TPL_ERR_SHAPE), V < 2^31, dtype TPL_BF16 (TPL_ERR_DTYPE), X and W 16-byte
 * aligned, outputs 4-byte aligned (TPL_ERR_ALIGN), outputs disjoint from the
 * inputs and the workspace (TPL_ERR_ALIAS), ws of at least the size
 * tpl_vocab_parallel_topk_workspace reports (TPL_ERR_WORKSPACE; nothing in it
 * needs to start at zero), and the sm_103 tensor-core path
 * (TPL_ERR_UNSUPPORTED otherwise).  Two kernels on `stream`; asynchronous.
 * ------------------------------------------------------------------------ */
tpl_status tpl_vocab_parallel_topk_workspace(int64_t B, int64_t V, int tp, int k, size_t* bytes);
tpl_status tpl_vocab_parallel_topk(const void* X, const void* W, int64_t B, int64_t D, int64_t V,
                                   int tp, int k, int dtype, int32_t* top_idx, float* top_val,
                                   int32_t* shard_idx, float* shard_val, void* ws,
                                   size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * Launch timing, for measurement only (off by default).
 * tpl_profile_enable(n > 0) creates n pairs of CUDA events (host objects; no
 * device memory) and from then on brackets each kernel launch with a pair on
 * the launch's stream, tagged with the step it implements ("qkv", "oproj",
 * "gateup", "down", "matmul", "reduce", "reduce_norm", "rmsnorm",
 * "fused_stack", "lm_head_topk" (both lm_head kernels), "quantize_w8",
 * "w8_gateup", "w8_down").  Launches
 * beyond n are not recorded.  tpl_profile_enable(0) turns it off and frees the
 * events.  tpl_profile_count() is the number of recorded launches;
 * tpl_profile_read(i, ...) waits for launch i and returns its tag and its
 * device time in milliseconds.  Under CUDA-graph capture the event records
 * become nodes of the graph; the times read are those of its latest replay.
 * ------------------------------------------------------------------------ */
tpl_status tpl_profile_enable(int max_launches);
int tpl_profile_count(void);
tpl_status tpl_profile_read(int i, char* tag, size_t tag_len, float* ms);

/* --------------------------------------------------------------------------
 * Phase trace of the fused decode stack, for measurement only.  An
 * instrumented build of the library (build.py --trace: libtpl_trace.so, the
 * kernels compiled with TPL_FUSED_TRACE) records, for every CTA and phase of
 * its last fused launch, %globaltimer stamps (ns) of 12 events:
 *   0 the activation producer found the first unit's inputs final,
 *   1 the first MMA of the phase was issued, 2 the first unit was delivered
 *   (counted on its tile ticket, or its tagged words stored), 3 the CTA
 *   drained its last unit of the phase, 4 its
 *   first finalize of the phase passed its waits, 5 it published its last
 *   finalized tile, 6 the weight producer issued its first tile of the
 *   phase, 7 the activation producer began waiting for the phase's inputs,
 *   8 the MMA issuer committed the phase's first unit, 9 the weight
 *   producer issued its last tile of the phase, 10 the epilogue saw the
 *   first unit's accumulator full, 11 the activation producer issued its
 *   last activation tile of the phase.
 * Layout [148 CTAs][1 + 4*32 phases][12 events] uint64, 0 = not reached.
 * tpl_fused_trace_read synchronises the device and copies up to `bytes` of
 * it to host memory; the normal build returns TPL_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------ */
tpl_status tpl_fused_trace_read(void* host, size_t bytes);

/* --------------------------------------------------------------------------
 * Test hook for the failure path of the fused decode stack (off by default).
 * Not a step of the method: the pages name the failure it stands in for -- a
 * collective that never completes because one rank never arrives (the NCCL
 * hang and timeout modes of the TP serving pages) -- and this makes that
 * happen on one GPU without a fault.
 *
 * Every wait of the fused stack (between CTAs: tile tickets or tagged partial
 * words, tile readiness, phase completion; inside a CTA: the mbarriers of its
 * pipeline and the phase watcher's posts) gives up
 * after a time limit, raises the launch's abort flag so that every CTA stops
 * waiting, drains its copies and MMAs in flight, frees its tensor memory and
 * returns; the sticky device error word then holds TPL_DEVERR_TIMEOUT
 * (tpl_device_status).  tpl_test_fused_fault(cta, phase, wait_limit_ns)
 * applies to the fused-stack launches issued after it:
 *   - cta >= 0: CTA `cta` does not deliver its first unit of phase `phase`
 *     (>= 1; phase 4 l + 1 + j is projection j of layer l of the launch, in
 *     the block's phase order): no count on its tile's ticket or, up to 16
 *     tokens, no tagged partial words, so the tile's finalize waits until
 *     the limit passes.  cta < 0 turns the omission off.
 *   - wait_limit_ns > 0 sets the limit (10 us .. 2 s); <= 0 restores 2 s.
 * After such a launch the workspace needs nothing: the next launch starts
 * from zeroed counters and tagged words and rewrites every buffer before
 * reading it.
 * Returns TPL_ERR_UNSUPPORTED for arguments out of range.
 * ------------------------------------------------------------------------ */
tpl_status tpl_test_fused_fault(int cta, int phase, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* TPL_H */
