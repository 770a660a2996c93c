/*
 * blk.h - C ABI of the GB300 (sm_103a) prefill forward of one decoder block.
 *
 * The block, as the pages state it:
 *   - sequential pre-norm (nnterp encyclopedia "stablelm", 03 Notes, "The
 *     block is sequential on 1.6B and 3B"): h = x + attn(LN1(x)); y = h + mlp(LN2(h))
 *   - parallel (same section, 12B): n = LN(x); y = x + attn(n) + mlp(n)
 *   - reordered post-norm ("OLMo-2: reordered (post) normalization", section 1):
 *     no input norm; h = x + RMS(attn(x)); y = h + RMS(mlp(h))
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller. The library
 *     allocates no device memory, frees nothing and never synchronises a
 *     stream (blk_check_device_status is the one call that does, by design).
 *   - Work is enqueued on the caller's stream `s` (a cudaStream_t; NULL is the
 *     legacy default stream) and runs asynchronously. Stream order holds as
 *     for any kernel: each call's first kernel reads nothing before the work
 *     enqueued ahead of it on `s` has completed. Outside stream capture the
 *     hot-path kernels are launched with programmatic stream serialization,
 *     so a kernel may begin its set-up (shared memory, barriers, TMEM)
 *     while the previous one drains; it waits for that grid's completion
 *     (griddepcontrol.wait) before its first global access. A kernel the
 *     caller enqueues after a call is ordered as usual, unless the caller
 *     launches it with the same attribute.
 *   - Row-major, contiguous, 16-byte-aligned tensors. Linear weights follow the
 *     torch convention W[out, in], y = x W^T + b (nnterp "stablelm" Printout).
 *   - Storage dtype `dt` is fp16 or bf16 for every tensor of a call, except
 *     ALiBi slopes (fp32). All accumulation and statistics are fp32. K/V are
 *     read at the stated dtype: nothing is silently converted.
 *   - Every call validates its arguments before any launch and returns a
 *     blk_status; a rejected call has no side effects. blk_last_error() gives a
 *     thread-local message for the last failure.
 *   - Every wait inside a kernel is bounded (about 2 s); on timeout the kernel
 *     sets a device error word and exits. blk_check_device_status() reports it.
 */
#ifndef BLK_H
#define BLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* blk_stream_t; /* same type as cudaStream_t */

typedef enum {
    BLK_OK = 0,
    BLK_EINVAL = 1,        /* bad argument: null pointer, bad size, misalignment */
    BLK_EUNSUPPORTED = 2,  /* valid request outside what the kernels implement */
    BLK_ECUDA = 3,         /* a CUDA runtime/driver call failed */
    BLK_ETIMEOUT = 4,      /* a bounded in-kernel wait gave up (device error word) */
    BLK_EWORKSPACE = 5     /* workspace pointer null or smaller than required */
} blk_status;

typedef enum { BLK_F16 = 0, BLK_BF16 = 1 } blk_dtype;

typedef enum { BLK_QKV_STACKED = 0, BLK_QKV_HEAD_INTERLEAVED = 1 } blk_qkv_layout;
typedef enum { BLK_QKNORM_NONE = 0, BLK_QKNORM_RMS_FULL = 1, BLK_QKNORM_LN_PER_HEAD = 2 } blk_qk_norm;
typedef enum { BLK_NORM_LAYERNORM = 0, BLK_NORM_RMS = 1 } blk_norm_kind;
typedef enum { BLK_NORM_PRE = 0, BLK_NORM_POST = 1 } blk_norm_place;
typedef enum { BLK_RESIDUAL_SEQUENTIAL = 0, BLK_RESIDUAL_PARALLEL = 1 } blk_residual;
typedef enum { BLK_ACT_SWIGLU = 0, BLK_ACT_GELU_TANH = 1 } blk_act;

/* ---- status ---------------------------------------------------------- */

const char* blk_status_string(blk_status s);
/* Message for the last failed call on this host thread ("" if none). */
const char* blk_last_error(void);
/* ABI version: (major << 16) | minor. */
int blk_version(void);
/* Synchronises `s`, then reads and clears the device error word of the
 * current device. BLK_ETIMEOUT if an in-kernel bounded wait gave up since the
 * last check; BLK_ECUDA on a CUDA error. */
blk_status blk_check_device_status(blk_stream_t s);

/* Self-test of the failure path: enqueues one single-thread kernel that
 * waits on a barrier nothing ever completes, with a wait limit of limit_ns
 * (1 us .. 5 s) instead of the kernels' ~2 s. The wait gives up, sets the
 * device error word and the kernel returns, so the next
 * blk_check_device_status(s) reports BLK_ETIMEOUT (and clears it) while the
 * context stays usable. No GPU fault, trap or hang is involved. */
blk_status blk_selftest_bounded_wait(uint64_t limit_ns, blk_stream_t s);

/* ---- norms ------------------------------------------------------------ */

/* LayerNorm with bias ("StableLM-2: partial RoPE and a first
 * LayerNorm-with-bias path", section 1; nnterp "stablelm" Printout):
 *   y[r,:] = (x[r,:] - mean) / sqrt(var + eps) * gamma + beta  [+ residual[r,:]]
 * population variance over `cols`. x, residual, y: [rows, cols]; gamma,
 * beta: [cols]. beta NULL = bias-free LayerNorm. residual NULL = no add (the
 * add, when given, comes after the norm). y may alias x. cols % 8 == 0,
 * cols <= 16384. */
blk_status blk_layernorm_bias(const void* x, const void* residual, const void* gamma,
                              const void* beta, void* y, int64_t rows, int64_t cols, float eps,
                              blk_dtype dt, blk_stream_t s);

/* RMSNorm ("OLMo-2: reordered (post) normalization", section 1):
 *   y[r,:] = x[r,:] / sqrt(mean(x[r,:]^2) + eps) * weight  [+ residual[r,:]]
 * Same layout and rules as blk_layernorm_bias. With a residual this is the
 * OLMo-2 post-norm add: h = residual + RMS(sublayer_out). */
blk_status blk_rmsnorm(const void* x, const void* residual, const void* weight, void* y,
                       int64_t rows, int64_t cols, float eps, blk_dtype dt, blk_stream_t s);

/* ---- projection, rotary, qk-norm -------------------------------------- */

typedef struct {
    int64_t batch, seq, hidden, n_heads, n_kv_heads, head_dim;
    int32_t qkv_layout;  /* blk_qkv_layout; HEAD_INTERLEAVED needs n_heads == n_kv_heads */
    int32_t qk_norm;     /* blk_qk_norm */
    float qk_norm_eps;
    int32_t rotary_span; /* 0..head_dim, even; 0 = rotary off (no trig evaluated) */
    float rope_base;     /* theta_j = rope_base^(-2j/rotary_span), positions 0..seq-1 */
} blk_qkv_desc;

/* QKV projection with bias, de-interleave/head split, optional qk-norm and
 * partial NeoX split-half rotary ("StableLM-2: partial RoPE ...", section 1;
 * nnterp "stablelm" 03 Notes: bias added before the rotary, first
 * rotary_span dims of each q/k head rotate as two halves, the rest pass
 * through; "Bloom in a sovereign engine", Contribution: fused QKV
 * de-interleave; "OLMo-2 ...", section 1: full-width QK RMSNorm; nnterp
 * 03 Notes "Per-head LayerNorms on queries and keys on 12B").
 *   x      [batch*seq, hidden]
 *   w_qkv  [(H + 2*Hk)*d, hidden]: STACKED rows [Wq; Wk; Wv], or
 *          HEAD_INTERLEAVED rows [head][q,k,v][d]
 *   b_qkv  [(H + 2*Hk)*d] in the same row order, or NULL
 *   q_norm_w / k_norm_w: RMS_FULL -> [H*d] / [Hk*d]; LN_PER_HEAD -> [H, d] /
 *          [Hk, d] (bias-free LayerNorm per head, before the rotary); NONE -> NULL
 *   q [batch, H, seq, d], k and v [batch, Hk, seq, d] (outputs).
 * hidden % 8 == 0; head_dim a multiple of 32, at most 256. */
blk_status blk_qkv_bias_rope_partial(const blk_qkv_desc* d, const void* x, const void* w_qkv,
                                     const void* b_qkv, const void* q_norm_w,
                                     const void* k_norm_w, void* q, void* k, void* v,
                                     blk_dtype dt, blk_stream_t s);

/* In-place optional bias add then partial NeoX rotary on a head-split tensor
 * x [batch, n_heads, seq, head_dim] (positions 0..seq-1). bias: [n_heads*head_dim]
 * or NULL. rotary_span 0 = bias only. Same rotary as blk_qkv_bias_rope_partial. */
blk_status blk_rope_inplace(void* x, const void* bias, int64_t batch, int64_t n_heads,
                            int64_t seq, int64_t head_dim, int32_t rotary_span, float rope_base,
                            blk_dtype dt, blk_stream_t s);

/* ---- attention -------------------------------------------------------- */

typedef struct {
    int64_t batch, seq, n_heads, n_kv_heads, head_dim;
    float softmax_scale; /* <= 0 -> head_dim^-0.5 (nnterp "stablelm" 03 Notes) */
    int32_t causal;      /* must be 1: prefill is causal */
    int32_t alibi;       /* 0 off; 1: score -= slope_h * (query_pos - key_pos) */
} blk_attn_desc;

/* Causal softmax attention, flash-style on tcgen05 tensor cores, with
 * optional ALiBi ("Bloom in a sovereign engine", Contribution: per-head
 * geometric slope, linear pre-softmax bias; the bias is added after the
 * score scale and is not scaled itself). GQA: kv head = h / (H / Hk).
 *   q [batch, H, seq, d]; k, v [batch, Hk, seq, d]
 *   alibi_slopes: device fp32 [H], or NULL with alibi=1 for the standard
 *     slopes 2^(-8(h+1)/H) (H a power of two)
 *   o [batch, seq, H, d] (= [batch*seq, H*d], what o_proj reads)
 * head_dim in {64, 128, 160}. Rotary and ALiBi are exclusive at the block
 * level: blk_forward rejects rotary_span > 0 together with alibi. */
blk_status blk_attn_prefill(const blk_attn_desc* d, const void* q, const void* k, const void* v,
                            const float* alibi_slopes, void* o, blk_dtype dt, blk_stream_t s);

/* ---- decode step ------------------------------------------------------ */

typedef struct {
    int64_t batch, max_seq, n_heads, n_kv_heads, head_dim;
    float softmax_scale; /* <= 0 -> head_dim^-0.5 */
    int32_t alibi;       /* 0 off; 1: score -= slope_h * (query_pos - key_pos) */
} blk_decode_desc;

/* One decode step of attention over a KV cache: the step after prefill (the
 * pages state prefill; this applies the same attention, nnterp "stablelm" 03
 * Notes and "Bloom in a sovereign engine", Contribution, to one new token).
 *   q [batch, H, d]: each sequence's newest token, at position lens[b] - 1
 *   k_cache, v_cache [batch, Hk, max_seq, d]: positions 0 .. lens[b] - 1 of
 *     sequence b (the newest already written); later entries are not read
 *   lens: device int32 [batch], each in [1, max_seq]. They are read on the
 *     device, so they cannot be checked here: a value outside the range is
 *     clamped to it, and a length of 0 gives a zero output row
 *   alibi_slopes: as for blk_attn_prefill
 *   o [batch, H, d]
 * GQA: kv head = h / (H / Hk), H / Hk in {1, 2, 4, 8}; head_dim 64 or 128.
 * Two launches (key ranges per (batch, kv head), then their merge); the
 * workspace holds the partial results, at least
 * blk_attn_decode_workspace_size bytes, 16-byte aligned. */
blk_status blk_attn_decode_workspace_size(const blk_decode_desc* d, size_t* bytes);
blk_status blk_attn_decode(const blk_decode_desc* d, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* lens, const float* alibi_slopes,
                           void* o, void* workspace, size_t ws_bytes, blk_dtype dt,
                           blk_stream_t s);

/* ---- linear and MLP --------------------------------------------------- */

/* y = x W^T [+ bias] [+ res1] [+ res2] on tcgen05 tensor cores.
 * x [m, k], w [n, k], bias [n], res1/res2/y [m, n]. k % 8 == 0, n % 8 == 0. */
blk_status blk_linear(const void* x, const void* w, const void* bias, const void* res1,
                      const void* res2, void* y, int64_t m, int64_t n, int64_t k, blk_dtype dt,
                      blk_stream_t s);

/* ---- Q8_0 weights ------------------------------------------------------ */

/* The q8/int8 weight path that the pages report as a secondary precision
 * ("StableLM-2: partial RoPE ...", section 3 Results: q8 prefill-logit
 * cosine 0.998910, 11/12 argmax; "OLMo-2: reordered (post) normalization
 * ...", section 4: int8 cosine 0.998700), in the one format they name: Q8_0
 * ("RoFormer HIP FP32 layout optimization": BS-RoFormer Q8_0), the GGML
 * format. A weight W[n, k] (torch convention, k % 32 == 0) is stored as
 *   q  int8 [n, k] row-major: one code per weight;
 *   d  fp16 [k/32, n]: one scale per row and 32-input block, block-major
 *      (the scale of row r, inputs 32j .. 32j+31 is d[j * n + r]).
 * Both pointers 16-byte aligned, owned by the caller. */

/* Quantize w [n, k] (dt) to Q8_0 on the GPU, with the float32 arithmetic of
 * GGML's reference quantizer: d = absmax / 127 per block, codes
 * round(w * (1 / d)) half away from zero (0 where d = 0), and d rounded to
 * fp16 only after the codes are taken. Bit-exact: the same w gives the same
 * q and d as any IEEE float32 implementation of those steps.
 * BLK_EINVAL: k not a positive multiple of 32, NULL or misaligned pointers. */
blk_status blk_q8_0_quantize(const void* w, int64_t n, int64_t k, int8_t* q, void* d,
                             blk_dtype dt, blk_stream_t s);

/* y = x W^T [+ bias] [+ res1] [+ res2] with W given as Q8_0 (q, d): blk_linear
 * with each weight element q * d rounded once to dt on chip (a W8A16 tcgen05
 * GEMM). x [m, k], bias [n], res1/res2/y [m, n] in dt; n % 8 == 0,
 * k % 32 == 0. Errors as blk_linear. */
blk_status blk_linear_q8_0(const void* x, const int8_t* q, const void* d, const void* bias,
                           const void* res1, const void* res2, void* y, int64_t m, int64_t n,
                           int64_t k, blk_dtype dt, blk_stream_t s);

typedef struct {
    int64_t tokens, hidden, intermediate;
    int32_t act; /* blk_act */
} blk_mlp_desc;

/* Workspace bytes blk_mlp needs (the [tokens, intermediate] activation). */
blk_status blk_mlp_workspace_size(const blk_mlp_desc* d, size_t* bytes);

/* The MLP (nnterp "stablelm" Printout and 02 support(): mlp_neurons =
 * act(gate)*up on a gated MLP):
 *   SWIGLU:    a = silu(x Wg^T) * (x Wu^T)               (w_gate required, b_up NULL)
 *   GELU_TANH: a = gelu_tanh(x Wu^T + b_up)              (w_gate NULL)
 *   y = a Wd^T [+ b_down] [+ res1] [+ res2]
 * x [tokens, hidden]; w_gate, w_up [intermediate, hidden]; w_down
 * [hidden, intermediate]; res1, res2, y [tokens, hidden]. workspace holds a. */
blk_status blk_mlp(const blk_mlp_desc* d, const void* x, const void* w_gate, const void* w_up,
                   const void* b_up, const void* w_down, const void* b_down, const void* res1,
                   const void* res2, void* y, void* workspace, size_t ws_bytes, blk_dtype dt,
                   blk_stream_t s);

/* Size of the device scratch array blk_mlp_noalloc keeps for its activation. */
#define BLK_MLP_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* blk_mlp without a workspace argument, for callers that cannot allocate
 * device memory: code running inside an engine or plugin host that owns all
 * device memory and forbids allocation once it has started, and latency-bound
 * callers that cannot take cudaMalloc's implicit device synchronisation.
 * The pages have no counterpart of this call; it only changes where the
 * [tokens, intermediate] activation lives.
 *
 * That activation goes to one fixed array of BLK_MLP_NOALLOC_SCRATCH_BYTES
 * (32 MiB) in the library's device memory, which every GPU that loads the
 * library keeps until the process exits. tokens * intermediate * 2 bytes must
 * fit in it; larger requests return BLK_EWORKSPACE and launch nothing. The
 * call allocates and frees nothing. Its first call on a device looks up the
 * array's device address (cudaGetSymbolAddress), so make that first call
 * before any stream capture. That address is kept for the life of the
 * process: after a cudaDeviceReset (or any reset of the device's primary
 * context) it is stale, so do not call blk_mlp_noalloc on a device that the
 * process has reset. All calls share the one array: calls whose
 * kernels overlap on the GPU (other streams, other host threads) race on it.
 * Every element the MLP reads from it is written first in the same call, so
 * nothing has to be cleared between calls. Arguments, results and errors are
 * otherwise those of blk_mlp. */
blk_status blk_mlp_noalloc(const blk_mlp_desc* d, const void* x, const void* w_gate,
                           const void* w_up, const void* b_up, const void* w_down,
                           const void* b_down, const void* res1, const void* res2, void* y,
                           blk_dtype dt, blk_stream_t s);

/* ---- the block -------------------------------------------------------- */

typedef struct {
    blk_qkv_desc qkv;     /* shapes, QKV layout, qk-norm, rotary */
    int32_t norm_kind;    /* blk_norm_kind, for the block norms */
    int32_t norm_place;   /* blk_norm_place: PRE (input norm) or POST (OLMo-2 reordered) */
    int32_t residual;     /* blk_residual */
    float eps;            /* block norm eps */
    int32_t alibi;        /* 1: ALiBi with standard slopes (or w->alibi_slopes); needs rotary_span 0 */
    int64_t intermediate; /* MLP width */
    int32_t act;          /* blk_act */
} blk_block_desc;

/* Named weight slots. Each norm has its own slot; no slot is read in place of
 * another ("OLMo-2 ...", section 1: the loader-clobber root cause). Unused
 * slots must be NULL. */
typedef struct {
    const void *attn_norm_w, *attn_norm_b;       /* PRE: input norm (LayerNorm bias nullable) */
    const void *mlp_norm_w, *mlp_norm_b;         /* PRE + SEQUENTIAL: MLP norm */
    const void *post_attn_norm_w, *post_mlp_norm_w; /* POST: RMSNorms on sublayer outputs */
    const void *w_qkv, *b_qkv, *q_norm_w, *k_norm_w;
    const void *w_o, *b_o;
    const void *w_gate, *w_up, *b_up, *w_down, *b_down;
    const float* alibi_slopes;                   /* optional device fp32 [H] */
} blk_block_weights;

/* Workspace bytes blk_forward needs for this descriptor. */
blk_status blk_forward_workspace_size(const blk_block_desc* d, size_t* bytes);

/* The prefill forward of one decoder block: x [batch, seq, hidden] ->
 * y [batch, seq, hidden]. y must not alias x. Every step runs in this
 * library's kernels on stream s; workspace (caller-owned device memory of at
 * least blk_forward_workspace_size bytes) holds the intermediates. */
blk_status blk_forward(const blk_block_desc* d, const blk_block_weights* w, const void* x,
                       void* y, void* workspace, size_t ws_bytes, blk_dtype dt, blk_stream_t s);

/* Kinds of the kernel launches blk_forward enqueues, in the order they run. */
typedef enum {
    BLK_STEP_INPUT_NORM = 0,   /* input LayerNorm/RMSNorm (pre-norm blocks) */
    BLK_STEP_QKV = 1,          /* projection + bias (+ fused rotary) + head split */
    BLK_STEP_QK_NORM_ROPE = 2, /* qk-norm and/or rotary wider than the fused span */
    BLK_STEP_ATTENTION = 3,    /* causal flash attention (+ALiBi) */
    BLK_STEP_O_PROJ = 4,       /* output projection (+bias, +residual) */
    BLK_STEP_POST_ATTN_NORM = 5, /* OLMo-2: h = x + RMS(attn_out) */
    BLK_STEP_MLP_NORM = 6,     /* LN/RMS of h (sequential pre-norm) */
    BLK_STEP_MLP_UP = 7,       /* gate/up GEMM + SwiGLU, or up GEMM + bias + GELU */
    BLK_STEP_MLP_DOWN = 8,     /* down GEMM (+bias, +residuals) */
    BLK_STEP_POST_MLP_NORM = 9, /* OLMo-2: y = h + RMS(mlp_out) */
    BLK_STEP_Q8_DEQUANT = 10   /* Q8_0 weights expanded for the dense GEMMs (blk_forward_q8_0) */
} blk_step_kind;

/* blk_forward, also reporting its kernel launches. If `events` is non-NULL
 * it points to n_events cudaEvent_t handles (created by the caller): events[0]
 * is recorded on s before the first launch and events[i] right after launch
 * i, for i < n_events; the time between events[i-1] and events[i] is launch
 * i's duration on the stream. If step_kinds is non-NULL it receives the
 * blk_step_kind of each launch (room for n_events - 1 entries, or 12 when
 * events is NULL; at most 12 are written, and a block makes at most 9
 * launches).
 * *n_launches (nullable) receives the number of launches. */
blk_status blk_forward_ex(const blk_block_desc* d, const blk_block_weights* w, const void* x,
                          void* y, void* workspace, size_t ws_bytes, blk_dtype dt, blk_stream_t s,
                          void* const* events, int n_events, int32_t* step_kinds, int* n_launches);

/* The block with Q8_0 projection weights (the q8 rows of "StableLM-2: partial
 * RoPE ...", section 3 Results and "OLMo-2 ...", section 4; format above):
 * blk_forward with every projection (QKV, output, MLP gate/up, down) taken
 * with weights q * d, each rounded once to dt. w holds the norms, biases,
 * qk-norm weights and ALiBi slopes as for blk_forward; its five projection
 * slots (w_qkv, w_o, w_gate, w_up, w_down) must be NULL, and q8 gives them,
 * with the same shapes ([out, in] codes, [in/32, out] scales; q_gate/d_gate
 * NULL unless the MLP is SwiGLU). hidden, n_heads * head_dim and
 * intermediate must be multiples of 32.
 * Two ways to run the projections, with the same weight values (sums may
 * differ in fp32 accumulation order):
 *   - W8A16 GEMMs that expand the codes on chip, tile by tile: with a
 *     workspace of blk_forward_workspace_size bytes, or below 512 tokens;
 *   - dequantize once: with at least 512 tokens and a workspace of
 *     blk_forward_q8_0_workspace_size bytes, all projections' weights are
 *     first expanded into the workspace's tail (one extra launch, step kind
 *     BLK_STEP_Q8_DEQUANT), then multiplied by the dense GEMMs: at large
 *     token counts the W8A16 kernel would expand every weight tile once per
 *     128 tokens.
 * Errors and everything else as blk_forward. */
typedef struct {
    const int8_t *q_qkv, *q_o, *q_gate, *q_up, *q_down;  /* codes */
    const void *d_qkv, *d_o, *d_gate, *d_up, *d_down;    /* fp16 scales */
} blk_q8_weights;
/* Workspace bytes of blk_forward_q8_0's dequantize-once path:
 * blk_forward_workspace_size plus every projection's weights in the storage
 * dtype (QKV, output, gate for SwiGLU, up, down; each 256-byte aligned).
 * Errors as blk_forward_workspace_size. */
blk_status blk_forward_q8_0_workspace_size(const blk_block_desc* d, size_t* bytes);
blk_status blk_forward_q8_0(const blk_block_desc* d, const blk_block_weights* w,
                            const blk_q8_weights* q8, const void* x, void* y, void* workspace,
                            size_t ws_bytes, blk_dtype dt, blk_stream_t s);
/* blk_forward_q8_0 with per-launch events, as blk_forward_ex. */
blk_status blk_forward_q8_0_ex(const blk_block_desc* d, const blk_block_weights* w,
                               const blk_q8_weights* q8, const void* x, void* y, void* workspace,
                               size_t ws_bytes, blk_dtype dt, blk_stream_t s,
                               void* const* events, int n_events, int32_t* step_kinds,
                               int* n_launches);

/* blk_forward on host buffers, with the copies overlapped with the compute.
 * x_host and y_host are [batch, seq, hidden] in pinned host memory; x_dev and
 * y_dev are device buffers of the same size (caller-owned, reused as
 * staging); workspace holds at least blk_forward_workspace_size(d) bytes.
 * The batch is split into n_chunks groups of whole sequences (1..16, at most
 * batch): chunk c's host-to-device copy, forward and device-to-host copy run
 * on two copy streams the library keeps per device and on s, so chunk c+1
 * is copied in while chunk c is computed and chunk c-1 copied out. The call
 * is ordered on s like any other: when s reaches the end of the call, y_host
 * holds the result. Calls must not overlap on the GPU (they share x_dev, y_dev
 * and the workspace). */
blk_status blk_forward_host(const blk_block_desc* d, const blk_block_weights* w,
                            const void* x_host, void* y_host, void* x_dev, void* y_dev,
                            void* workspace, size_t ws_bytes, int32_t n_chunks, blk_dtype dt,
                            blk_stream_t s);

/* ---- model-level wrap ------------------------------------------------- */

/* A stack of n_layers blocks of one shape between the token embedding and
 * the logits: x = embed[tokens]; for Bloom ("Bloom in a sovereign engine",
 * Contribution (2): a layernorm on the embeddings before the first block)
 * x = LN(x); x = block_l(x) for l = 0 .. n_layers-1; logits = norm(x)
 * lm_head^T (nnterp "stablelm" Printout and Config: a final LayerNorm with
 * bias, then lm_head, tie_word_embeddings False). */
typedef struct {
    blk_block_desc block; /* every layer's shapes and variant */
    int32_t n_layers;     /* >= 0 */
    int64_t vocab;        /* >= 8, a multiple of 8 */
    int32_t embed_norm;   /* 1: LayerNorm (bias nullable) on the embeddings before layer 0 */
    int32_t final_norm;   /* blk_norm_kind of the final norm */
    float final_eps;
} blk_model_desc;

typedef struct {
    const void* embed;                       /* [vocab, hidden] */
    const void *embed_norm_w, *embed_norm_b; /* embed_norm only (bias nullable) */
    const blk_block_weights* layers;         /* HOST array of n_layers weight sets */
    const void *final_norm_w, *final_norm_b; /* final_norm_b: LayerNorm bias, nullable */
    const void* lm_head;                     /* [vocab, hidden] */
} blk_model_weights;

/* Workspace bytes blk_model_forward needs: two [batch, seq, hidden]
 * activations, the final norm's output and one block's workspace. */
blk_status blk_model_workspace_size(const blk_model_desc* d, size_t* bytes);

/* tokens: device int32 [batch, seq]; logits: device [batch, seq, vocab] in
 * the storage dtype. Token ids live in device memory, so the host cannot
 * check them: an id outside [0, vocab) reads row 0 of the embedding (the
 * kernel clamps the index; nothing outside the table is read). Weights are
 * validated per layer as blk_forward does; everything runs on stream s. */
blk_status blk_model_forward(const blk_model_desc* d, const blk_model_weights* w,
                             const int32_t* tokens, void* logits, void* workspace,
                             size_t ws_bytes, blk_dtype dt, blk_stream_t s);

/* A pipeline of block forwards over a stream of host batches, for serving:
 * blk_host_pipe_submit enqueues one batch and returns. Batch n is copied in
 * (pinned x_host, [batch, seq, hidden] as in the desc) on a copy stream the
 * pipe owns while batch n-1's forward runs on s, and copied out (to pinned
 * y_host) on a second copy stream while batch n+1's forward runs, through
 * depth (2..4) device staging slots. The forwards themselves run in order on
 * s. Two departures from plain stream order, by design:
 *  - x_host must already hold the batch when submit is called: its copy may
 *    start at once (the first depth submits after create or a flush wait
 *    for the work enqueued on s before the first of them);
 *  - y_host of a batch is complete once s has passed a later
 *    blk_host_pipe_flush.
 * All submits between two flushes use the same stream s (BLK_EINVAL
 * otherwise). Each slot's forward is recorded as a CUDA graph on the slot's
 * first submit (and again when the weight pointers differ from the ones it
 * was recorded with) and replayed by later submits; the graph reads the
 * weights through those pointers, so their contents may change between
 * submits. The pipe is not thread-safe. dev_mem (blk_host_pipe_mem_size
 * bytes, 16-byte aligned, caller-owned) holds the staging slots and the
 * forward's workspace; it must stay valid until the submitted work has
 * completed. destroy does not wait for that work. */
typedef struct blk_host_pipe blk_host_pipe;
blk_status blk_host_pipe_mem_size(const blk_block_desc* d, int32_t depth, size_t* bytes);
blk_status blk_host_pipe_create(const blk_block_desc* d, int32_t depth, blk_dtype dt,
                                void* dev_mem, size_t bytes, blk_host_pipe** out);
blk_status blk_host_pipe_submit(blk_host_pipe* p, const blk_block_weights* w, const void* x_host,
                                void* y_host, blk_stream_t s);
blk_status blk_host_pipe_flush(blk_host_pipe* p, blk_stream_t s);
blk_status blk_host_pipe_destroy(blk_host_pipe* p);

/* A block forward recorded once as a CUDA graph and replayed: the same seven
 * to nine kernels with the same pointers, without per-launch host work or
 * the gaps between separately submitted launches. blk_forward_graph_create
 * captures blk_forward_ex(d, w, x, y, workspace, ...) with its optional
 * events (recorded inside the graph, re-recorded by every launch) on a
 * private stream; nothing runs until blk_graph_launch. *out receives a
 * handle owned by the caller (free with blk_graph_destroy). The buffers must
 * stay valid and keep their addresses while the handle is used; their
 * contents are read at launch time. step_kinds / n_launches as for
 * blk_forward_ex. blk_graph_launch enqueues one forward on s. */
typedef struct blk_graph blk_graph;
blk_status blk_forward_graph_create(const blk_block_desc* d, const blk_block_weights* w,
                                    const void* x, void* y, void* workspace, size_t ws_bytes,
                                    blk_dtype dt, void* const* events, int n_events,
                                    int32_t* step_kinds, int* n_launches, blk_graph** out);
blk_status blk_graph_launch(blk_graph* g, blk_stream_t s);
/* Point the graph's recorded events (created with n_events > 0; it records
 * min(n_events, launches + 1) of them) at other cudaEvent_t handles for the
 * launches enqueued after this call (earlier launches keep theirs), so
 * consecutive launches can be timed per kernel without waiting in between.
 * events[0 .. recorded-1] are used; n_events must be at least that. */
blk_status blk_graph_set_events(blk_graph* g, void* const* events, int n_events);
blk_status blk_graph_destroy(blk_graph* g);

#ifdef __cplusplus
}
#endif
#endif /* BLK_H */
