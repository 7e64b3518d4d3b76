/*
 * moe_ffn.h - C ABI of the GB300 (sm_103a) DeepSeek-V4 routed-MoE FFN block with
 * hyper-connections.
 *
 * The block is the FFN sublayer of docs.rs "hf2q 0.1.3 src/inference/models/deepseek4/
 * ffn_forward.rs", function forward_ffn_rows: for `rows` tokens of one layer it maps the
 * hyper-connection state f32 [rows, hc, hidden] to a new state of the same shape through
 *   hc prelude   rms_norm_no_scale_f32 -> raw_matmul "HC FFN function" -> hc_split_sinkhorn
 *                -> hc_pre -> rms_norm (ffn_norm)
 *   router       raw_matmul "MoE gate" -> score route (layer >= hash_layer_count) or hash
 *                route (layer < hash_layer_count) -> sanitize indices
 *   experts      routed + shared gate/up projections -> SwiGLU -> down projections
 *                -> weighted reduce (routed slots weighted, shared added)
 *   hc post      hc_post (post * ffn_output + comb * state)
 * Every stage runs in this library's CUDA kernels; there is no host or CPU fallback.
 *
 * Conventions where the page leaves the arithmetic open (each fixed here, not by the page):
 *   - mixes split as [pre (hc) | post (hc) | comb (hc*hc, row-major i*hc+j)]; segment s is
 *     multiplied by hc_scale[s] and then hc_base is added; pre = sigmoid, post = 2*sigmoid;
 *     comb = Sinkhorn(exp(a - rowmax)), `sinkhorn_iters` sweeps of row then column
 *     normalisation, no epsilon;
 *   - hc_post: out[i] = post[i] * ffn_output + sum_j comb[i][j] * state[j];
 *   - score route: s = sigmoid(logit); top_k experts by s + exp_probs_b, slots in descending
 *     order of that value, exact ties to the lower expert index; weights s / sum(s) over the
 *     chosen experts (no extra scaling factor);
 *   - hash route: experts = tid2eid[token] in table order; weights sigmoid(logit) normalised
 *     over the slots whose expert is valid;
 *   - sanitize: an index outside [0, experts) is replaced by 0 for the projections, and the
 *     weighted reduce gives that slot no weight;
 *   - SwiGLU: silu(gate) * up, no clamp, no bias.
 *
 * Memory: all tensor arguments are DEVICE pointers owned by the caller, row-major and
 * contiguous.  bf16 arguments are passed as uint16_t bit patterns.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (negative = error, the call did nothing on the device). */
#define MOE_FFN_OK 0
#define MOE_FFN_ERR_NULL_PTR (-1)          /* a required pointer is NULL */
#define MOE_FFN_ERR_BAD_CONFIG (-2)        /* config outside the supported shapes (see below) */
#define MOE_FFN_ERR_LAYER_RANGE (-3)       /* layer >= n_layers (the page's first guard) */
#define MOE_FFN_ERR_ROWS_ZERO (-4)         /* rows == 0 ("requires at least one token row") */
#define MOE_FFN_ERR_ROWS_RANGE (-5)        /* rows < 0, rows > max_rows, or rows*top_k overflows */
#define MOE_FFN_ERR_NO_ROUTING_SOURCE (-6) /* score layer without exp_probs_b, hash layer without tid2eid */
#define MOE_FFN_ERR_ALIAS (-7)             /* out_state overlaps state */
#define MOE_FFN_ERR_CUDA (-8)              /* a CUDA runtime/driver call failed; see moe_ffn_last_error */
#define MOE_FFN_ERR_NO_MEMORY (-9)         /* device or host allocation failed */
#define MOE_FFN_ERR_UNSUPPORTED (-10)      /* no sm_103 device */
#define MOE_FFN_ERR_ALIGNMENT (-11)        /* a pointer is not 16-byte aligned */
#define MOE_FFN_ERR_NO_WEIGHTS (-12)       /* forward on a layer whose weights were not given */

/* Device-side status bits (moe_ffn_status returns their OR since the previous call). */
#define MOE_FFN_DEV_TOKEN_RANGE 0x1   /* hash layer: token id outside [0, vocab); its slots masked */
#define MOE_FFN_DEV_ROUTE_RANGE 0x2   /* a routed expert index outside [0, experts); slot masked */
#define MOE_FFN_DEV_NONFINITE 0x4     /* a router logit, a SwiGLU output or an expert's output was NaN or infinite */
#define MOE_FFN_DEV_TIMEOUT 0x8       /* a bounded wait inside a kernel gave up (kernel returned) */

/* Shapes and constants of the block (the page's cfg fields).  Supported:
 *   1 <= hc <= 4;  128 <= hidden <= 4096, hidden % 128 == 0;  128 <= inter <= 2048, inter % 128 == 0;  shared_inter == inter;
 *   16 <= experts <= 512, experts % 16 == 0;  1 <= top_k <= 8, top_k <= experts;
 *   hash_layer_count <= n_layers;  1 <= max_rows <= 65536;  vocab >= 1;  sinkhorn_iters >= 0. */
typedef struct moe_ffn_config {
  int32_t hidden;            /* hidden_size (4096) */
  int32_t hc;                /* hyper_connection_count (4) */
  int32_t experts;           /* num_experts (256) */
  int32_t top_k;             /* num_experts_per_tok (6) */
  int32_t inter;             /* expert_intermediate_size (2048) */
  int32_t shared_inter;      /* shared expert intermediate size (= inter) */
  int32_t vocab;             /* vocab_size: token ids must lie in [0, vocab) on hash layers */
  int32_t n_layers;          /* num_hidden_layers */
  int32_t hash_layer_count;  /* layers below this use hash routing */
  int32_t max_rows;          /* largest `rows` a forward will be given; sizes the scratch */
  int32_t sinkhorn_iters;    /* Sinkhorn sweeps (20) */
  float rms_eps;             /* rms_norm_eps (1e-6) */
} moe_ffn_config;

/* Weights of one layer: DEVICE pointers, caller-owned, 16-byte aligned, valid for the life of
 * the handle.  A layer whose pointers are all NULL has no weights; forward on it fails.  The six
 * expert matrices may be NULL together (and only together): the layer's experts then come later
 * in MXFP8 (moe_ffn_set_mxfp8_experts), and a forward before that fails with NO_WEIGHTS. */
typedef struct moe_ffn_layer_weights {
  const uint16_t *hc_fn;       /* bf16 [(2+hc)*hc, hc*hidden]  hc_ffn_fn */
  const float *hc_base;        /* f32 [(2+hc)*hc]              hc_ffn_base */
  const float *hc_scale;       /* f32 [3]                      hc_ffn_scale */
  const float *ffn_norm;       /* f32 [hidden]                 ffn_norm */
  const uint16_t *gate;        /* bf16 [experts, hidden]       ffn_gate_inp (router) */
  const float *exp_probs_b;    /* f32 [experts]; required on score layers, else may be NULL */
  const int32_t *tid2eid;      /* i32 [vocab, top_k]; required on hash layers, else may be NULL */
  const uint16_t *gate_exps;   /* bf16 [experts, inter, hidden] */
  const uint16_t *up_exps;     /* bf16 [experts, inter, hidden] */
  const uint16_t *down_exps;   /* bf16 [experts, hidden, inter] */
  const uint16_t *gate_sh;     /* bf16 [shared_inter, hidden] */
  const uint16_t *up_sh;       /* bf16 [shared_inter, hidden] */
  const uint16_t *down_sh;     /* bf16 [hidden, shared_inter] */
} moe_ffn_layer_weights;

typedef struct moe_ffn_handle moe_ffn_handle;

/* Creates a handle on the current CUDA device.  Validates the config (BAD_CONFIG) and, for every
 * layer with weights, the routing source its layer type needs (NO_ROUTING_SOURCE) and pointer
 * alignment (ALIGNMENT).  Allocates the scratch for max_rows; the weights are read in place (no
 * copies: the tensor-core kernels take the bf16 matrices as they are).  Synchronous.  On failure
 * *out is NULL and nothing stays allocated. */
int moe_ffn_init(const moe_ffn_config *cfg, const moe_ffn_layer_weights *layers, moe_ffn_handle **out);

/* Enqueues the block for `rows` tokens of `layer` on `stream` (a cudaStream_t; NULL = legacy
 * default stream) and returns without waiting.
 *   state      f32 [rows, hc, hidden]  input hyper-connection state (read only)
 *   token_ids  i32 [rows]              token ids (read on hash layers only; may be NULL on score layers)
 *   out_state  f32 [rows, hc, hidden]  output state; must not overlap state
 * Returns MOE_FFN_OK or a negative code from the host-side checks (nothing enqueued then).
 * Rows <= 4 take the weight-streaming decode path; larger batches the tensor-core grouped-GEMM
 * path.  Forwards on one handle share its scratch: enqueue them on one stream (or order them),
 * never concurrently.  Data-dependent problems (a token id out of range, an expert index out of
 * range, a non-finite logit) do not fail the call: they set device status bits, masked slots
 * contribute nothing, and moe_ffn_status reports them. */
int moe_ffn_forward(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                    int32_t layer, float *out_state, void *stream);

/* Several layers in one submission: enqueues the blocks of layers first_layer .. first_layer +
 * n_layers - 1 for the same `rows` tokens on `stream`, each taking the state the previous one made:
 * state -> layer first_layer -> ... -> out_state.  A decode step's loop over layers is its unit of
 * submission (docs.rs "hf2q 0.1.10 .../deepseek4/decode_cohort.rs", forward_verifier_decode_cohort:
 * two layers per command buffer, a B=4 step encoded as four rows=1 passes per layer); here each
 * layer is one launch for all rows and the whole chain is one CUDA graph.  The chain runs FFN
 * blocks back to back; the attention sublayer a model puts between them is the caller's (every
 * entry point of this library can be captured into the caller's own graph, which is how a step
 * with attention is batched).
 * The first call for a given (state, token_ids, rows, first_layer, n_layers, out_state) captures
 * the chain into a CUDA graph that the handle owns (the 8 most recently used are kept); later calls
 * with the same arguments launch it, reading whatever the buffers then hold.  The intermediate
 * states live in a handle-owned f32 [max_rows, hc, hidden] buffer, allocated by the first call with
 * n_layers > 1.  So make the first call of each argument set outside any stream capture, and not
 * while another thread captures in global mode.  Per-kernel stage timing does not apply.
 * Returns the codes of moe_ffn_forward, checked for every layer of the chain (LAYER_RANGE also when
 * n_layers < 1 or the chain passes the last layer), NO_MEMORY or CUDA; nothing is enqueued on an
 * error. */
int moe_ffn_forward_layers(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                           int32_t first_layer, int32_t n_layers, float *out_state, void *stream);

/* The same block on HOST buffers: copies state [rows, hc, hidden] and token_ids [rows] (may be NULL
 * on score layers) from host memory into library-owned device buffers, runs moe_ffn_forward on
 * `stream`, copies the new state back into out_state (host), and waits for the stream.  Pinned
 * (page-locked) host memory gives the fastest copies.  Same return codes as moe_ffn_forward, plus
 * MOE_FFN_ERR_CUDA when a copy fails. */
int moe_ffn_forward_host(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                         int32_t layer, float *out_state, void *stream);

/* Waits for the stream of the last forward and returns the OR of device status bits set since the
 * previous moe_ffn_status call (>= 0, then cleared), or MOE_FFN_ERR_CUDA. */
int moe_ffn_status(moe_ffn_handle *h);

/* Copies to host memory an intermediate of the last forward (after waiting for it), for stage-by-
 * stage checks.  `which` selects the buffer; `bytes` must equal its size for the last `rows`:
 *   0 pre f32 [rows, hc]      1 post f32 [rows, hc]      2 comb f32 [rows, hc, hc]
 *   3 ffn_norm f32 [rows, hidden]   4 logits f32 [rows, experts]
 *   5 indices i32 [rows, top_k]     6 route weights f32 [rows, top_k]
 *   7 safe indices u32 [rows, top_k] 8 ffn_output f32 [rows, hidden]
 * Returns MOE_FFN_OK, MOE_FFN_ERR_BAD_CONFIG for an unknown `which` or a size mismatch, or
 * MOE_FFN_ERR_CUDA. */
int moe_ffn_debug_copy(moe_ffn_handle *h, int32_t which, void *host_dst, size_t bytes);

/* Per-kernel timing (off by default).  While enabled, each forward records a CUDA event on its
 * stream before its first kernel and after every kernel; this adds a few microseconds per forward. */
int moe_ffn_set_stage_timing(moe_ffn_handle *h, int32_t enable);

/* After a forward made with stage timing on: waits for it and writes the duration (ms) of each of
 * its kernels, in launch order, to ms[i] and the kernel's name (a static string) to names[i] (names
 * may be NULL).  Returns the number of kernels written (at most max_stages), 0 when nothing was
 * timed, or a negative code. */
int moe_ffn_stage_times(moe_ffn_handle *h, float *ms, const char **names, int32_t max_stages);

/* Allocation-free HC split: the first stage of the block (HC RMSNorm, mix GEMV with hc_fn, split
 * into pre/post and the Sinkhorn comb, the same kernel and conventions as moe_ffn_forward) for
 * callers that cannot allocate device memory at call time: serving or real-time loops that forbid
 * allocation after start-up (cudaMalloc may synchronise the device), or hosts whose memory pool
 * owns the whole GPU, where cudaMalloc fails.  The pages have no counterpart of this entry point;
 * it exists for such callers.
 *   state    f32 [rows, hc, hidden] (device, 16-byte aligned)    hc_fn bf16 [(2+hc)*hc, hc*hidden]
 *   hc_scale f32 [3], hc_base f32 [(2+hc)*hc]                    (device)
 *   pre, post f32 [rows, hc]; comb f32 [rows, hc, hc]            (device outputs)
 * No handle and no allocation: the scratch is a fixed 1 MiB array inside the library (held by every
 * GPU that loads the library until exit), shared by all calls; each call clears the part that
 * must start at zero (one cudaMemsetAsync on the array) before its kernel.  Limits: 1 <= rows <=
 * 4096 and rows * (partial sums of the chosen split) must fit the 1 MiB; larger inputs return
 * MOE_FFN_ERR_ROWS_RANGE with a message in moe_ffn_last_error(NULL).  The first call on each device
 * looks the array's address up (and may load the module onto that device): make it before any
 * stream capture.  Calls whose kernels overlap on the GPU race on the shared scratch: order them on
 * one stream.  Returns MOE_FFN_OK or a negative code.  A CUDA error already pending from earlier
 * work is reported as MOE_FFN_ERR_CUDA before anything is enqueued; every other negative code
 * except a failed kernel launch also means nothing was enqueued (a failed launch comes after the
 * memset). */
int moe_ffn_hc_split_noalloc(const float *state, const uint16_t *hc_fn, const float *hc_scale,
                             const float *hc_base, int32_t rows, int32_t hc, int32_t hidden,
                             int32_t sinkhorn_iters, float rms_eps, float *pre, float *post, float *comb,
                             void *stream);

/* ---- The hyper-connection prelude and post of a sublayer ------------------------------------
 * Every sublayer of a layer wraps its body in the same hyper-connection stages: the attention
 * sublayer (docs.rs "hf2q 0.1.3 src/inference/models/deepseek4/attention_forward.rs", with the "HC
 * attention function" and attn_norm) as the FFN sublayer (ffn_forward.rs, with the "HC FFN
 * function" and ffn_norm).  Before the body: RMSNorm of the flattened state (no weight), the mix
 * GEMV with the sublayer's hc_fn, split + Sinkhorn into pre/post/comb (the conventions above),
 * hc_pre (x = sum_h pre[h] * state[h]) and the sublayer's RMSNorm of x.  After the body: hc_post
 * folds the body's output f back into the state.  The FFN sublayer's HC weights come with
 * moe_ffn_init; the attention sublayer's are registered with moe_ffn_set_attn_hc. */
#define MOE_FFN_SUBLAYER_ATTN 0
#define MOE_FFN_SUBLAYER_FFN 1

/* HC weights of one sublayer: DEVICE pointers, caller-owned, 16-byte aligned. */
typedef struct moe_ffn_hc_weights {
  const uint16_t *hc_fn;   /* bf16 [(2+hc)*hc, hc*hidden]  hc_attn_fn */
  const float *hc_base;    /* f32 [(2+hc)*hc]              hc_attn_base */
  const float *hc_scale;   /* f32 [3]                      hc_attn_scale */
  const float *norm;       /* f32 [hidden]                 attn_norm */
} moe_ffn_hc_weights;

/* Registers the attention sublayer's HC weights for `layer`; they must stay valid for the life of
 * the handle, and a later call for the same layer replaces them (hc_fn is read in place, also by
 * the tensor-core mix of the many-row path).  Synchronous.  Returns MOE_FFN_OK,
 * LAYER_RANGE, NULL_PTR, ALIGNMENT, NO_MEMORY or CUDA. */
int moe_ffn_set_attn_hc(moe_ffn_handle *h, int32_t layer, const moe_ffn_hc_weights *w);

/* Enqueues the HC prelude of `sublayer` (MOE_FFN_SUBLAYER_ATTN or _FFN) of `layer` for `rows`
 * tokens on `stream` and returns without waiting.
 *   state   f32 [rows, hc, hidden]  the state entering the sublayer (read only)
 *   x_norm  f32 [rows, hidden]      out: the body's input, RMSNorm(hc_pre(state, pre)) * norm
 *   pre     f32 [rows, hc]          out; may be NULL
 *   post    f32 [rows, hc]          out, for moe_ffn_hc_post
 *   comb    f32 [rows, hc, hc]      out, for moe_ffn_hc_post (row-major i*hc + j)
 * state and x_norm must be 16-byte aligned; no output may overlap state.  Uses the handle's scratch
 * like moe_ffn_forward (order the calls on one stream).  Returns MOE_FFN_OK, LAYER_RANGE, ROWS_ZERO,
 * ROWS_RANGE, NULL_PTR, ALIGNMENT, ALIAS, BAD_CONFIG (unknown sublayer), NO_WEIGHTS (the sublayer's
 * HC weights are not there) or CUDA; nothing is enqueued on an error. */
int moe_ffn_hc_pre(moe_ffn_handle *h, int32_t layer, int32_t sublayer, const float *state, int32_t rows,
                   float *x_norm, float *pre, float *post, float *comb, void *stream);

/* Enqueues hc_post: out_state[r, i, d] = post[r, i] * f[r, d] + sum_j comb[r, i, j] * state[r, j, d].
 *   f          f32 [rows, hidden]      the sublayer body's output
 *   state      f32 [rows, hc, hidden]  the state given to moe_ffn_hc_pre
 *   post, comb f32 [rows, hc], [rows, hc, hc] from moe_ffn_hc_pre
 *   out_state  f32 [rows, hc, hidden]  must not overlap any input
 * f, state and out_state must be 16-byte aligned.  Needs no scratch.  Returns MOE_FFN_OK,
 * ROWS_ZERO, ROWS_RANGE, NULL_PTR, ALIGNMENT, ALIAS or CUDA. */
int moe_ffn_hc_post(moe_ffn_handle *h, const float *f, const float *state, const float *post, const float *comb,
                    int32_t rows, float *out_state, void *stream);

/* ---- Quantised expert weights -----------------------------------------------------------------
 * The page consumes the expert matrices as raw GGUF types without naming a format; the quantised
 * mode here reads them as MXFP8 (OCP Microscaling): E4M3 codes (1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; no infinities) in the bf16 matrices' layouts, and one E8M0 scale (2^(s-127))
 * per 32 consecutive elements of a row, so element k of a row is value(code) * 2^(scale[k/32] - 127).
 * The rest of the block is unchanged.  Rows <= 4 stream the codes and scales (about half the bytes
 * of bf16).  At four rows the decode kernel turns each tile into exact f16 weights in tensor memory
 * for the tensor cores (the batch rows go in as three f16 planes: values of magnitude 2^32 and
 * above come out infinite); that needs every scale of the layer within 22 binades of its largest
 * and no NaN code or scale, and a layer outside that, or one to three rows, decodes on the
 * CUDA-core kernel instead.  Larger batches run the tensor-core path on a bf16 expansion made at
 * registration, exact wherever code x scale is a normal bf16. */
typedef struct moe_ffn_mxfp8_experts {
  const uint8_t *gate_exps, *gate_exps_scale;  /* E4M3 [experts, inter, hidden], E8M0 [experts, inter, hidden/32] */
  const uint8_t *up_exps, *up_exps_scale;      /* the same layouts */
  const uint8_t *down_exps, *down_exps_scale;  /* E4M3 [experts, hidden, inter], E8M0 [experts, hidden, inter/32] */
  const uint8_t *gate_sh, *gate_sh_scale;      /* E4M3 [shared_inter, hidden], E8M0 [shared_inter, hidden/32] */
  const uint8_t *up_sh, *up_sh_scale;          /* the same layouts */
  const uint8_t *down_sh, *down_sh_scale;      /* E4M3 [hidden, shared_inter], E8M0 [hidden, shared_inter/32] */
} moe_ffn_mxfp8_experts;

/* Makes `layer` run on these MXFP8 experts (DEVICE pointers, caller-owned, 16-byte aligned, valid
 * for the life of the handle), in place of any bf16 experts given at init; a later call replaces
 * them.  The layer must have its other weights from moe_ffn_init.  Reads every code and scale once
 * on the device (NaN codes, the range of the scales).  On a handle with max_rows > 4 this also fills the bf16 expansion the
 * tensor-core path reads (allocating it on first use).  Synchronous.  Returns MOE_FFN_OK, LAYER_RANGE, NO_WEIGHTS, NULL_PTR, ALIGNMENT, NO_MEMORY or CUDA. */
int moe_ffn_set_mxfp8_experts(moe_ffn_handle *h, int32_t layer, const moe_ffn_mxfp8_experts *w);

/* Test hook: failure detection without a GPU fault.  Every wait inside the kernels is bounded; on
 * expiry a kernel sets MOE_FFN_DEV_TIMEOUT, stops its work, waits (bounded) for its own copies and
 * tensor-core operations in flight, frees its tensor memory and returns, leaving the handle usable.
 * This call makes one such wait run out on purpose, on the handle's later forwards:
 *   which = MOE_FFN_INJECT_DECODE_WAIT: rows <= 4, the decode kernel's final phase first waits for
 *           a count that nothing reaches;
 *   which = MOE_FFN_INJECT_GEMM_WAIT:   rows > 4, CTA 0 of the gate/up GEMM first waits on an
 *           mbarrier that nothing arrives at;
 *   which = MOE_FFN_INJECT_NONE:        no injected wait (the default).
 * wait_limit_us bounds every in-kernel wait of those forwards (0: the kernels' defaults, 1-2 s).
 * Outputs of a forward with an injected wait are not meaningful; its status carries the timeout bit.
 * Returns MOE_FFN_OK, NULL_PTR or BAD_CONFIG.  Nothing in the pages corresponds to it. */
#define MOE_FFN_INJECT_NONE 0
#define MOE_FFN_INJECT_DECODE_WAIT 1
#define MOE_FFN_INJECT_GEMM_WAIT 2
int moe_ffn_set_fault_injection(moe_ffn_handle *h, int32_t which, uint32_t wait_limit_us);

/* Text of the last error on this handle, or, when h is NULL, of the last failed call made without
 * a handle (init, the allocation-free split, a NULL handle) on the calling thread: that message
 * is kept per thread, so threads that fail at the same time do not overwrite each other's text.
 * The pointer stays valid until the same handle (or, for NULL, the same thread) fails again. */
const char *moe_ffn_last_error(const moe_ffn_handle *h);

/* Waits for outstanding work, frees everything the handle owns.  NULL is ignored. */
void moe_ffn_destroy(moe_ffn_handle *h);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FFN_H */
