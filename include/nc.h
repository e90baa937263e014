/*
 * nc.h -- C ABI of the B300 (sm_103a) forward pass of a nanochat-style
 * decoder-only GPT.
 *
 * What the forward computes (web pages cited by title and section):
 *
 *  - "Nanochat在nanoGPT之上的新增功能" (what nanochat adds over nanoGPT),
 *    section 1 feature table and the notes under it: rotary position
 *    embedding and no position table; RMSNorm without learned parameters;
 *    squared-ReLU MLP; separate q, k, v and output projections, no biases;
 *    grouped-query attention; q and k RMS-normalised after RoPE; logits
 *    soft-capped by tanh to (-15, 15); per-layer sliding windows, three
 *    short (a quarter of the context) then one full, the last layer always
 *    full; value embeddings added to v through a gate on alternating layers
 *    including the last; smear (the previous token's embedding mixed in
 *    through a sigmoid gate); backout (a lambda times the residual stream
 *    cached at mid depth is subtracted before the final norm); per-layer
 *    resid_lambdas / x0_lambdas; untied embedding and lm_head.
 *  - "NanoChat基础训练报告" (NanoChat base-training report), section
 *    "模型架构": the d12 shape (12 layers, 768 wide, 6 heads of 128, 6 kv
 *    heads, 32,768 vocabulary, value embeddings with a learned gate on the
 *    odd layers).
 *  - "nanochat — 架构与原理" (nanochat architecture and principles), section
 *    2 component table: GPT.forward(idx) maps token ids to logits; the
 *    attention backend and the FP8 path it lists are prior art here.
 *
 * Readings of what the pages leave open (all fixed by nc_config fields):
 *  - RMSNorm is x / sqrt(mean(x^2) + rms_eps).
 *  - RoPE pairs channel d with d + head_dim/2, angle pos * rope_base^(-2d/D),
 *    y1 = x1 cos + x2 sin, y2 = -x1 sin + x2 cos; positions restart at 0 in
 *    every batch row (no document mask).
 *  - Window W (window_left[i] >= 0): query i sees keys max(0, i-W) .. i.
 *    window_left[i] < 0: plain causal.
 *  - GQA: query head h reads kv head h / (n_head / n_kv_head).
 *  - Smear gate: sigmoid(e_t[:c_s] . smear_gate), one scalar per token,
 *    times the previous token's (pre-smear) embedding; the first token of a
 *    row is unchanged.  The smeared embedding is x0.
 *  - Value-embedding gate: ve_gate_scale * sigmoid(a_t[:c_g] . ve_gate[g])
 *    per token and kv head g, a_t the block's normalised input;
 *    v <- v + gate * ve_table[token].  The product a_t . ve_gate[g] runs on
 *    the tensor cores with the q|k|v projection, from the same bf16 copy of
 *    the block input as q, k and v.
 *  - x <- resid_lambdas[i] * x + x0_lambdas[i] * x0 at the start of block i.
 *  - Backout caches x after block n_layer/2 - 1 (x0 when n_layer == 1).
 *
 * Numerics: bf16 weights and activations into the tensor cores, fp32
 * accumulation, fp32 residual stream, fp32 softmax statistics.
 *
 * Threading: a model is not re-entrant; calls on one model must not overlap.
 *
 * Devices: a model belongs to the device that was current when nc_model_create ran (its
 * packed buffer lives there); every call that launches work on it must be made with that
 * device current, else it returns NC_ERR_INVALID_ARG before any device work.  Kernel set-up
 * (shared-memory limits, occupancy) is done once per device, so one process may run models
 * on several GPUs.
 */
#ifndef NC_H
#define NC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NC_API __attribute__((visibility("default")))
#else
#define NC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NC_OK = 0,
  NC_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, inconsistent shape */
  NC_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. head_dim not 64/128) */
  NC_ERR_WORKSPACE = 3,       /* caller buffer smaller than the size query returned */
  NC_ERR_CUDA = 4,            /* a CUDA runtime call failed */
  NC_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait ran out (kernel returned early) */
  NC_ERR_TOKEN_RANGE = 6      /* a token id outside [0, vocab_size); that row used zeros */
} nc_status;

/* Model hyper-parameters.  Host memory; copied by nc_model_create. */
typedef struct {
  int n_layer;
  int n_embd;                 /* C; must equal n_head * head_dim; multiple of 128 */
  int n_head;                 /* H */
  int n_kv_head;              /* Hkv; divides n_head */
  int head_dim;               /* D: 64 or 128 */
  int mlp_hidden;             /* F; multiple of 64 */
  int vocab_size;             /* V; multiple of 64 */
  int seq_len_ctx;            /* largest T accepted by nc_forward */
  const int *window_left;     /* [n_layer]; < 0 = full causal */
  const unsigned char *has_ve;/* [n_layer]; nonzero = value-embedding layer */
  int use_smear;
  int use_backout;
  int embed_norm;             /* RMSNorm the token embedding before smear (default 0) */
  int smear_gate_channels;    /* c_s, 0 = n_embd */
  int ve_gate_channels;       /* c_g, 0 = n_embd; multiple of 8 */
  float ve_gate_scale;        /* default 1 */
  float rms_eps;              /* default 1e-6 */
  float rope_base;            /* default 10000 */
  float softcap;              /* default 15 */
  int logits_bf16;            /* 0: logits are fp32 (default); 1: bf16 (the same soft-capped values
                                 rounded to nearest even: half the bytes to write and to copy out) */
  int fp8;                    /* 0: bf16 linear layers (default); 1: every linear layer (q, k, v, output
                                 projection, MLP up and down projections, lm_head) in e4m3 with
                                 tensorwise scales, see nc_forward; needs mlp_hidden % 128 == 0 */
} nc_config;

/* Weights.  Matrices are bf16, row-major in the nn.Linear layout [out, in],
 * in device memory.  BORROWED: they must outlive the model.  Per-layer
 * arrays are host arrays of n_layer device pointers; entries of ve_table and
 * ve_gate are ignored (may be NULL) on layers without value embeddings. */
typedef struct {
  const void *wte;                    /* [V, C] */
  const void *const *wq;              /* [H*D, C] per layer */
  const void *const *wk;              /* [Hkv*D, C] */
  const void *const *wv;              /* [Hkv*D, C] */
  const void *const *wo;              /* [C, H*D] */
  const void *const *wfc;             /* [F, C] */
  const void *const *wproj;           /* [C, F] */
  const void *const *ve_table;        /* [V, Hkv*D] */
  const void *const *ve_gate;         /* [Hkv, c_g] */
  const void *smear_gate;             /* [c_s]; unused if !use_smear */
  const void *lm_head;                /* [V, C] */
  const float *resid_lambdas;         /* host [n_layer], copied */
  const float *x0_lambdas;            /* host [n_layer], copied */
  float backout_lambda;
} nc_weights;

typedef struct nc_model nc_model;

/* Size in bytes of the device buffer nc_model_create fills with the packed
 * q|k|v weights, the rotary table for seq_len_ctx positions and the device
 * status word.  Host-only; validates the config. */
NC_API nc_status nc_model_packed_bytes(const nc_config *cfg, size_t *bytes);

/* Validate cfg, copy it, pack W_q|W_k|W_v of each layer into packed_buf
 * (device, >= nc_model_packed_bytes, 256-byte aligned, caller-owned, must
 * outlive the model) and fill the rotary table, on `stream`
 * (cudaStream_t; NULL = legacy default stream).  The model itself owns only
 * host state.  On error *out is NULL. */
NC_API nc_status nc_model_create(const nc_config *cfg, const nc_weights *w, void *packed_buf,
                          size_t packed_bytes, void *stream, nc_model **out);

/* Device workspace needed by nc_forward for a [B, T] batch.  Host-only. */
NC_API nc_status nc_workspace_bytes(const nc_model *m, int B, int T, size_t *bytes);

/* Forward pass: tokens (device int32 [B, T]) -> logits (device [B, T, V], row-major, fp32 or,
 * with cfg.logits_bf16, bf16), soft-capped.  Asynchronous on `stream`; argument
 * errors are returned synchronously before any device work; device-side
 * errors (token range, wait timeout) are recorded in the status word and
 * returned by nc_get_status.  workspace: device, >= nc_workspace_bytes,
 * 256-byte aligned, caller-owned; T <= seq_len_ctx. */
NC_API nc_status nc_forward(nc_model *m, const int32_t *tokens, int B, int T, void *logits,
                     void *workspace, size_t ws_bytes, void *stream);

/* Same forward with HOST buffers: copies tokens (host int32 [B, T]) in,
 * runs nc_forward, copies logits (host [B, T, V], fp32 or bf16 as nc_forward) out and synchronises
 * `stream`.  Staging areas live in `workspace`, sized by
 * nc_workspace_bytes_host.  Pinned host memory gives full copy bandwidth. */
NC_API nc_status nc_workspace_bytes_host(const nc_model *m, int B, int T, size_t *bytes);
NC_API nc_status nc_forward_host(nc_model *m, const int32_t *tokens_host, int B, int T,
                          void *logits_host, void *workspace, size_t ws_bytes, void *stream);

/* Forward pass for callers that cannot allocate device memory when they run the model
 * (for example code hosted by a framework that owns all device memory through its own pool
 * and forbids raw cudaMalloc, or a latency-bound serving loop where cudaMalloc/cudaFree
 * would synchronise the device).  The source pages have no counterpart to this call; it
 * only changes where the forward's scratch lives.
 *
 * Identical to nc_forward, except that the activation scratch is a fixed array of
 * NC_STATIC_SCRATCH_BYTES built into the library (every GPU that loads the library keeps
 * it reserved until the process exits) instead of a caller workspace.  The caller passes
 * only the model, tokens (device int32 [B, T]) and logits (device [B, T, V], as nc_forward).
 *  - Limit: returns NC_ERR_WORKSPACE, before any device work, when nc_workspace_bytes(B, T)
 *    exceeds NC_STATIC_SCRATCH_BYTES (at d12 width that is roughly 1,400 tokens per call).
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.  Keep
 *    per-kernel timing (nc_timing_enable) off, since it creates CUDA events.
 *  - The first call on each device looks up the array's device address with that device
 *    current.  With CUDA's lazy module loading (the default) that first call is also when
 *    the library's device code is loaded on the device and the array is reserved, so it can
 *    fail with NC_ERR_CUDA if the device is short of memory: make it at set-up time, and
 *    before any stream capture.
 *  - All calls share the one array, which keeps the previous call's contents (nothing in it
 *    needs to start at zero: every region is written before it is read within one call).
 *    Calls that overlap on the GPU (other streams, other models, other threads) race on it:
 *    serialise them. */
#define NC_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
NC_API nc_status nc_forward_static_scratch(nc_model *m, const int32_t *tokens, int B, int T,
                                           void *logits, void *stream);

/* ---- loss path: fused lm_head + soft-cap + next-token cross-entropy, no logits ----
 * "nanochat — 架构与原理", section 2 component table (metrics row: bits per byte from the
 * loss evaluation) and "NanoChat基础训练报告", loss progression table (training loss and
 * validation bits per byte).  The forward is that of nc_forward up to the final norm; the
 * lm_head GEMM then keeps, per row and 128-column group, the sum of exp(logit) and the
 * target's logit instead of writing the [B, T, V] logits, and two small kernels reduce them:
 *   loss[b, t] = log(sum_v exp(z[b, t, v])) - z[b, t, targets[b, t]]      (nats)
 * with z the soft-capped logits of nc_forward.  A negative target marks an ignored position
 * (loss 0, not counted); a target >= V is recorded as NC_ERR_TOKEN_RANGE in the status word
 * and ignored the same way.
 *   stats[0] = mean loss over the counted positions (NaN if there are none);
 *   stats[1] = bits per byte: the summed loss of the positions whose target has a nonzero
 *              byte count, over ln 2 times the sum of those byte counts (NaN without
 *              token_bytes or when no counted target has bytes).
 * targets: device int32 [B, T], the token each position predicts (the caller shifts);
 * token_bytes: device int32 [V] byte length of each vocabulary entry, or NULL;
 * loss: device fp32 [B, T], or NULL; stats: device fp32 [2].  Both statistics are reduced in
 * fp64 in a fixed order (bitwise repeatable).  workspace: device, >= nc_workspace_bytes_loss,
 * 256-byte aligned, caller-owned.  Asynchronous on `stream`, errors as nc_forward. */
NC_API nc_status nc_workspace_bytes_loss(const nc_model *m, int B, int T, size_t *bytes);
NC_API nc_status nc_forward_loss(nc_model *m, const int32_t *tokens, const int32_t *targets, int B, int T,
                                 const int32_t *token_bytes, float *loss, float *stats, void *workspace,
                                 size_t ws_bytes, void *stream);

/* ---- Backward, first part: the gradient of the mean loss at the tail of the network ----
 * "NanoChat基础训练报告", performance section (the training step the pages measure) and loss
 * progression table (the training loss); "Nanochat在nanoGPT之上的新增功能", section 1 table and
 * notes (untied lm_head, logit soft-cap, final RMSNorm, backout, ReLU^2 MLP).  The loss is that of
 * nc_forward_loss: the mean over counted positions (target in [0, V)) of the cross-entropy of the
 * soft-capped logits.  nc_forward_loss_grad_tail runs that loss path and then the backward as far
 * as the last block's attention output projection, writing the exact gradient of the mean loss
 * (up to rounding) with respect to four weights, fp32, row-major like the weights themselves:
 *   grad_lm_head [V, C]        the lm_head
 *   grad_wproj   [C, F]        the last block's MLP down projection (c_proj)
 *   grad_wfc     [F, C]        the last block's MLP up projection (c_fc)
 *   grad_wo      [C, H * D]    the last block's attention output projection (c_proj)
 * Each is overwritten (not accumulated).  The last block's weights get no gradient through the
 * backout term: the backed-out stream is that of block n_layer/2 - 1 (or x0), never the last
 * block's.  stats: device fp32 [2] as nc_forward_loss (mean loss, bits per byte with token_bytes);
 * token_bytes may be NULL.  The lm_head is evaluated twice (once for the log-sum-exp of each row,
 * once for the gradient), so no logits are stored; the gradient at the lm_head's pre-cap output is
 * rounded to bf16 before the two products that use it, as the forward's activations are.  tokens,
 * targets: device int32 [B, T]; gradients: device, 16-byte aligned, caller-owned; workspace: device,
 * >= nc_workspace_bytes_grad_tail (the loss path's plus about M * (2 V + 2 F + 18 C) bytes), 256-byte
 * aligned.  Asynchronous on `stream`; errors as nc_forward.  nc_grad_tail_launch_count gives the
 * kernels one call launches (5 * n_layer + 14). */
NC_API nc_status nc_workspace_bytes_grad_tail(const nc_model *m, int B, int T, size_t *bytes);
NC_API nc_status nc_forward_loss_grad_tail(nc_model *m, const int32_t *tokens, const int32_t *targets, int B, int T,
                                           const int32_t *token_bytes, float *stats, float *grad_lm_head,
                                           float *grad_wproj, float *grad_wfc, float *grad_wo, void *workspace,
                                           size_t ws_bytes, void *stream);

/* ---- KV cache: prefill + single-token decode ----
 * "nanochat — 架构与原理", section 2 component table (inference engine: KV cache and sampling)
 * and section 7 code map (Engine, KVCache); "Nanochat在nanoGPT之上的新增功能", section 1 table
 * and notes (per-layer sliding windows, GQA).  The cache keeps, per layer and batch row, the
 * post-RoPE, post-QK-norm keys and the values (value embedding included) of the positions the
 * layer can still attend to: all T_max positions on full layers, the last W+1 on a layer with
 * window W (position j in slot j % (W+1)).  Layout per layer: keys then values, each
 * [B][cap][Hkv*D] bf16, 256-byte aligned; the caller owns the buffer (>= nc_kv_cache_bytes,
 * 256-byte aligned) and T_max <= seq_len_ctx.
 *
 * nc_prefill: nc_forward over tokens [B, T] (T <= T_max) that also fills the cache with
 * positions 0..T-1; logits [B, T, V] (fp32 or bf16 as nc_forward); workspace as nc_forward
 * (nc_workspace_bytes(B, T)).
 *
 * nc_decode_step: one new token per batch row, all at position pos (1 <= pos < T_max):
 * tokens (device int32 [B]) are the tokens at pos, prev_tokens those at pos - 1 (the smear
 * reads the previous token's embedding); appends the new keys and values at pos and writes the
 * logits of position pos, [B, V] (fp32 or bf16 as nc_forward).  The result equals row pos of
 * nc_forward over the whole sequence up to rounding: the step's products accumulate in another
 * order, and its attention keeps p in fp32 where the batched one rounds it to bf16.  workspace:
 * >= nc_workspace_bytes_decode(B), 256-byte aligned.  A step runs the embedding, per layer the
 * q|k|v product, the attention (q|k|v epilogue, cache append, split attention and its combine in
 * one launch), the out-projection, fc and down-projection products, then the lm_head: each
 * product a small-row kernel that reads every weight once.
 * Both are asynchronous on `stream`; errors as nc_forward.  nc_kv_launch_count gives the kernels a
 * decode step launches (2 + 5 * n_layer; a prefill launches 2 + 6 * n_layer).  After a first call on
 * the device (per-device kernel set-up), nc_forward and nc_decode_step make no host synchronisation
 * or allocation, so a caller can capture them in a CUDA graph. */
NC_API nc_status nc_kv_cache_bytes(const nc_model *m, int B, int T_max, size_t *bytes);
NC_API nc_status nc_prefill(nc_model *m, const int32_t *tokens, int B, int T, void *kv_cache, size_t cache_bytes,
                            int T_max, void *logits, void *workspace, size_t ws_bytes, void *stream);
NC_API nc_status nc_workspace_bytes_decode(const nc_model *m, int B, size_t *bytes);
NC_API nc_status nc_decode_step(nc_model *m, const int32_t *prev_tokens, const int32_t *tokens, int B, int pos,
                                void *kv_cache, size_t cache_bytes, int T_max, void *logits, void *workspace,
                                size_t ws_bytes, void *stream);
NC_API int nc_kv_launch_count(const nc_model *m);

/* Synchronise `stream`, read and clear the device status word. */
NC_API nc_status nc_get_status(nc_model *m, void *stream);

NC_API const char *nc_status_string(nc_status s);

/* Name of the CUDA runtime error behind the most recent NC_ERR_CUDA returned to the calling
 * thread by any nc_* call ("cudaSuccess" if there was none).  Host-only. */
NC_API const char *nc_last_cuda_error(void);

/* Frees host state only (the caller owns every device buffer). */
NC_API void nc_model_destroy(nc_model *m);

/* ---- per-kernel timing (CUDA events recorded on the launch stream) ---- */

/* Kernel classes timed when timing is enabled. */
typedef enum {
  NC_K_EMBED = 0,     /* embedding gather + smear + first block's residual mix */
  NC_K_QKV = 1,       /* q|k|v GEMM: input RMSNorm, RoPE, QK-norm, value-embedding gate */
  NC_K_ATTN = 2,      /* windowed causal GQA attention */
  NC_K_OPROJ = 3,     /* attention output projection + residual add (+ next norm's inputs) */
  NC_K_FC = 4,        /* MLP up projection: input RMSNorm + squared ReLU */
  NC_K_PROJ = 5,      /* MLP down projection + residual add, next block's mix / backout */
  NC_K_LMHEAD = 6,    /* lm_head GEMM: final RMSNorm + tanh soft-cap (+ cross-entropy partials) */
  NC_K_LOSS = 7,      /* cross-entropy reduction of the loss path */
  NC_K_LMHEAD_GRAD = 8, /* backward: lm_head output gradient, its input and weight gradients */
  NC_K_MLP_GRAD = 9,  /* backward: the last block's MLP gradient products */
  NC_K_OPROJ_GRAD = 10, /* backward: the last block's attention output projection weight gradient */
  NC_K_RMS_GRAD = 11, /* backward: RMSNorm backward (+ residual gradient) */
  NC_K_QUANT = 12,    /* 8-bit path: tensorwise amax and e4m3 quantisation of a layer's input */
  NC_K_COUNT = 13
} nc_kernel_class;

/* enable != 0: every following nc_forward records an event pair around each
 * launch; nc_timing_read sums them (syncs the events) and resets. */
NC_API nc_status nc_timing_enable(nc_model *m, int enable);
NC_API nc_status nc_timing_read(nc_model *m, nc_kernel_class k, double *total_ms, int *launches);
NC_API const char *nc_kernel_class_name(nc_kernel_class k);

/* Number of kernels one nc_forward (nc_forward_loss) launches for this model. */
NC_API int nc_forward_launch_count(const nc_model *m);
NC_API int nc_forward_loss_launch_count(const nc_model *m);
NC_API int nc_grad_tail_launch_count(const nc_model *m);

#ifdef __cplusplus
}
#endif

#endif /* NC_H */
