/*
 * nc_ops.h -- per-kernel entry points of libnc.so.
 *
 * The same kernels nc_forward launches, exposed one by one so that each can be
 * checked against the step it implements.  All pointers are DEVICE pointers
 * owned by the caller; all calls are asynchronous on `stream` (cudaStream_t,
 * NULL = legacy default stream) and return NC_ERR_INVALID_ARG / _UNSUPPORTED
 * synchronously, before any device work, for bad arguments, NC_ERR_CUDA if a
 * launch fails.  `status` (device int32, may be NULL) receives device-side
 * errors (first error wins).  Matrices are row-major; bf16 unless stated.
 * Definitions are those of nc.h (sources cited there by page title and
 * section).
 */
#ifndef NC_OPS_H
#define NC_OPS_H

#include "nc.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NC_EPI_BF16 = 0,        /* out bf16 [M, ldo] = acc */
  NC_EPI_RELU2_BF16 = 2,  /* out bf16 = relu(rs * acc)^2     (squared-ReLU row of the feature table) */
  NC_EPI_SOFTCAP_F32 = 3, /* out fp32 = cap*tanh(rs * acc/cap) (logit soft-cap row of the feature table) */
  NC_EPI_SOFTCAP_BF16 = 6, /* out bf16 = the same, rounded to nearest even */
  NC_EPI_F32 = 7           /* out fp32 = rs * acc (the backward's weight and input gradients) */
} nc_epilogue;

/* Partial sums of squares ("ssp"): fp32 [M, C/128]; ssp[m, g] = sum of x[m, c]^2 over the 128
 * columns c of group g.  A consumer turns them into the RMSNorm row scale
 * rs[m] = 1 / sqrt(sum_g ssp[m, g] / C + eps), so that norm(x) W^T = rs * (x W^T). */

/* acc[M, N] = A[M, K] . B[N, K]^T (tcgen05, fp32 accumulation), then the epilogue; rs from
 * `ssp` over C columns (ssp == NULL: rs = 1).  K % 64 == 0, N % 32 == 0, ldo >= N, rows 16-byte
 * aligned.  (nc_op_gemm_t below adds operand layouts and ragged K.) */
NC_API nc_status nc_op_gemm(const void *A, const void *B, int M, int N, int K, nc_epilogue epi,
                            void *out, int ldo, const float *ssp, int C, float eps, float cap,
                            int *status, void *stream);

/* Residual-stream update of an output projection, N = C columns (C % 128 == 0):
 *   xr = resid + A . B^T;  xm_out <- xr (if non-NULL);  x' = a * xr + b * Y (Y may be NULL);
 *   x_out <- x' (if non-NULL; may equal resid);  xb <- bf16(x');  ssp <- partial sums of x'^2.
 * resid, Y, x_out, xm_out fp32 [M, C]; xb bf16 [M, C]. */
NC_API nc_status nc_op_gemm_residual(const void *A, const void *B, int M, int N, int K,
                                     const float *resid, float a, float b, const float *Y,
                                     float *x_out, float *xm_out, void *xb, float *ssp, int *status,
                                     void *stream);

/* Rows that follow each kv head's v rows in a value-embedding layer's packed q|k|v weight. */
#define NC_QKV_GATE_ROWS 16

/* Packed q|k|v projection of a block: acc = xb[M, C] . wqkv[N, C]^T scaled by the input RMSNorm
 * row scale rs (from ssp), split into q [M, H*D], k [M, Hkv*D], v [M, Hkv*D] (bf16).
 * q and k: RoPE at position (row % T) from `rope` (see nc_op_rope_table; rope_ld = its
 * position count, >= T), then RMSNorm over each head (eps).
 * vgate == 0: wqkv rows are W_q (H*D), W_k (Hkv*D), W_v (Hkv*D); N = (H + 2 Hkv) D.
 * vgate != 0 (a value-embedding layer): wqkv rows are W_q, W_k, then for each kv head g its D rows
 * of W_v, then one row holding the gate weights ve_gate[g] (zero beyond c_g) and
 * NC_QKV_GATE_ROWS - 1 zero rows; N = (H + Hkv) D + Hkv (D + NC_QKV_GATE_ROWS).  Then
 * v[:, g] += gate_scale * sigmoid(rs * (xb . gate row g)) * ve[tokens[m], g*D:(g+1)*D]
 * (ve bf16 [V, Hkv*D]); out-of-range tokens add nothing. */
NC_API nc_status nc_op_qkv(const void *xb, const void *wqkv, int M, int T, int C, int H, int Hkv,
                           int D, const float *rope, int rope_ld, float eps, const float *ssp,
                           int vgate, float gate_scale, const void *ve, const int32_t *tokens,
                           int V, void *q, void *k, void *v, int *status, void *stream);

/* rope[i][t] = (cos, sin)(t * base^(-2i/D)), i < D/2, t < T, fp32 pairs, position fastest
 * (angles in fp64). */
NC_API nc_status nc_op_rope_table(float *rope, int T, int D, float base, void *stream);

/* Windowed causal GQA attention: q [B*T, H*D], k, v [B*T, Hkv*D] -> y [B*T, H*D] (bf16);
 * window < 0 = plain causal; D in {64, 128}. */
NC_API nc_status nc_op_attention(const void *q, const void *k, const void *v, int B, int T, int H,
                                 int Hkv, int D, int window, void *y, int *status, void *stream);

/* x0[b*T+t] = e_t + sigmoid(e_t[:c_s] . smear_gate) * e_{t-1} (t >= 1, same row b), e = wte[token]
 * (RMS-normalised first if embed_norm); smear_gate NULL = no smear.  Then x = a * x0, xb = bf16(x)
 * and ssp = partial sums of x^2.  Out-of-range tokens give a zero embedding and NC_ERR_TOKEN_RANGE
 * in *status.  x0, x fp32 [B*T, C]. */
NC_API nc_status nc_op_embed_smear(const int32_t *tokens, int B, int T, const void *wte, int V,
                                   int C, const void *smear_gate, int c_s, int embed_norm,
                                   float eps, float a, float *x0, float *x, void *xb, float *ssp,
                                   int *status, void *stream);

/* Fused lm_head + soft-cap + cross-entropy partials (the loss path of nc_forward_loss): with
 * z = cap * tanh(rs * (xf . wlm^T) / cap) (rs from ssp over C columns, as nc_op_gemm), for each
 * row m and 128-column group g of the V columns:
 *   part[g * M + m] = sum over the group's columns v of exp(z[m, v])     (group-major)
 *   zt[m] = z[m, targets[m]] when 0 <= targets[m] < V (not written otherwise).
 * xf bf16 [M, C], wlm bf16 [V, C]; part fp32 [ceil(V/128) * M]; zt, targets [M].  C % 64 == 0,
 * V % 32 == 0. */
NC_API nc_status nc_op_lmhead_ce(const void *xf, const void *wlm, int M, int V, int C, const float *ssp,
                                 float eps, float cap, const int32_t *targets, float *part, float *zt,
                                 int *status, void *stream);

/* Cross-entropy from the partials of nc_op_lmhead_ce: loss[m] and stats[2] exactly as
 * nc_forward_loss defines them (loss may be NULL; token_bytes device int32 [V] or NULL).
 * lse (NULL or fp32 [M]) receives log sum_v exp(z[m, v]) of each counted row (0 on ignored rows),
 * inv_count (NULL or one fp32) 1 / (rows counted), 0 when none is: the inputs of
 * nc_op_lmhead_ce_grad.  scratch: device, >= nc_op_ce_scratch_bytes(M), 8-byte aligned. */
NC_API size_t nc_op_ce_scratch_bytes(int M);
NC_API nc_status nc_op_ce_finalize(const float *part, const float *zt, const int32_t *targets, int M, int V,
                                   const int32_t *token_bytes, float *loss, float *stats, void *scratch,
                                   size_t scratch_bytes, float *lse, float *inv_count, int *status, void *stream);

/* ---- Backward pieces (nc_forward_loss_grad_tail chains them) ---- */

/* nc_op_gemm with operand layouts: a_mn = 0 reads A as [M][K] (K contiguous), a_mn = 1 as [K][M]
 * (M contiguous, i.e. A^T stored row-major); b_mn likewise for B ([N][K] or [K][N]).  A weight
 * gradient dW = G^T X of token-major G [T][N_out] and X [T][N_in] is (a_mn, b_mn) = (1, 1) with
 * K = T; an input gradient dX = G W of a weight W [N_out][N_in] is (0, 1).  K need not be a
 * multiple of 64; K % 8 == 0 when either operand is K-contiguous, M % 8 (N % 8) == 0 for an
 * M- (N-) contiguous one.  Epilogues as nc_op_gemm (bf16, relu2_bf16, softcap_f32, softcap_bf16,
 * f32). */
NC_API nc_status nc_op_gemm_t(const void *A, const void *B, int M, int N, int K, int a_mn, int b_mn,
                              nc_epilogue epi, void *out, int ldo, const float *ssp, int C, float eps, float cap,
                              void *split_ws, size_t split_ws_bytes, int *status, void *stream);

/* Split over K of an NC_EPI_F32 product (weight gradients: few output tiles, K = tokens): with
 * split_ws non-NULL (device, 16-byte aligned, >= nc_op_gemm_split_ws_bytes bytes, which is 0 when
 * the shape is not split) nc_op_gemm_t cuts the k-blocks into ranges that fill the device, writes
 * each range's fp32 partial product to its own slab of split_ws and adds the slabs in a fixed order
 * into out (a second kernel), so repeated calls are bit-identical. */
NC_API size_t nc_op_gemm_split_ws_bytes(int M, int N, int K, int ldo);

/* Gradient of the mean cross-entropy at the lm_head's pre-cap output, the logits recomputed
 * (nothing stored between the passes): with u = rs * (xf . wlm^T) (rs from ssp over C columns, as
 * nc_op_lmhead_ce) and z = cap * tanh(u / cap),
 *   out[m, v] = rs * inv_count * (exp(z[m, v] - lse[m]) - [v == targets[m]]) * (1 - (z[m, v] / cap)^2)
 * in bf16 [M, ldo]; rows whose target lies outside [0, V) are zero.  lse and inv_count as written
 * by nc_op_ce_finalize.  The row scale rs is kept in the output because the weight gradient
 * needs it: dW_lm = out^T . xf, and dL/dxf-hat = out . wlm / rs. */
NC_API nc_status nc_op_lmhead_ce_grad(const void *xf, const void *wlm, int M, int V, int C, const float *ssp,
                                      float eps, float cap, const int32_t *targets, const float *lse,
                                      const float *inv_count, void *out, int ldo, int *status, void *stream);

/* Backward of the MLP's squared ReLU through its down projection: with w the down projection's
 * weight [C][F] (nn.Linear [out][in]) and h = relu(u)^2 [M, F] bf16 the forward's hidden layer,
 *   out[m, f] = rs[m] * (dy[m, :] . w[:, f]) * 2 sqrt(h[m, f])        (bf16 [M, F])
 * i.e. the gradient at u scaled by the MLP input's RMSNorm row scale rs (from ssp over C columns;
 * NULL: 1), the operand of the up projection's weight gradient. dy bf16 [M, C]. */
NC_API nc_status nc_op_mlp_hidden_grad(const void *dy, const void *w, int M, int F, int C, const float *ssp,
                                       float eps, const void *h, void *out, int *status, void *stream);

/* Backward of the weightless RMSNorm xn = rs * x, rs = 1 / sqrt(mean(x^2) + eps) (from the
 * forward's partial sums ssp [M, C / 128] of x^2): given G = rs * dL/dxn (fp32 [M, C]),
 *   dx = G - rs^2 * x * mean(G * x)  (+ add [M, C] fp32 if non-NULL),
 * written to dx_f32 (fp32, if non-NULL) and dx_b16 (bf16, if non-NULL).  C % 128 == 0, C <= 2048. */
NC_API nc_status nc_op_rms_backward(const float *G, const float *x, const float *ssp, const float *add, int M,
                                    int C, float eps, float *dx_f32, void *dx_b16, void *stream);

/* ---- 8-bit (e4m3) tensorwise quantisation and product (the fp8 path of nc_forward) ---- */

/* q = e4m3(v * s) with s = 448 / max|v| over the whole [M, C] tensor (s = 1 if it is all zero),
 * round to nearest even, saturating at +-448; v = src[m, c] (bf16, or fp32 with src_f32), times the
 * row's RMSNorm scale 1 / sqrt(sum_g ssp[m, g] / C + eps) when ssp (fp32 [M, C / 128]) is given.
 * dst: e4m3 bytes [M, C], 8-byte aligned; inv_scale: one fp32, receives 1 / s.  scratch: device,
 * >= nc_op_fp8_scratch_bytes() bytes, 4-byte aligned.  C % 8 == 0 (C % 128 == 0 with ssp). */
NC_API size_t nc_op_fp8_scratch_bytes(void);
NC_API nc_status nc_op_fp8_quantize(const void *src, int src_f32, int M, int C, const float *ssp, float eps,
                                    void *dst, float *inv_scale, void *scratch, void *stream);

/* acc[M, N] = A8[M, K] . B8[N, K]^T of e4m3 operands (tcgen05 kind::f8f6f4, fp32 accumulation),
 * dequantised by inv_sa[0] * inv_sb[0] (device fp32 scalars), then the epilogue (NC_EPI_BF16,
 * NC_EPI_RELU2_BF16, NC_EPI_SOFTCAP_F32, NC_EPI_SOFTCAP_BF16 or NC_EPI_F32; no row scale).
 * K % 16 == 0, N % 32 == 0, ldo >= N, 16-byte aligned rows. */
NC_API nc_status nc_op_gemm_fp8(const void *A8, const void *B8, int M, int N, int K, nc_epilogue epi, void *out,
                                int ldo, const float *inv_sa, const float *inv_sb, float cap, int *status,
                                void *stream);

/* Test of the bounded device-side waits (failure detection without a GPU fault): the GEMM of
 * nc_op_gemm with NC_EPI_BF16, every wait of the launch limited to limit_ns (1e5 .. 1e8 ns), and the
 * tensor-core issuer withholding the "accumulator ready" signal of pair tile skip_tile (pair tiles
 * are 256 x 256 output blocks, numbered along the columns first).  The epilogue waiting for that
 * tile runs out of time: the kernel records NC_ERR_DEVICE_TIMEOUT in *status (device int32,
 * required), every role of the CTA pair leaves its loop, drains the copies and tensor-core work in
 * flight, frees its tensor memory and returns, so the context stays usable.  The other tiles are
 * computed as by nc_op_gemm; the skipped tile's part of `out` is left unwritten.  Returns the launch
 * status. */
NC_API nc_status nc_op_test_wait_timeout(const void *A, const void *B, int M, int N, int K, void *out,
                                         int ldo, unsigned long long limit_ns, int skip_tile,
                                         int *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NC_OPS_H */
