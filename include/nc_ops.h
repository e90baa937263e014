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
  NC_EPI_RESID_F32 = 1,   /* out fp32 [M, ldo] = resid + acc; resid may equal out */
  NC_EPI_RELU2_BF16 = 2,  /* out bf16 = relu(acc)^2     (squared-ReLU row of the feature table) */
  NC_EPI_SOFTCAP_F32 = 3  /* out fp32 = cap*tanh(acc/cap) (logit soft-cap row of the feature table) */
} nc_epilogue;

/* acc[M, N] = A[M, K] . B[N, K]^T (tcgen05, fp32 accumulation), then the epilogue.
 * K % 64 == 0, N % 32 == 0, ldo >= N, rows 16-byte aligned. */
NC_API nc_status nc_op_gemm(const void *A, const void *B, int M, int N, int K, nc_epilogue epi,
                            void *out, int ldo, const float *resid, float cap, int *status,
                            void *stream);

/* Packed q|k|v projection of a block: acc = xn[M, C] . wqkv[(H+2Hkv)*D, C]^T, split into
 * q [M, H*D], k [M, Hkv*D], v [M, Hkv*D] (bf16).  q and k: RoPE at position (row % T) from
 * `rope` (fp32 pairs (cos, sin), [>= T][D/2], see nc_op_rope_table), then RMSNorm over each
 * head (eps).  v: if gate != NULL, v += gate[m, g] * ve[tokens[m], g*D:(g+1)*D] (gate fp32
 * [M, Hkv], ve [V, Hkv*D]); out-of-range tokens add nothing. */
NC_API nc_status nc_op_qkv(const void *xn, const void *wqkv, int M, int T, int C, int H, int Hkv,
                           int D, const float *rope, float eps, const float *gate, const void *ve,
                           const int32_t *tokens, int V, void *q, void *k, void *v, int *status,
                           void *stream);

/* rope[t][i] = (cos, sin)(t * base^(-2i/D)), t < T, i < D/2, fp32 (angles in fp64). */
NC_API nc_status nc_op_rope_table(float *rope, int T, int D, float base, void *stream);

/* Windowed causal GQA attention: q [B*T, H*D], k, v [B*T, Hkv*D] -> y [B*T, H*D] (bf16);
 * window < 0 = plain causal; D in {64, 128}. */
NC_API nc_status nc_op_attention(const void *q, const void *k, const void *v, int B, int T, int H,
                                 int Hkv, int D, int window, void *y, int *status, void *stream);

/* Row kernel: x' = a*x + b*y (y may be NULL: x' = a*x), stored to x_out if non-NULL (may equal
 * x); xn = bf16(x' / sqrt(mean(x'^2) + eps)); if gate != NULL also
 * gate[m, g] = gate_scale * sigmoid(xn32[m, :c_g] . wg[g, :c_g]) (xn32 = unrounded).
 * x, y, x_out fp32 [M, C]; C % 128 == 0; c_g % 4 == 0. */
NC_API nc_status nc_op_rownorm(const float *x, const float *y, float a, float b, float *x_out,
                               void *xn, int M, int C, float eps, const void *wg, int Hkv, int c_g,
                               float gate_scale, float *gate, void *stream);

/* x0[b*T+t] = e_t + sigmoid(e_t[:c_s] . smear_gate) * e_{t-1} (t >= 1, same row b), e = wte[token]
 * (RMS-normalised first if embed_norm); smear_gate NULL = no smear.  Out-of-range tokens give a
 * zero embedding and NC_ERR_TOKEN_RANGE in *status.  x0 fp32 [B*T, C]. */
NC_API nc_status nc_op_embed_smear(const int32_t *tokens, int B, int T, const void *wte, int V,
                                   int C, const void *smear_gate, int c_s, int embed_norm,
                                   float eps, float *x0, int *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NC_OPS_H */
