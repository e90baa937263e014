// decode.h -- KV-cache kernels of the prefill + single-token decode path.
#pragma once
#include "internal.h"

namespace nc {

// Copies the keys and values of positions pos_base + t, t in [t_first, t_first + t_count), of
// every batch row b from k / v ([B * Tsrc, Hkv*D], row b * Tsrc + t) into a layer's cache
// ([B][cap][Hkv*D], position j in slot j % cap).  Copies that would land in the same slot must
// not be requested together (t_count <= cap).
cudaError_t launch_kv_append(const bf16* k, const bf16* v, int B, int Tsrc, int t_first, int t_count,
                             int pos_base, int kvcols, bf16* kcache, bf16* vcache, int cap, cudaStream_t stream);

// The decode step's attention of one layer (one new token per batch row at position pos), from
// the layer's q|k|v products: raw row b (fp32, pitch ldraw) holds rs * (x . W^T) over the packed
// q|k|v columns.  Per batch row and head: q rotated at pos, RMS-normed per head, rounded to bf16;
// the new key and value of each kv head (the key rotated and normed, the value plus the gated
// value embedding of tokens[b] on value-embedding layers), rounded to bf16, written into the
// layer's cache slot pos % cap and used directly; softmax(q k^T / sqrt(D)) v over the cached
// keys of positions max(0, pos - window) .. pos (all of 0 .. pos when window < 0), GQA head h
// reading kv head h / (H / Hkv), rounded to bf16 into y + b * ldy + h * D.  One launch: the keys
// split over a cluster of CTAs per (row, head), the splits combined through shared memory.
//   kc, vc: the layer's cache, [B][cap][Hkv * D] bf16.
struct DecodeAttn {
  const float* raw = nullptr;
  int ldraw = 0;
  int B = 0, H = 0, Hkv = 0, D = 0;
  int vgate = 0;
  float gate_scale = 1.f;
  const bf16* ve = nullptr;
  const int32_t* tokens = nullptr;
  int V = 0;
  const float2* rope = nullptr;   // [D/2][rope_ld] (cos, sin), position fastest
  int rope_ld = 0;
  int pos = 0;
  float eps = 1e-6f;
  bf16* kc = nullptr;
  bf16* vc = nullptr;
  int cap = 0;
  int window = -1;
  bf16* y = nullptr;
  int ldy = 0;
};

cudaError_t launch_decode_attention(const DecodeAttn& a, cudaStream_t stream);

// The products of a decode step (csrc/gemv.cu): B rows of A (bf16, row pitch lda elements, K
// columns, K % 32 == 0) times the weight W [N][K] (bf16, N % 8 == 0), each weight element read
// once, with the epilogue `kind` (GEMV_*).  Deterministic: the same inputs give the same bits.
enum GemvKind { GEMV_RAW = 0, GEMV_RESID = 1, GEMV_RELU2 = 2, GEMV_SOFTCAP_F32 = 3, GEMV_SOFTCAP_BF16 = 4 };

struct GemvEpi {
  int kind = GEMV_RAW;
  // Row scale rs[b] = 1 / sqrt(sum_{i < ssp_n} ssp[b * ssp_ld + i] * inv_ncols + eps): the input's
  // RMSNorm from its partial sums of squares; ssp == null -> 1.  Used by RAW, RELU2, SOFTCAP.
  const float* ssp = nullptr;
  int ssp_ld = 0, ssp_n = 0;
  float inv_ncols = 0.f, eps = 1e-6f;
  // RAW: fp32 rs * acc; RELU2: bf16 relu(rs * acc)^2; SOFTCAP: cap * tanh(rs * acc / cap), fp32
  // or bf16.  Row b at out + b * ldo elements.
  void* out = nullptr;
  int ldo = 0;
  float cap = 15.f;
  // RESID: xr = resid + acc; xm_out <- xr (if set); x' = a * xr + b * Y (Y may be null);
  // x_out <- x' (if set; may alias resid); xb <- bf16(x'); rows at b * ldx (fp32) and b * ldb (xb);
  // ssp_out[b * ssp_out_ld + n / 8] = sum of x'^2 over columns [n, n + 8) -- N / 8 partials per row.
  const float* resid = nullptr;
  float a = 1.f, b = 0.f;
  const float* Y = nullptr;
  float* x_out = nullptr;
  float* xm_out = nullptr;
  int ldx = 0;
  bf16* xb = nullptr;
  int ldb = 0;
  float* ssp_out = nullptr;
  int ssp_out_ld = 0;
};

cudaError_t launch_gemv(const bf16* A, int lda, int B, const bf16* W, int N, int K, const GemvEpi& ep,
                        cudaStream_t stream);

}  // namespace nc
