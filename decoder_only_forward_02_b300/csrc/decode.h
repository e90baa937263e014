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

// Attention of one query position per batch row against a layer's cache: the query of row b is
// q row b * Tq + tq ([B * Tq, H*D]), at position pos; it sees the cached keys of positions
// max(0, pos - window) .. pos (all of 0 .. pos when window < 0).  y row b * Tq + tq receives
// softmax(q k^T / sqrt(D)) v for every head (GQA: head h reads kv head h / (H/Hkv)); the other
// rows of y are left as they are.  scratch: fp32, at least B * H * decode_attention_splits(T)
// * (D + 2) floats for any pos < T.
int decode_attention_splits(int T_max);
cudaError_t launch_decode_attention(const bf16* q, int B, int Tq, int tq, int H, int Hkv, int D, const bf16* kcache,
                                    const bf16* vcache, int cap, int pos, int window, bf16* y, float* scratch,
                                    size_t scratch_floats, cudaStream_t stream);

}  // namespace nc
