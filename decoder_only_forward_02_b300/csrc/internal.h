// internal.h -- launchers shared between the kernels and the model orchestration.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include "nc.h"

namespace nc {

using bf16 = __nv_bfloat16;

enum EpiKind : int {
  EPI_BF16 = 0,         // out(bf16) = acc
  EPI_RESID_F32 = 1,    // out(f32) = resid + acc   (resid may alias out)
  EPI_RELU2_BF16 = 2,   // out(bf16) = relu(acc)^2
  EPI_SOFTCAP_F32 = 3,  // out(f32) = cap * tanh(acc / cap)
  EPI_QKV = 4,          // q|k|v split, RoPE + RMSNorm on q and k, value-embedding gate on v
};

struct GemmEpi {
  int kind = EPI_BF16;
  void* out = nullptr;
  int ldo = 0;
  const float* resid = nullptr;
  int ldr = 0;
  float cap = 15.f;
  // EPI_QKV
  bf16* q = nullptr;
  bf16* k = nullptr;
  bf16* v = nullptr;
  int H = 0, Hkv = 0, D = 0, T = 1;
  const float2* rope = nullptr;   // [T_ctx][D/2] (cos, sin)
  float eps = 1e-6f;
  const float* gate = nullptr;    // [M, Hkv] or null (no value embedding on this layer)
  const bf16* ve = nullptr;       // [V, Hkv*D]
  const int32_t* tokens = nullptr;
  int V = 0;
  int* status = nullptr;
};

// Encodes a 2-D TMA descriptor with 128-byte swizzling through the driver entry point
// (no link-time libcuda).  inner/outer are extents in elements, row stride in bytes.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

inline bool make_tmap_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, inner, outer, row_stride_bytes,
                      box_inner, box_outer);
}

// C[M, N] = epi(A[M, K] . B[N, K]^T); A, B bf16 row-major (K contiguous).
// Requires K % 64 == 0, N % 32 == 0, 16-byte aligned rows.
cudaError_t launch_gemm(const bf16* A, const bf16* B, int M, int N, int K, const GemmEpi& epi,
                        int num_sms, cudaStream_t stream);

cudaError_t launch_embed_smear(const int32_t* tokens, int B, int T, const bf16* wte, int V, int C,
                               const bf16* smear_gate, int c_s, int embed_norm, float eps,
                               float* x0, int* status, cudaStream_t stream);

// x_new = a*x + b*y (y may be null when b == 0); optionally stored to x_out;
// xn = bf16(x_new / rms(x_new)); optionally gate[m, g] = scale*sigmoid(xn32[:c_g] . wg[g]).
cudaError_t launch_rownorm(const float* x, const float* y, float a, float b, float* x_out, bf16* xn,
                           int M, int C, float eps, const bf16* wg, int Hkv, int c_g,
                           float gate_scale, float* gate, cudaStream_t stream);

cudaError_t launch_rope_table(float2* table, int T, int D, float base, cudaStream_t stream);

// y[M, H*D] = windowed causal GQA attention of q [M, H*D], k/v [M, Hkv*D].
cudaError_t launch_attention(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H,
                             int Hkv, int D, int window, bf16* y, int* status, cudaStream_t stream);

}  // namespace nc
