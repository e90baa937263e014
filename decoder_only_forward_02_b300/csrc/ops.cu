// ops.cu -- per-kernel entry points declared in include/nc_ops.h.
#include "internal.h"
#include "nc_ops.h"

namespace {

int device_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

inline bool al(const void* p, size_t a) { return p != nullptr && reinterpret_cast<uintptr_t>(p) % a == 0; }
inline nc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NC_OK : NC_ERR_CUDA; }

}  // namespace

extern "C" {

nc_status nc_op_gemm(const void* A, const void* B, int M, int N, int K, nc_epilogue epi, void* out, int ldo,
                     const float* resid, float cap, int* status, void* stream) {
  if (!al(A, 16) || !al(B, 16) || !al(out, 16) || M < 1 || N < 1 || K < 1 || ldo < N || ldo % 8 != 0)
    return NC_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 32 != 0) return NC_ERR_UNSUPPORTED;
  if (epi == NC_EPI_RESID_F32 && !al(resid, 16)) return NC_ERR_INVALID_ARG;
  if (epi == NC_EPI_SOFTCAP_F32 && !(cap > 0.f)) return NC_ERR_INVALID_ARG;
  nc::GemmEpi e;
  switch (epi) {
    case NC_EPI_BF16: e.kind = nc::EPI_BF16; break;
    case NC_EPI_RESID_F32: e.kind = nc::EPI_RESID_F32; break;
    case NC_EPI_RELU2_BF16: e.kind = nc::EPI_RELU2_BF16; break;
    case NC_EPI_SOFTCAP_F32: e.kind = nc::EPI_SOFTCAP_F32; break;
    default: return NC_ERR_INVALID_ARG;
  }
  e.out = out;
  e.ldo = ldo;
  e.resid = resid;
  e.ldr = ldo;
  e.cap = cap;
  e.status = status;
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(A), static_cast<const nc::bf16*>(B), M, N, K,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_qkv(const void* xn, const void* wqkv, int M, int T, int C, int H, int Hkv, int D,
                    const float* rope, float eps, const float* gate, const void* ve, const int32_t* tokens, int V,
                    void* q, void* k, void* v, int* status, void* stream) {
  if (!al(xn, 16) || !al(wqkv, 16) || !al(rope, 16) || !al(q, 16) || !al(k, 16) || !al(v, 16) || M < 1 ||
      T < 1 || C < 1 || H < 1 || Hkv < 1 || H % Hkv != 0)
    return NC_ERR_INVALID_ARG;
  if (gate != nullptr && (!al(ve, 16) || tokens == nullptr || V < 1)) return NC_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || C % 64 != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  e.kind = nc::EPI_QKV;
  e.q = static_cast<nc::bf16*>(q);
  e.k = static_cast<nc::bf16*>(k);
  e.v = static_cast<nc::bf16*>(v);
  e.H = H;
  e.Hkv = Hkv;
  e.D = D;
  e.T = T;
  e.rope = reinterpret_cast<const float2*>(rope);
  e.eps = eps;
  e.gate = gate;
  e.ve = static_cast<const nc::bf16*>(ve);
  e.tokens = tokens;
  e.V = V;
  e.status = status;
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(xn), static_cast<const nc::bf16*>(wqkv), M,
                                     (H + 2 * Hkv) * D, C, e, device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_rope_table(float* rope, int T, int D, float base, void* stream) {
  if (!al(rope, 16) || T < 1 || D < 2 || D % 2 != 0 || !(base > 0.f)) return NC_ERR_INVALID_ARG;
  return cuda_status(nc::launch_rope_table(reinterpret_cast<float2*>(rope), T, D, base,
                                           static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_attention(const void* q, const void* k, const void* v, int B, int T, int H, int Hkv, int D,
                          int window, void* y, int* status, void* stream) {
  if (!al(q, 16) || !al(k, 16) || !al(v, 16) || !al(y, 16) || B < 1 || T < 1 || H < 1 || Hkv < 1 ||
      H % Hkv != 0)
    return NC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return NC_ERR_UNSUPPORTED;
  return cuda_status(nc::launch_attention(static_cast<const nc::bf16*>(q), static_cast<const nc::bf16*>(k),
                                          static_cast<const nc::bf16*>(v), B, T, H, Hkv, D, window,
                                          static_cast<nc::bf16*>(y), status, static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_rownorm(const float* x, const float* y, float a, float b, float* x_out, void* xn, int M, int C,
                        float eps, const void* wg, int Hkv, int c_g, float gate_scale, float* gate, void* stream) {
  if (!al(x, 16) || !al(xn, 16) || M < 1 || C < 1) return NC_ERR_INVALID_ARG;
  if ((y != nullptr && !al(y, 16)) || (x_out != nullptr && !al(x_out, 16))) return NC_ERR_INVALID_ARG;
  if (gate != nullptr && (!al(wg, 8) || Hkv < 1 || c_g < 4 || c_g > C)) return NC_ERR_INVALID_ARG;
  if (C % 128 != 0 || C > 2048 || (gate != nullptr && c_g % 4 != 0)) return NC_ERR_UNSUPPORTED;
  return cuda_status(nc::launch_rownorm(x, y, a, b, x_out, static_cast<nc::bf16*>(xn), M, C, eps,
                                        static_cast<const nc::bf16*>(wg), Hkv, c_g, gate_scale, gate,
                                        static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_embed_smear(const int32_t* tokens, int B, int T, const void* wte, int V, int C,
                            const void* smear_gate, int c_s, int embed_norm, float eps, float* x0, int* status,
                            void* stream) {
  if (tokens == nullptr || !al(wte, 16) || !al(x0, 16) || B < 1 || T < 1 || V < 1 || C < 1)
    return NC_ERR_INVALID_ARG;
  if (smear_gate != nullptr && (!al(smear_gate, 8) || c_s < 4 || c_s > C)) return NC_ERR_INVALID_ARG;
  if (C % 128 != 0 || C > 2048 || (smear_gate != nullptr && c_s % 4 != 0)) return NC_ERR_UNSUPPORTED;
  return cuda_status(nc::launch_embed_smear(tokens, B, T, static_cast<const nc::bf16*>(wte), V, C,
                                            static_cast<const nc::bf16*>(smear_gate), c_s, embed_norm, eps, x0,
                                            status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
