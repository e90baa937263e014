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
inline bool al_or_null(const void* p, size_t a) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % a == 0; }
using nc::cuda_status;
static_assert(NC_QKV_GATE_ROWS == nc::VGATE_ROWS, "packed gate rows of the public header and the kernels");

}  // namespace

extern "C" {

nc_status nc_op_gemm(const void* A, const void* B, int M, int N, int K, nc_epilogue epi, void* out, int ldo,
                     const float* ssp, int C, float eps, float cap, int* status, void* stream) {
  if (!al(A, 16) || !al(B, 16) || !al(out, 16) || M < 1 || N < 1 || K < 1 || ldo < N || ldo % 8 != 0)
    return NC_ERR_INVALID_ARG;
  if (!al_or_null(ssp, 4) || (ssp != nullptr && (C < nc::SS_GROUP || C % nc::SS_GROUP != 0)))
    return NC_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 32 != 0) return NC_ERR_UNSUPPORTED;
  if ((epi == NC_EPI_SOFTCAP_F32 || epi == NC_EPI_SOFTCAP_BF16) && !(cap > 0.f)) return NC_ERR_INVALID_ARG;
  nc::GemmEpi e;
  switch (epi) {
    case NC_EPI_BF16: e.kind = nc::EPI_BF16; break;
    case NC_EPI_RELU2_BF16: e.kind = nc::EPI_RELU2_BF16; break;
    case NC_EPI_SOFTCAP_F32: e.kind = nc::EPI_SOFTCAP_F32; break;
    case NC_EPI_SOFTCAP_BF16: e.kind = nc::EPI_SOFTCAP_BF16; break;
    default: return NC_ERR_INVALID_ARG;
  }
  e.out = out;
  e.ldo = ldo;
  e.cap = cap;
  e.status = status;
  if (ssp != nullptr && epi != NC_EPI_BF16) {
    e.ssp_in = ssp;
    e.ncg = C / nc::SS_GROUP;
    e.inv_ncols = 1.0f / static_cast<float>(C);
    e.eps = eps;
  }
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(A), static_cast<const nc::bf16*>(B), M, N, K,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
}

size_t nc_op_gemm_split_ws_bytes(int M, int N, int K, int ldo) {
  if (M < 1 || N < 1 || K < 1 || ldo < N) return 0;
  return nc::gemm_split_ws_bytes(M, N, K, ldo, device_sms());
}

nc_status nc_op_gemm_t(const void* A, const void* B, int M, int N, int K, int a_mn, int b_mn, nc_epilogue epi,
                       void* out, int ldo, const float* ssp, int C, float eps, float cap, void* split_ws,
                       size_t split_ws_bytes, int* status, void* stream) {
  if (!al(A, 16) || !al(B, 16) || !al(out, 16) || M < 1 || N < 1 || K < 1 || ldo < N || ldo % 8 != 0)
    return NC_ERR_INVALID_ARG;
  if ((a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1)) return NC_ERR_INVALID_ARG;
  if (!al_or_null(ssp, 4) || (ssp != nullptr && (C < nc::SS_GROUP || C % nc::SS_GROUP != 0)))
    return NC_ERR_INVALID_ARG;
  if (N % 32 != 0 || ((!a_mn || !b_mn) && K % 8 != 0) || (a_mn && M % 8 != 0) || (b_mn && N % 8 != 0))
    return NC_ERR_UNSUPPORTED;
  if ((epi == NC_EPI_SOFTCAP_F32 || epi == NC_EPI_SOFTCAP_BF16) && !(cap > 0.f)) return NC_ERR_INVALID_ARG;
  nc::GemmEpi e;
  switch (epi) {
    case NC_EPI_BF16: e.kind = nc::EPI_BF16; break;
    case NC_EPI_RELU2_BF16: e.kind = nc::EPI_RELU2_BF16; break;
    case NC_EPI_SOFTCAP_F32: e.kind = nc::EPI_SOFTCAP_F32; break;
    case NC_EPI_SOFTCAP_BF16: e.kind = nc::EPI_SOFTCAP_BF16; break;
    case NC_EPI_F32: e.kind = nc::EPI_F32; break;
    default: return NC_ERR_INVALID_ARG;
  }
  e.a_mn = a_mn;
  e.b_mn = b_mn;
  if (split_ws != nullptr) {   // split over K when the shape calls for it (fp32 output only)
    if (epi != NC_EPI_F32 || !al(split_ws, 16)) return NC_ERR_INVALID_ARG;
    if (split_ws_bytes < nc::gemm_split_ws_bytes(M, N, K, ldo, device_sms())) return NC_ERR_WORKSPACE;
    e.split_ws = static_cast<float*>(split_ws);
  }
  e.out = out;
  e.ldo = ldo;
  e.cap = cap;
  e.status = status;
  if (ssp != nullptr && epi != NC_EPI_BF16) {
    e.ssp_in = ssp;
    e.ncg = C / nc::SS_GROUP;
    e.inv_ncols = 1.0f / static_cast<float>(C);
    e.eps = eps;
  }
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(A), static_cast<const nc::bf16*>(B), M, N, K,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_lmhead_ce_grad(const void* xf, const void* wlm, int M, int V, int C, const float* ssp, float eps,
                               float cap, const int32_t* targets, const float* lse, const float* inv_count, void* out,
                               int ldo, int* status, void* stream) {
  if (!al(xf, 16) || !al(wlm, 16) || !al(out, 16) || !al(lse, 4) || !al(inv_count, 4) || targets == nullptr ||
      M < 1 || V < 1 || C < 1 || ldo < V || ldo % 8 != 0 || !(cap > 0.f))
    return NC_ERR_INVALID_ARG;
  if (!al_or_null(ssp, 4) || (ssp != nullptr && C % nc::SS_GROUP != 0)) return NC_ERR_INVALID_ARG;
  if (C % 8 != 0 || V % 32 != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  e.kind = nc::EPI_CE_GRAD;
  e.status = status;
  e.cap = cap;
  e.targets = targets;
  e.ce_lse = lse;
  e.inv_count = inv_count;
  e.out = out;
  e.ldo = ldo;
  if (ssp != nullptr) {
    e.ssp_in = ssp;
    e.ncg = C / nc::SS_GROUP;
    e.inv_ncols = 1.0f / static_cast<float>(C);
    e.eps = eps;
  }
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(xf), static_cast<const nc::bf16*>(wlm), M, V, C,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_mlp_hidden_grad(const void* dy, const void* w, int M, int F, int C, const float* ssp, float eps,
                                const void* h, void* out, int* status, void* stream) {
  if (!al(dy, 16) || !al(w, 16) || !al(h, 16) || !al(out, 16) || M < 1 || F < 1 || C < 1) return NC_ERR_INVALID_ARG;
  if (!al_or_null(ssp, 4) || (ssp != nullptr && C % nc::SS_GROUP != 0)) return NC_ERR_INVALID_ARG;
  if (C % 8 != 0 || F % 32 != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  e.kind = nc::EPI_DRELU2;
  e.status = status;
  e.b_mn = 1;   // w [C][F]: the product's K = C rows, its N = F columns contiguous
  e.h_in = static_cast<const nc::bf16*>(h);
  e.out = out;
  e.ldo = F;
  if (ssp != nullptr) {
    e.ssp_in = ssp;
    e.ncg = C / nc::SS_GROUP;
    e.inv_ncols = 1.0f / static_cast<float>(C);
    e.eps = eps;
  }
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(dy), static_cast<const nc::bf16*>(w), M, F, C, e,
                                     device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_rms_backward(const float* G, const float* x, const float* ssp, const float* add, int M, int C,
                             float eps, float* dx_f32, void* dx_b16, void* stream) {
  if (!al(G, 16) || !al(x, 16) || !al(ssp, 4) || !al_or_null(add, 16) || !al_or_null(dx_f32, 16) ||
      !al_or_null(dx_b16, 8) || (dx_f32 == nullptr && dx_b16 == nullptr) || M < 1 || C < 1 || !(eps >= 0.f))
    return NC_ERR_INVALID_ARG;
  if (C % nc::SS_GROUP != 0 || C > 2048) return NC_ERR_UNSUPPORTED;
  return cuda_status(nc::launch_rms_backward(G, x, ssp, add, M, C, eps, dx_f32, static_cast<nc::bf16*>(dx_b16),
                                             static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_gemm_residual(const void* A, const void* B, int M, int N, int K, const float* resid, float a,
                              float b, const float* Y, float* x_out, float* xm_out, void* xb, float* ssp,
                              int* status, void* stream) {
  if (!al(A, 16) || !al(B, 16) || !al(resid, 4) || !al(xb, 2) || !al(ssp, 4) || M < 1 || N < 1 || K < 1)
    return NC_ERR_INVALID_ARG;
  if (!al_or_null(Y, 4) || !al_or_null(x_out, 4) || !al_or_null(xm_out, 4)) return NC_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % nc::SS_GROUP != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  e.kind = nc::EPI_RESID;
  e.status = status;
  e.resid = resid;
  e.a = a;
  e.b = b;
  e.Y = Y;
  e.x_out = x_out;
  e.xm_out = xm_out;
  e.xb = static_cast<nc::bf16*>(xb);
  e.ssp_out = ssp;
  e.ncg = N / nc::SS_GROUP;
  return cuda_status(nc::launch_gemm_resid(static_cast<const nc::bf16*>(A), static_cast<const nc::bf16*>(B), M, N,
                                           K, e, device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_qkv(const void* xb, const void* wqkv, int M, int T, int C, int H, int Hkv, int D, const float* rope,
                    int rope_ld, float eps, const float* ssp, int vgate, float gate_scale, const void* ve,
                    const int32_t* tokens, int V, void* q, void* k, void* v, int* status, void* stream) {
  if (!al(xb, 16) || !al(wqkv, 16) || !al(rope, 16) || !al(q, 16) || !al(k, 16) || !al(v, 16) || !al(ssp, 4) ||
      M < 1 || T < 1 || C < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || rope_ld < T)
    return NC_ERR_INVALID_ARG;
  if (vgate && (!al(ve, 16) || tokens == nullptr || V < 1)) return NC_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || C % nc::SS_GROUP != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  e.kind = nc::EPI_QKV;
  e.status = status;
  e.ssp_in = ssp;
  e.ncg = C / nc::SS_GROUP;
  e.inv_ncols = 1.0f / static_cast<float>(C);
  e.eps = eps;
  e.q = static_cast<nc::bf16*>(q);
  e.k = static_cast<nc::bf16*>(k);
  e.v = static_cast<nc::bf16*>(v);
  e.H = H;
  e.Hkv = Hkv;
  e.D = D;
  e.T = T;
  e.rope = reinterpret_cast<const float2*>(rope);
  e.rope_ld = rope_ld;
  e.vgate = vgate ? 1 : 0;
  e.gate_scale = gate_scale;
  e.ve = static_cast<const nc::bf16*>(ve);
  e.tokens = tokens;
  e.V = V;
  const int N = (H + 2 * Hkv) * D + (vgate ? Hkv * nc::VGATE_ROWS : 0);
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(xb), static_cast<const nc::bf16*>(wqkv), M, N, C,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
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

nc_status nc_op_embed_smear(const int32_t* tokens, int B, int T, const void* wte, int V, int C,
                            const void* smear_gate, int c_s, int embed_norm, float eps, float a, float* x0, float* x,
                            void* xb, float* ssp, int* status, void* stream) {
  if (tokens == nullptr || !al(wte, 16) || !al(x0, 16) || !al(x, 16) || !al(xb, 16) || !al(ssp, 4) || B < 1 ||
      T < 1 || V < 1 || C < 1)
    return NC_ERR_INVALID_ARG;
  if (smear_gate != nullptr && (!al(smear_gate, 8) || c_s < 4 || c_s > C)) return NC_ERR_INVALID_ARG;
  if (C % 128 != 0 || C > 2048 || (smear_gate != nullptr && c_s % 4 != 0)) return NC_ERR_UNSUPPORTED;
  return cuda_status(nc::launch_embed_smear(tokens, B, T, static_cast<const nc::bf16*>(wte), V, C,
                                            static_cast<const nc::bf16*>(smear_gate), c_s, embed_norm, eps, a, x0,
                                            x, static_cast<nc::bf16*>(xb), ssp, status,
                                            static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_lmhead_ce(const void* xf, const void* wlm, int M, int V, int C, const float* ssp, float eps,
                          float cap, const int32_t* targets, float* part, float* zt, int* status, void* stream) {
  if (!al(xf, 16) || !al(wlm, 16) || !al(part, 4) || !al(zt, 4) || targets == nullptr || M < 1 || V < 1 ||
      C < 1 || !(cap > 0.f))
    return NC_ERR_INVALID_ARG;
  if (!al_or_null(ssp, 4) || (ssp != nullptr && C % nc::SS_GROUP != 0)) return NC_ERR_INVALID_ARG;
  if (C % 64 != 0 || V % 32 != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  e.kind = nc::EPI_CE;
  e.status = status;
  e.cap = cap;
  e.targets = targets;
  e.ce_part = part;
  e.ce_zt = zt;
  if (ssp != nullptr) {
    e.ssp_in = ssp;
    e.ncg = C / nc::SS_GROUP;
    e.inv_ncols = 1.0f / static_cast<float>(C);
    e.eps = eps;
  }
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(xf), static_cast<const nc::bf16*>(wlm), M, V, C,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
}

size_t nc_op_ce_scratch_bytes(int M) {
  return M < 1 ? 0 : static_cast<size_t>(nc::ce_scratch_doubles(M)) * sizeof(double);
}

nc_status nc_op_ce_finalize(const float* part, const float* zt, const int32_t* targets, int M, int V,
                            const int32_t* token_bytes, float* loss, float* stats, void* scratch,
                            size_t scratch_bytes, float* lse, float* inv_count, int* status, void* stream) {
  if (!al(part, 4) || !al(zt, 4) || targets == nullptr || !al(stats, 4) || !al(scratch, 8) ||
      !al_or_null(loss, 4) || !al_or_null(token_bytes, 4) || !al_or_null(lse, 4) || !al_or_null(inv_count, 4) ||
      M < 1 || V < 1)
    return NC_ERR_INVALID_ARG;
  if (scratch_bytes < nc_op_ce_scratch_bytes(M)) return NC_ERR_WORKSPACE;
  return cuda_status(nc::launch_ce_finalize(part, zt, targets, M, (V + 127) / 128, V, token_bytes, loss, stats,
                                            static_cast<double*>(scratch), status,
                                            static_cast<cudaStream_t>(stream), lse, inv_count));
}

size_t nc_op_fp8_scratch_bytes(void) { return static_cast<size_t>(nc::FP8_AMAX_BLOCKS) * sizeof(float); }

nc_status nc_op_fp8_quantize(const void* src, int src_f32, int M, int C, const float* ssp, float eps, void* dst,
                             float* inv_scale, void* scratch, void* stream) {
  if (!al(src, 16) || !al(dst, 8) || !al(inv_scale, 4) || !al(scratch, 4) || M < 1 || C < 8 ||
      (src_f32 != 0 && src_f32 != 1) || !al_or_null(ssp, 4) || !(eps >= 0.f))
    return NC_ERR_INVALID_ARG;
  if (C % 8 != 0 || (ssp != nullptr && C % nc::SS_GROUP != 0)) return NC_ERR_UNSUPPORTED;
  float* part = static_cast<float*>(scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = nc::launch_fp8_amax(src, src_f32, M, C, C, ssp, eps, part, s);
  if (e == cudaSuccess)
    e = nc::launch_fp8_quantize(src, src_f32, M, C, C, ssp, eps, part, nc::FP8_AMAX_BLOCKS, static_cast<uint8_t*>(dst),
                                C, 0, 0, inv_scale,
                                s);
  return cuda_status(e);
}

nc_status nc_op_gemm_fp8(const void* A8, const void* B8, int M, int N, int K, nc_epilogue epi, void* out, int ldo,
                         const float* inv_sa, const float* inv_sb, float cap, int* status, void* stream) {
  if (!al(A8, 16) || !al(B8, 16) || !al(out, 16) || !al(inv_sa, 4) || !al(inv_sb, 4) || M < 1 || N < 1 || K < 1 ||
      ldo < N || ldo % 8 != 0)
    return NC_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 32 != 0) return NC_ERR_UNSUPPORTED;
  nc::GemmEpi e;
  switch (epi) {
    case NC_EPI_BF16: e.kind = nc::EPI_BF16; break;
    case NC_EPI_RELU2_BF16: e.kind = nc::EPI_RELU2_BF16; break;
    case NC_EPI_SOFTCAP_F32: e.kind = nc::EPI_SOFTCAP_F32; break;
    case NC_EPI_SOFTCAP_BF16: e.kind = nc::EPI_SOFTCAP_BF16; break;
    case NC_EPI_F32: e.kind = nc::EPI_F32; break;
    default: return NC_ERR_INVALID_ARG;
  }
  if ((epi == NC_EPI_SOFTCAP_F32 || epi == NC_EPI_SOFTCAP_BF16) && !(cap > 0.f)) return NC_ERR_INVALID_ARG;
  e.fp8 = 1;
  e.fp8_sa = inv_sa;
  e.fp8_sw = inv_sb;
  e.out = out;
  e.ldo = ldo;
  e.cap = cap;
  e.status = status;
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(A8), static_cast<const nc::bf16*>(B8), M, N, K, e,
                                     device_sms(), static_cast<cudaStream_t>(stream)));
}

nc_status nc_op_test_wait_timeout(const void* A, const void* B, int M, int N, int K, void* out, int ldo,
                                  unsigned long long limit_ns, int skip_tile, int* status, void* stream) {
  if (!al(A, 16) || !al(B, 16) || !al(out, 16) || status == nullptr || M < 1 || N < 1 || K < 1 || ldo < N ||
      ldo % 8 != 0 || skip_tile < 0)
    return NC_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 32 != 0) return NC_ERR_UNSUPPORTED;
  // a limit long enough for the tiles that do run, short enough to end the test quickly
  if (limit_ns < 100000ull || limit_ns > 100000000ull) return NC_ERR_INVALID_ARG;
  nc::GemmEpi e;
  e.kind = nc::EPI_BF16;
  e.out = out;
  e.ldo = ldo;
  e.status = status;
  e.wait_ns = limit_ns;
  e.test_skip_tile = skip_tile;
  return cuda_status(nc::launch_gemm(static_cast<const nc::bf16*>(A), static_cast<const nc::bf16*>(B), M, N, K,
                                     e, device_sms(), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
