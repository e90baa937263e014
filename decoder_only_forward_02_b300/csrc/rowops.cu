// rowops.cu -- memory-bound per-row kernels: the token embedding with smear and the first
// block's residual mix, the rotary-angle table, and the backward of the weightless RMSNorm.
//
// One warp per row, 8 rows per 256-thread block; each lane owns C/128 groups of 4
// consecutive channels (offset 128*i + 4*lane), so every load and store is a coalesced
// 128-bit (fp32) or 64-bit (bf16 x4) access; reductions are warp shuffles.  Group i of a lane
// is column group i of the row (128 channels), the unit of the partial sums the GEMM
// epilogues consume.
//
// Definitions ("Nanochat在nanoGPT之上的新增功能", section 1 table and notes): smear adds
// sigmoid(gate(x)) times the previous token's embedding; blocks rescale the residual stream by
// resid_lambdas and add x0_lambdas * x0 (for the first block x = x0, so x = (l_r + l_0) x0);
// RMSNorm has no learned weight.
#include "internal.h"
#include "ptx.cuh"

namespace nc {
namespace {

constexpr int ROWS_PER_BLOCK = 8;

__device__ __forceinline__ float4 ld_bf16x4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void st_bf16x4(bf16* p, float4 v) {
  uint2 u;
  u.x = pack_bf16(v.x, v.y);
  u.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }

template <int NV4>
__device__ __forceinline__ void load_embedding(const bf16* wte, int tok, int V, int lane, bool norm,
                                               float eps, float4 (&e)[NV4]) {
  constexpr int C = NV4 * 128;
  const bool ok = tok >= 0 && tok < V;
#pragma unroll
  for (int i = 0; i < NV4; ++i)
    e[i] = ok ? ld_bf16x4(wte + static_cast<size_t>(tok) * C + i * 128 + lane * 4)
              : make_float4(0.f, 0.f, 0.f, 0.f);
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV4; ++i) ss += dot4(e[i], e[i]);
    const float r = rsqrtf(warp_sum(ss) * (1.0f / C) + eps);
#pragma unroll
    for (int i = 0; i < NV4; ++i) {
      e[i].x *= r; e[i].y *= r; e[i].z *= r; e[i].w *= r;
    }
  }
}

template <int NV4>
__global__ void __launch_bounds__(32 * ROWS_PER_BLOCK)
    embed_smear_kernel(const int32_t* __restrict__ tokens, int M, int T, const bf16* __restrict__ wte,
                       int V, const bf16* __restrict__ smear_gate, int c_s, int embed_norm, float eps,
                       float a, float* __restrict__ x0, float* __restrict__ x, bf16* __restrict__ xb,
                       float* __restrict__ ssp, int* status) {
  constexpr int C = NV4 * 128;
  griddep_wait();   // the previous kernel on the stream (still reading xb, ssp, ...) has completed
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * ROWS_PER_BLOCK + (threadIdx.x >> 5);
  if (row >= M) return;
  const int t = row % T;
  const int tok = tokens[row];
  if ((tok < 0 || tok >= V) && lane == 0) record_error(status, NC_ERR_TOKEN_RANGE);
  float4 e[NV4];
  load_embedding<NV4>(wte, tok, V, lane, embed_norm != 0, eps, e);
  if (smear_gate != nullptr && t > 0) {
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < NV4; ++i) {
      const int c = i * 128 + lane * 4;
      if (c < c_s) dot += dot4(e[i], ld_bf16x4(smear_gate + c));
    }
    const float gate = sigmoidf_(warp_sum(dot));
    float4 p[NV4];
    load_embedding<NV4>(wte, tokens[row - 1], V, lane, embed_norm != 0, eps, p);
#pragma unroll
    for (int i = 0; i < NV4; ++i) {
      e[i].x = fmaf(gate, p[i].x, e[i].x);
      e[i].y = fmaf(gate, p[i].y, e[i].y);
      e[i].z = fmaf(gate, p[i].z, e[i].z);
      e[i].w = fmaf(gate, p[i].w, e[i].w);
    }
  }
  const size_t base = static_cast<size_t>(row) * C;
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    *reinterpret_cast<float4*>(x0 + base + i * 128 + lane * 4) = e[i];
    const float4 v = make_float4(a * e[i].x, a * e[i].y, a * e[i].z, a * e[i].w);
    *reinterpret_cast<float4*>(x + base + i * 128 + lane * 4) = v;
    st_bf16x4(xb + base + i * 128 + lane * 4, v);
    const float s = warp_sum(dot4(v, v));
    if (lane == 0) ssp[static_cast<size_t>(row) * NV4 + i] = s;
  }
}

// Backward of xn = rs * x, rs = 1 / sqrt(mean(x^2) + eps), given G = rs * dL/dxn (the gradient
// GEMMs fold the forward's row scale into their operand):  dL/dx_j = rs g_j - rs^3 x_j mean(g x)
// = G_j - rs^2 x_j mean(G x).  rs^2 comes from the forward's partial sums of squares (the same
// value the forward's consumers used); `add` is a gradient reaching x by another path (the
// residual connection), added before the bf16 rounding.
template <int NV4>
__global__ void __launch_bounds__(32 * ROWS_PER_BLOCK)
    rms_backward_kernel(const float* __restrict__ G, const float* __restrict__ x, const float* __restrict__ ssp,
                        const float* __restrict__ add, int M, float eps, float* __restrict__ dx_f32,
                        bf16* __restrict__ dx_b16) {
  constexpr int C = NV4 * 128;
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * ROWS_PER_BLOCK + (threadIdx.x >> 5);
  if (row >= M) return;
  const size_t base = static_cast<size_t>(row) * C;
  float ss = lane < NV4 ? ssp[static_cast<size_t>(row) * NV4 + lane] : 0.f;
  float4 g[NV4], xv[NV4];
  float gx = 0.f;
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    g[i] = *reinterpret_cast<const float4*>(G + base + i * 128 + lane * 4);
    xv[i] = *reinterpret_cast<const float4*>(x + base + i * 128 + lane * 4);
    gx += dot4(g[i], xv[i]);
  }
  ss = warp_sum(ss);
  gx = warp_sum(gx);
  const float rs2 = 1.0f / (ss * (1.0f / C) + eps);
  const float k = rs2 * gx * (1.0f / C);
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    float4 d = make_float4(fmaf(-k, xv[i].x, g[i].x), fmaf(-k, xv[i].y, g[i].y), fmaf(-k, xv[i].z, g[i].z),
                           fmaf(-k, xv[i].w, g[i].w));
    if (add != nullptr) {
      const float4 a = *reinterpret_cast<const float4*>(add + base + i * 128 + lane * 4);
      d.x += a.x; d.y += a.y; d.z += a.z; d.w += a.w;
    }
    if (dx_f32 != nullptr) *reinterpret_cast<float4*>(dx_f32 + base + i * 128 + lane * 4) = d;
    if (dx_b16 != nullptr) st_bf16x4(dx_b16 + base + i * 128 + lane * 4, d);
  }
}

// table[i * T + t] = (cos, sin)(t * base^(-2i/D)): position fastest, so the threads of a warp
// (consecutive rows, i.e. consecutive positions) read one contiguous run per pair index i.
__global__ void rope_table_kernel(float2* table, int T, int half, double base) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= T * half) return;
  const int i = idx / T, t = idx % T;
  const double inv = pow(base, -2.0 * i / (2.0 * half));
  double s, c;
  sincos(static_cast<double>(t) * inv, &s, &c);
  table[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

template <template <int> class Fn, typename... Args>
cudaError_t dispatch_nv4(int C, Args&&... args) {
  switch (C / 128) {
#define NC_CASE(n) case n: return Fn<n>::run(args...);
    NC_CASE(1) NC_CASE(2) NC_CASE(3) NC_CASE(4) NC_CASE(5) NC_CASE(6) NC_CASE(7) NC_CASE(8)
    NC_CASE(9) NC_CASE(10) NC_CASE(11) NC_CASE(12) NC_CASE(13) NC_CASE(14) NC_CASE(15) NC_CASE(16)
#undef NC_CASE
    default: return cudaErrorInvalidValue;
  }
}

template <int NV4>
struct EmbedLaunch {
  static cudaError_t run(const int32_t* tokens, int M, int T, const bf16* wte, int V,
                         const bf16* smear_gate, int c_s, int embed_norm, float eps, float a, float* x0,
                         float* x, bf16* xb, float* ssp, int* status, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = dim3((M + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK);
    cfg.blockDim = dim3(32 * ROWS_PER_BLOCK);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, embed_smear_kernel<NV4>, tokens, M, T, wte, V, smear_gate, c_s,
                                             embed_norm, eps, a, x0, x, xb, ssp, status);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
  }
};

template <int NV4>
struct RmsBackwardLaunch {
  static cudaError_t run(const float* G, const float* x, const float* ssp, const float* add, int M, float eps,
                         float* dx_f32, bf16* dx_b16, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = dim3((M + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK);
    cfg.blockDim = dim3(32 * ROWS_PER_BLOCK);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, rms_backward_kernel<NV4>, G, x, ssp, add, M, eps, dx_f32, dx_b16);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
  }
};

}  // namespace

cudaError_t launch_rms_backward(const float* G, const float* x, const float* ssp, const float* add, int M, int C,
                                float eps, float* dx_f32, bf16* dx_b16, cudaStream_t stream) {
  if (G == nullptr || x == nullptr || ssp == nullptr || M < 1 || C % 128 != 0 || C > 16 * 128 ||
      (dx_f32 == nullptr && dx_b16 == nullptr))
    return cudaErrorInvalidValue;
  return dispatch_nv4<RmsBackwardLaunch>(C, G, x, ssp, add, M, eps, dx_f32, dx_b16, stream);
}

cudaError_t launch_embed_smear(const int32_t* tokens, int B, int T, const bf16* wte, int V, int C,
                               const bf16* smear_gate, int c_s, int embed_norm, float eps, float a,
                               float* x0, float* x, bf16* xb, float* ssp, int* status, cudaStream_t stream) {
  if (C % 128 != 0 || c_s % 4 != 0) return cudaErrorInvalidValue;
  return dispatch_nv4<EmbedLaunch>(C, tokens, B * T, T, wte, V, smear_gate, c_s, embed_norm, eps, a, x0,
                                   x, xb, ssp, status, stream);
}

cudaError_t launch_rope_table(float2* table, int T, int D, float base, cudaStream_t stream) {
  const int n = T * (D / 2);
  rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(table, T, D / 2, static_cast<double>(base));
  return cudaGetLastError();
}

}  // namespace nc
