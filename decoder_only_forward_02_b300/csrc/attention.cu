// attention.cu -- causal grouped-query attention with a per-layer left window.
//
//   y[b, i, h, :] = sum_j softmax_j(q[b,i,h] . k[b,j,g] / sqrt(D)) v[b,j,g],   g = h / (H/Hkv),
//   over keys max(0, i - W) <= j <= i (all j <= i when W < 0).
//
// "Nanochat在nanoGPT之上的新增功能", section 1 table: grouped-query attention (fewer kv heads
// than query heads) and per-layer sliding-window attention; the notes give the repeating
// three-short-one-long pattern with the last layer full.  "nanochat — 架构与原理", section 5:
// the reference's Blackwell path falls back to an attention without windows.
//
// This version: one CTA per (32 queries, head, batch row); K/V tiles of 32 keys staged in
// shared memory as fp32; scores with one key per lane, online softmax in base 2 with the
// 1/sqrt(D)*log2(e) scale folded into q; key tiles entirely outside the window or in the
// causal future are never visited.
#include "internal.h"
#include "ptx.cuh"

namespace nc {
namespace {

constexpr int QB = 32, KB = 32, NT = 128;

template <int D>
__global__ void __launch_bounds__(NT)
    attn_simt_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k,
                     const bf16* __restrict__ v, int T, int H, int Hkv, int window,
                     bf16* __restrict__ y) {
  constexpr int DP = D + 1, DL = D / 32;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ks = Qs + QB * D;
  float* Vs = Ks + KB * DP;
  const int q0 = blockIdx.x * QB, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (H / Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t qs = static_cast<size_t>(H) * D, ks = static_cast<size_t>(Hkv) * D;
  const float sl2 = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;

  for (int idx = threadIdx.x; idx < QB * D; idx += NT) {
    const int r = idx / D, d = idx % D, t = q0 + r;
    Qs[idx] = t < T ? __bfloat162float(q[(static_cast<size_t>(b) * T + t) * qs + h * D + d]) * sl2 : 0.f;
  }
  const int qlast = min(q0 + QB - 1, T - 1);
  const int klo = window < 0 ? 0 : max(0, q0 - window);
  const int kt0 = klo / KB, kt1 = qlast / KB;

  float m[8], l[8], acc[8][DL];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < DL; ++c) acc[r][c] = 0.f;
  }

  for (int kt = kt0; kt <= kt1; ++kt) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < KB * D; idx += NT) {
      const int r = idx / D, d = idx % D, j = kt * KB + r;
      const size_t off = (static_cast<size_t>(b) * T + j) * ks + g * D + d;
      Ks[r * DP + d] = j < T ? __bfloat162float(k[off]) : 0.f;
      Vs[r * D + d] = j < T ? __bfloat162float(v[off]) : 0.f;
    }
    __syncthreads();
    const int j = kt * KB + lane;
    float s[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      const float kv = Ks[lane * DP + d];
#pragma unroll
      for (int r = 0; r < 8; ++r) s[r] = fmaf(Qs[(warp * 8 + r) * D + d], kv, s[r]);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = q0 + warp * 8 + r;
      const bool vis = i < T && j <= i && (window < 0 || j >= i - window);
      const float sv = vis ? s[r] : -INFINITY;
      const float mn = fmaxf(m[r], warp_max(sv));
      float p = 0.f, alpha = 1.f;
      if (mn != -INFINITY) {
        p = exp2f(sv - mn);
        alpha = exp2f(m[r] - mn);
      }
      l[r] = l[r] * alpha + warp_sum(p);
      m[r] = mn;
#pragma unroll
      for (int c = 0; c < DL; ++c) acc[r][c] *= alpha;
      s[r] = p;
    }
#pragma unroll 4
    for (int jj = 0; jj < KB; ++jj) {
      float vv[DL];
#pragma unroll
      for (int c = 0; c < DL; ++c) vv[c] = Vs[jj * D + c * 32 + lane];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float pj = __shfl_sync(0xffffffffu, s[r], jj);
#pragma unroll
        for (int c = 0; c < DL; ++c) acc[r][c] = fmaf(pj, vv[c], acc[r][c]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = q0 + warp * 8 + r;
    if (i >= T) continue;
    const float inv = 1.f / l[r];
    bf16* dst = y + (static_cast<size_t>(b) * T + i) * qs + h * D;
#pragma unroll
    for (int c = 0; c < DL; ++c) dst[c * 32 + lane] = __float2bfloat16_rn(acc[r][c] * inv);
  }
}

template <int D>
cudaError_t launch_d(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H, int Hkv,
                     int window, bf16* y, cudaStream_t stream) {
  constexpr int smem = (QB * D + KB * (D + 1) + KB * D) * 4;
  static cudaError_t attr = cudaFuncSetAttribute(attn_simt_kernel<D>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  dim3 grid((T + QB - 1) / QB, H, B);
  attn_simt_kernel<D><<<grid, NT, smem, stream>>>(q, k, v, T, H, Hkv, window, y);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H,
                             int Hkv, int D, int window, bf16* y, int* status, cudaStream_t stream) {
  (void)status;
  if (D == 128) return launch_d<128>(q, k, v, B, T, H, Hkv, window, y, stream);
  if (D == 64) return launch_d<64>(q, k, v, B, T, H, Hkv, window, y, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nc
