// decode.cu -- KV cache of the prefill + single-token decode path.
//
// "nanochat — 架构与原理", section 2 component table (the inference engine: KV cache, sampling)
// and section 7 code map (engine: KVCache); "Nanochat在nanoGPT之上的新增功能", section 1 table
// and notes (per-layer sliding windows, GQA).  The cache of a layer keeps, per batch row, the
// post-RoPE, post-QK-norm keys and the values (value embedding included) of the positions its
// window can still see: all positions on full layers, the last W+1 on a layer with window W
// (position j lives in slot j % cap, a ring).
//
//   kv_append      copies keys and values of new positions into their slots (16 B per thread).
//   decode_attn    one query position per batch row, split over the keys: one CTA per (row, head,
//                  64 visible keys), 4 warps of 8 key slots (4 lanes per key, each a quarter of
//                  the head dimension), online softmax in base 2 per slot (hardware exp2), slots
//                  combined through shared memory; a second kernel combines the splits in a fixed
//                  order.  A key's value row is loaded with its key row (not after its score) and
//                  two keys per slot are in flight, so the loads' latencies overlap.  fp32
//                  arithmetic; GQA reads kv head h / (H/Hkv).
#include "decode.h"
#include "ptx.cuh"

#include <algorithm>
#include <cmath>

namespace nc {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int DA_WARPS = 4;
constexpr int DA_KPS = 64;    // keys per split (2 steps of 32 keys for a CTA)

__global__ void __launch_bounds__(APPEND_THREADS)
    kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, int B, int Tsrc, int t_first,
                     int t_count, int pos_base, int chunks, uint4* __restrict__ kc, uint4* __restrict__ vc, int cap) {
  griddep_wait();   // the q/k/v projection that wrote k and v has completed
  griddep_launch();
  const long long i = static_cast<long long>(blockIdx.x) * APPEND_THREADS + threadIdx.x;
  const long long total = static_cast<long long>(B) * t_count * chunks;
  if (i >= total) return;
  const int c = static_cast<int>(i % chunks);
  const int t = static_cast<int>((i / chunks) % t_count) + t_first;
  const int b = static_cast<int>(i / (static_cast<long long>(chunks) * t_count));
  const size_t src = (static_cast<size_t>(b) * Tsrc + t) * chunks + c;
  const size_t dst = (static_cast<size_t>(b) * cap + (pos_base + t) % cap) * chunks + c;
  kc[dst] = k[src];
  vc[dst] = v[src];
}

// Split-key decode attention, pass 1: CTA (row b, head h, split) takes the visible keys
// [jlo + split * KPS, ...) (at most KPS); each warp scores 8 keys per step, 4 lanes per key (each
// lane a quarter of the head dimension), with an online softmax in base 2 per key slot; the 32
// slots of the CTA are combined through shared memory into (sum_j 2^(s_j - M) v_j, M, sum_j
// 2^(s_j - M)) for the split, written to part[(b*H + h) * nsplit + split][0 .. D+1].
template <int D>
__global__ void __launch_bounds__(32 * DA_WARPS)
    decode_attn_split_kernel(const bf16* __restrict__ q, int Tq, int tq, int H, int Hkv, const bf16* __restrict__ kc,
                             const bf16* __restrict__ vc, int cap, int pos, int window, float scale_log2, int nsplit,
                             float* __restrict__ part) {
  constexpr int EL = D / 4;        // head-dimension elements per lane
  constexpr int SLOTS = DA_WARPS * 8;
  __shared__ float s_m[SLOTS], s_l[SLOTS];
  __shared__ float s_o[SLOTS][D];
  griddep_wait();   // the cache append (and the q projection) have completed
  griddep_launch();
  const int bh = blockIdx.x, split = blockIdx.y;
  const int b = bh / H, h = bh % H;
  const int g = h / (H / Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kk = lane >> 2, quarter = lane & 3;   // key slot within the warp, quarter of the head dim
  const int kvcols = Hkv * D;
  float qv[EL];
  {
    const uint4* qp = reinterpret_cast<const uint4*>(q + (static_cast<size_t>(b) * Tq + tq) * (static_cast<size_t>(H) * D) +
                                                     h * D + quarter * EL);
#pragma unroll
    for (int u = 0; u < EL / 8; ++u) {
      const uint4 w = __ldg(qp + u);
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(w2[t]);
        qv[u * 8 + 2 * t] = f.x * scale_log2;
        qv[u * 8 + 2 * t + 1] = f.y * scale_log2;
      }
    }
  }
  const int jlo = window < 0 ? 0 : max(0, pos - window);
  const int j0 = jlo + split * DA_KPS, j1 = min(pos + 1, j0 + DA_KPS);
  float m = -INFINITY, l = 0.f, o[EL];
#pragma unroll
  for (int e = 0; e < EL; ++e) o[e] = 0.f;
  const size_t rowbase = static_cast<size_t>(b) * cap * kvcols + g * D + quarter * EL;
#pragma unroll 2
  for (int jb = j0 + warp * 8; jb < j1; jb += SLOTS) {   // uniform across the warp
    const int j = jb + kk;
    const bool valid = j < j1;
    const size_t off = rowbase + static_cast<size_t>((valid ? j : jb) % cap) * kvcols;
    const uint4* kp = reinterpret_cast<const uint4*>(kc + off);
    const uint4* vp = reinterpret_cast<const uint4*>(vc + off);
    uint4 kw[EL / 8], vw[EL / 8];   // the key's and the value's rows, loaded together
#pragma unroll
    for (int u = 0; u < EL / 8; ++u) {
      kw[u] = __ldg(kp + u);
      vw[u] = __ldg(vp + u);
    }
    float sc = 0.f;
#pragma unroll
    for (int u = 0; u < EL / 8; ++u) {
      const uint4 w = kw[u];
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(w2[t]);
        sc = fmaf(qv[u * 8 + 2 * t], f.x, sc);
        sc = fmaf(qv[u * 8 + 2 * t + 1], f.y, sc);
      }
    }
    sc += __shfl_xor_sync(0xffffffffu, sc, 1);
    sc += __shfl_xor_sync(0xffffffffu, sc, 2);   // the key's full score, in base-2 units
    if (valid) {
      const float mn = fmaxf(m, sc);
      const float corr = ex2_approx(m - mn);   // 0 on the slot's first key (m = -inf, sc finite)
      const float p = ex2_approx(sc - mn);
      l = fmaf(l, corr, p);
#pragma unroll
      for (int u = 0; u < EL / 8; ++u) {
        const uint4 w = vw[u];
        const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = __bfloat1622float2(w2[t]);
          o[u * 8 + 2 * t] = fmaf(p, f.x, o[u * 8 + 2 * t] * corr);
          o[u * 8 + 2 * t + 1] = fmaf(p, f.y, o[u * 8 + 2 * t + 1] * corr);
        }
      }
      m = mn;
    }
  }
  const int slot = warp * 8 + kk;
  if (quarter == 0) {
    s_m[slot] = m;
    s_l[slot] = l;
  }
#pragma unroll
  for (int e = 0; e < EL; ++e) s_o[slot][quarter * EL + e] = o[e];
  __syncthreads();
  float* dst = part + (static_cast<size_t>(bh) * nsplit + split) * (D + 2);
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < SLOTS; ++w) M = fmaxf(M, s_m[w]);
  for (int d = threadIdx.x; d < D; d += 32 * DA_WARPS) {
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < SLOTS; ++w)
      if (s_m[w] != -INFINITY) O = fmaf(s_o[w][d], exp2f(s_m[w] - M), O);
    dst[d] = O;
  }
  if (threadIdx.x == 0) {
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < SLOTS; ++w)
      if (s_m[w] != -INFINITY) L = fmaf(s_l[w], exp2f(s_m[w] - M), L);
    dst[D] = M;
    dst[D + 1] = L;
  }
}

// Pass 2: y[b, h] = sum_s 2^(M_s - M) O_s / sum_s 2^(M_s - M) L_s over the splits, in split order.
template <int D>
__global__ void __launch_bounds__(D)
    decode_attn_combine_kernel(const float* __restrict__ part, int nsplit, int Tq, int tq, int H,
                               bf16* __restrict__ y) {
  griddep_wait();
  griddep_launch();
  const int bh = blockIdx.x, b = bh / H, h = bh % H, d = threadIdx.x;
  const float* p = part + static_cast<size_t>(bh) * nsplit * (D + 2);
  float M = -INFINITY;
  for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, p[s2 * (D + 2) + D]);
  float L = 0.f, O = 0.f;
  for (int s2 = 0; s2 < nsplit; ++s2) {
    const float f = exp2f(p[s2 * (D + 2) + D] - M);
    L = fmaf(p[s2 * (D + 2) + D + 1], f, L);
    O = fmaf(p[s2 * (D + 2) + d], f, O);
  }
  y[(static_cast<size_t>(b) * Tq + tq) * (static_cast<size_t>(H) * D) + h * D + d] = __float2bfloat16(O / L);
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, int grid, int threads, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace

cudaError_t launch_kv_append(const bf16* k, const bf16* v, int B, int Tsrc, int t_first, int t_count,
                             int pos_base, int kvcols, bf16* kcache, bf16* vcache, int cap, cudaStream_t stream) {
  if (k == nullptr || v == nullptr || kcache == nullptr || vcache == nullptr || B < 1 || Tsrc < 1 || t_first < 0 ||
      t_count < 1 || t_first + t_count > Tsrc || pos_base < 0 || kvcols % 8 != 0 || cap < t_count)
    return cudaErrorInvalidValue;
  const int chunks = kvcols * 2 / 16;
  const long long total = static_cast<long long>(B) * t_count * chunks;
  const int grid = static_cast<int>((total + APPEND_THREADS - 1) / APPEND_THREADS);
  return launch_pdl(kv_append_kernel, grid, APPEND_THREADS, stream, reinterpret_cast<const uint4*>(k),
                    reinterpret_cast<const uint4*>(v), B, Tsrc, t_first, t_count, pos_base, chunks,
                    reinterpret_cast<uint4*>(kcache), reinterpret_cast<uint4*>(vcache), cap);
}

int decode_attention_splits(int T_max) { return (T_max + DA_KPS - 1) / DA_KPS; }

cudaError_t launch_decode_attention(const bf16* q, int B, int Tq, int tq, int H, int Hkv, int D, const bf16* kcache,
                                    const bf16* vcache, int cap, int pos, int window, bf16* y, float* scratch,
                                    size_t scratch_floats, cudaStream_t stream) {
  if (q == nullptr || kcache == nullptr || vcache == nullptr || y == nullptr || scratch == nullptr || B < 1 ||
      Tq < 1 || tq < 0 || tq >= Tq || H < 1 || Hkv < 1 || H % Hkv != 0 || pos < 0 || cap < 1 ||
      (window < 0 ? cap <= pos : cap <= window && cap <= pos))
    return cudaErrorInvalidValue;
  if (D != 64 && D != 128) return cudaErrorInvalidValue;
  const int jlo = window < 0 ? 0 : std::max(0, pos - window);
  const int nsplit = (pos - jlo + 1 + DA_KPS - 1) / DA_KPS;
  if (static_cast<size_t>(B) * H * nsplit * (D + 2) > scratch_floats) return cudaErrorInvalidValue;
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(B * H, nsplit);
  cfg.blockDim = dim3(32 * DA_WARPS);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = D == 128 ? cudaLaunchKernelEx(&cfg, decode_attn_split_kernel<128>, q, Tq, tq, H, Hkv, kcache, vcache,
                                                cap, pos, window, scale_log2, nsplit, scratch)
                           : cudaLaunchKernelEx(&cfg, decode_attn_split_kernel<64>, q, Tq, tq, H, Hkv, kcache, vcache,
                                                cap, pos, window, scale_log2, nsplit, scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  if (D == 128)
    return launch_pdl(decode_attn_combine_kernel<128>, B * H, 128, stream, static_cast<const float*>(scratch), nsplit,
                      Tq, tq, H, y);
  return launch_pdl(decode_attn_combine_kernel<64>, B * H, 64, stream, static_cast<const float*>(scratch), nsplit, Tq,
                    tq, H, y);
}

}  // namespace nc
