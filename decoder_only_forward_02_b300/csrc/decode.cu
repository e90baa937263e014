// decode.cu -- KV cache of the prefill + single-token decode path.
//
// "nanochat — 架构与原理", section 2 component table (the inference engine: KV cache, sampling)
// and section 7 code map (engine: KVCache); "Nanochat在nanoGPT之上的新增功能", section 1 table
// and notes (per-layer sliding windows, GQA).  The cache of a layer keeps, per batch row, the
// post-RoPE, post-QK-norm keys and the values (value embedding included) of the positions its
// window can still see: all positions on full layers, the last W+1 on a layer with window W
// (position j lives in slot j % cap, a ring).
//
//   kv_append      copies keys and values of new positions into their slots (16 B per thread);
//                  the prefill's append.
//   decode_attn    a decode step's attention, one launch per layer: the q|k|v epilogue of the new
//                  token (RoPE, QK-norm, gated value embedding) and its cache append, then one
//                  query position per batch row split over the keys: one CTA per (row, head, 64
//                  visible keys), 4 warps of 8 key slots (4 lanes per key, each a quarter of the
//                  head dimension), online softmax in base 2 per slot (hardware exp2), slots
//                  combined through shared memory; the last CTA of a (row, head) combines its
//                  splits in a fixed order.  A key's value row is loaded with its key row (not
//                  after its score) and two keys per slot are in flight, so the loads' latencies
//                  overlap.  fp32 arithmetic; GQA reads kv head h / (H/Hkv).
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

// The decode step's attention for one (batch row b, head h, split) CTA: the split takes the visible
// keys [jlo + split * KPS, ...) (at most KPS).
//   Prologue, from the q|k|v products raw = rs * (x . W^T) of row b: the head's q rotated at pos
//   and RMS-normed (threads 0 .. D/2-1, each the columns j and j + D/2), rounded to bf16 as the
//   cache keeps k; on the split that holds position pos also the new key (rotated, normed) and
//   value (+ gate * ve[token] on value-embedding layers) of kv head g = h / (H / Hkv), kept in
//   shared memory for this CTA's own use; the CTA of the group's first q head writes them into
//   the cache slot pos % cap.  No CTA reads that slot from memory in this launch.
//   Keys: each warp scores 8 keys per step, 4 lanes per key (each lane a quarter of the head
//   dimension), with an online softmax in base 2 per key slot (hardware exp2); a key's value row
//   is loaded with its key row and two keys per slot are in flight.  The CTA's 32 slots are
//   combined through shared memory into (sum_j 2^(s_j - M) v_j, M, sum_j 2^(s_j - M)), written to
//   part[(b*H + h) * nsplit + split][0 .. D+1].
//   The last CTA of (b, h) to finish (a counter, after a memory fence) combines the splits in
//   split order: y = sum_s 2^(M_s - M) O_s / sum_s 2^(M_s - M) L_s, rounded to bf16.
// fp32 arithmetic throughout.
template <int D>
__global__ void __launch_bounds__(32 * DA_WARPS)
    decode_attn_kernel(const __grid_constant__ DecodeAttn a, float scale_log2, int nsplit) {
  constexpr int EL = D / 4;        // head-dimension elements per lane
  constexpr int SLOTS = DA_WARPS * 8;
  constexpr int HALF = D / 2;
  __shared__ float s_m[SLOTS], s_l[SLOTS];
  __shared__ float s_o[SLOTS][D];
  __shared__ float s_q[D];
  __shared__ __align__(16) bf16 s_kn[D];
  __shared__ __align__(16) bf16 s_vn[D];
  __shared__ float s_red[2][2];
  __shared__ float s_mv[DA_MAX_SPLITS], s_lv[DA_MAX_SPLITS], s_f[DA_MAX_SPLITS];
  __shared__ int s_last;
  griddep_wait();   // the q|k|v products come from the preceding kernel
  griddep_launch();
  const int H = a.H, Hkv = a.Hkv;
  const int bh = blockIdx.x, split = blockIdx.y;
  const int b = bh / H, h = bh % H;
  const int g = h / (H / Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvcols = Hkv * D;
  const int pos = a.pos;
  const int jlo = a.window < 0 ? 0 : max(0, pos - a.window);
  const int j0 = jlo + split * DA_KPS, j1 = min(pos + 1, j0 + DA_KPS);
  const bool has_new = j1 == pos + 1;   // this split holds the new position
  const size_t slot = (static_cast<size_t>(b) * a.cap + pos % a.cap) * kvcols + static_cast<size_t>(g) * D;
  const float* r = a.raw + static_cast<size_t>(b) * a.ldraw;
  {
    // role 0: q head h; role 1 (on the new key's split): k and v of kv head g
    const int role = tid / HALF, j = tid % HALF;
    float c0 = 0.f, c1 = 0.f, ss = 0.f;
    if (role == 0 || (role == 1 && has_new)) {
      const int col = role == 0 ? h * D : (H + g) * D;
      c0 = r[col + j];
      c1 = r[col + j + HALF];
      ss = c0 * c0 + c1 * c1;
    }
    if (role < 2) {
      ss = warp_sum(ss);
      if (HALF > 32) {
        if (lane == 0) s_red[role][(tid % HALF) >> 5] = ss;
      }
    }
    __syncthreads();
    if (role == 0 || (role == 1 && has_new)) {
      if (HALF > 32) ss = s_red[role][0] + s_red[role][1];
      const float sc = rsqrtf(ss * (1.0f / D) + a.eps);
      const float2 cs = a.rope[static_cast<size_t>(j) * a.rope_ld + pos];
      const bf16 y1 = __float2bfloat16((c0 * cs.x + c1 * cs.y) * sc);
      const bf16 y2 = __float2bfloat16((c1 * cs.x - c0 * cs.y) * sc);
      if (role == 0) {
        s_q[j] = __bfloat162float(y1) * scale_log2;
        s_q[j + HALF] = __bfloat162float(y2) * scale_log2;
      } else {
        s_kn[j] = y1;
        s_kn[j + HALF] = y2;
        const int vcol = (H + Hkv) * D + g * (a.vgate ? D + VGATE_ROWS : D);
        float v0 = r[vcol + j], v1 = r[vcol + j + HALF];
        if (a.vgate) {
          const int tok = a.tokens[b];
          if (tok >= 0 && tok < a.V) {
            const float gg = a.gate_scale * (1.0f / (1.0f + __expf(-r[vcol + D])));
            const bf16* e = a.ve + static_cast<size_t>(tok) * kvcols + g * D;
            v0 = fmaf(gg, __bfloat162float(e[j]), v0);
            v1 = fmaf(gg, __bfloat162float(e[j + HALF]), v1);
          }
        }
        s_vn[j] = __float2bfloat16(v0);
        s_vn[j + HALF] = __float2bfloat16(v1);
        if (h % (H / Hkv) == 0) {   // one writer per kv head: the group's first q head
          a.kc[slot + j] = y1;
          a.kc[slot + j + HALF] = y2;
          a.vc[slot + j] = s_vn[j];
          a.vc[slot + j + HALF] = s_vn[j + HALF];
        }
      }
    }
    __syncthreads();
  }
  const int kk = lane >> 2, quarter = lane & 3;   // key slot within the warp, quarter of the head dim
  float qv[EL];
#pragma unroll
  for (int e = 0; e < EL; ++e) qv[e] = s_q[quarter * EL + e];
  float m = -INFINITY, l = 0.f, o[EL];
#pragma unroll
  for (int e = 0; e < EL; ++e) o[e] = 0.f;
  const size_t rowbase = static_cast<size_t>(b) * a.cap * kvcols + g * D + quarter * EL;
  const uint4* kn = reinterpret_cast<const uint4*>(s_kn + quarter * EL);
  const uint4* vn = reinterpret_cast<const uint4*>(s_vn + quarter * EL);
#pragma unroll 2
  for (int jb = j0 + warp * 8; jb < j1; jb += SLOTS) {   // uniform across the warp
    const int j = jb + kk;
    const bool valid = j < j1;
    const bool isnew = valid && j == pos;   // the new key: from shared memory
    const bool ld = valid && !isnew;
    const size_t off = rowbase + static_cast<size_t>(j % a.cap) * kvcols;
    const uint4* kp = reinterpret_cast<const uint4*>(a.kc + off);
    const uint4* vp = reinterpret_cast<const uint4*>(a.vc + off);
    uint4 kw[EL / 8], vw[EL / 8];   // the key's and the value's rows, loaded together
#pragma unroll
    for (int u = 0; u < EL / 8; ++u) {
      kw[u] = ld ? __ldg(kp + u) : (isnew ? kn[u] : make_uint4(0u, 0u, 0u, 0u));
      vw[u] = ld ? __ldg(vp + u) : (isnew ? vn[u] : make_uint4(0u, 0u, 0u, 0u));
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
  const int kslot = warp * 8 + kk;
  if (quarter == 0) {
    s_m[kslot] = m;
    s_l[kslot] = l;
  }
#pragma unroll
  for (int e = 0; e < EL; ++e) s_o[kslot][quarter * EL + e] = o[e];
  __syncthreads();
  float* part = a.scratch + static_cast<size_t>(bh) * nsplit * (D + 2);
  float* dst = part + static_cast<size_t>(split) * (D + 2);
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < SLOTS; ++w) M = fmaxf(M, s_m[w]);
  for (int d = tid; d < D; d += 32 * DA_WARPS) {
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < SLOTS; ++w)
      if (s_m[w] != -INFINITY) O = fmaf(s_o[w][d], exp2f(s_m[w] - M), O);
    dst[d] = O;
  }
  if (tid == 0) {
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < SLOTS; ++w)
      if (s_m[w] != -INFINITY) L = fmaf(s_l[w], exp2f(s_m[w] - M), L);
    dst[D] = M;
    dst[D + 1] = L;
  }
  // the last CTA of (b, h) combines the splits
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counters + bh, 1u) == static_cast<unsigned>(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int s2 = tid; s2 < nsplit; s2 += 32 * DA_WARPS) {
    s_mv[s2] = __ldcg(part + static_cast<size_t>(s2) * (D + 2) + D);
    s_lv[s2] = __ldcg(part + static_cast<size_t>(s2) * (D + 2) + D + 1);
  }
  __syncthreads();
  float Mx = -INFINITY;
  for (int s2 = 0; s2 < nsplit; ++s2) Mx = fmaxf(Mx, s_mv[s2]);
  for (int s2 = tid; s2 < nsplit; s2 += 32 * DA_WARPS) s_f[s2] = exp2f(s_mv[s2] - Mx);
  __syncthreads();
  float L = 0.f;
  for (int s2 = 0; s2 < nsplit; ++s2) L = fmaf(s_lv[s2], s_f[s2], L);
  for (int d = tid; d < D; d += 32 * DA_WARPS) {
    float O = 0.f;
#pragma unroll 8
    for (int s2 = 0; s2 < nsplit; ++s2) O = fmaf(__ldcg(part + static_cast<size_t>(s2) * (D + 2) + d), s_f[s2], O);
    a.y[static_cast<size_t>(b) * a.ldy + h * D + d] = __float2bfloat16(O / L);
  }
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

cudaError_t launch_decode_attention(const DecodeAttn& a, cudaStream_t stream) {
  if (a.raw == nullptr || a.kc == nullptr || a.vc == nullptr || a.y == nullptr || a.scratch == nullptr ||
      a.counters == nullptr || a.rope == nullptr || a.B < 1 || a.H < 1 || a.Hkv < 1 || a.H % a.Hkv != 0 ||
      a.pos < 0 || a.pos >= a.rope_ld || a.cap < 1 || a.ldy < a.H * a.D ||
      (a.window < 0 ? a.cap <= a.pos : a.cap <= a.window && a.cap <= a.pos) ||
      (a.vgate && (a.ve == nullptr || a.tokens == nullptr)) ||
      a.ldraw < (a.H + a.Hkv) * a.D + a.Hkv * (a.vgate ? a.D + VGATE_ROWS : a.D))
    return cudaErrorInvalidValue;
  if (a.D != 64 && a.D != 128) return cudaErrorInvalidValue;
  const int jlo = a.window < 0 ? 0 : std::max(0, a.pos - a.window);
  const int nsplit = (a.pos - jlo + 1 + DA_KPS - 1) / DA_KPS;
  if (nsplit > DA_MAX_SPLITS || static_cast<size_t>(a.B) * a.H * nsplit * (a.D + 2) > a.scratch_floats)
    return cudaErrorInvalidValue;
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(a.B * a.H, nsplit);
  cfg.blockDim = dim3(32 * DA_WARPS);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = a.D == 128 ? cudaLaunchKernelEx(&cfg, decode_attn_kernel<128>, a, scale_log2, nsplit)
                                   : cudaLaunchKernelEx(&cfg, decode_attn_kernel<64>, a, scale_log2, nsplit);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace nc
