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
//                  query position per batch row split over the keys: a cluster of 8 CTAs per
//                  (row, head), each an eighth of the cached keys, 8 warps reading whole key and
//                  value rows (D/8 lanes per row), online softmax in base 2 per key slot
//                  (hardware exp2), slots combined through shared memory; the cluster's rank 0
//                  combines the splits and the new key in a fixed order from its peers' shared
//                  memory.  A key's value row is loaded with its key row (not after its score)
//                  and two steps are in flight, so the loads' latencies overlap.  fp32
//                  arithmetic; GQA reads kv head h / (H/Hkv).
#include "decode.h"
#include "ptx.cuh"

#include <algorithm>
#include <cmath>

namespace nc {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int DA_WARPS = 8;
constexpr int DA_SPLITS = 8;  // CTAs per (row, head): one cluster, combined through shared memory

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

// The decode step's attention for one (batch row b, head h, split) CTA.  The keys before pos
// (all cached by earlier steps or the prefill) are split evenly over the DA_SPLITS CTAs of a
// cluster: split s takes [jlo + s * kps, ...) (at most kps); the new key at pos is a partial of
// its own.
//   Prologue, from the q|k|v products raw = rs * (x . W^T) of row b: the head's q rotated at pos
//   and RMS-normed (threads 0 .. D/2-1, each the columns j and j + D/2), rounded to bf16 as the
//   cache keeps k.  The cluster's rank 0 also computes the new key (rotated, normed) and value
//   (+ gate * ve[token] on value-embedding layers) of kv head g = h / (H / Hkv), rounded to bf16;
//   the rank 0 of the group's first q head writes them into the cache slot pos % cap, which no
//   CTA of this launch reads.
//   Keys: each warp takes 8 keys per step; a key's 256-byte row (D = 128; 128 at D = 64) is
//   read whole by D/8 lanes, 16 B each, so one load instruction of the warp covers 2 (4) rows;
//   those 2 (4) groups of lanes are the warp's key slots, each with an online softmax in base 2
//   (hardware exp2) over its keys.  A key's value row is loaded with its key row and two steps
//   are in flight.  The CTA's slots are combined through shared memory into
//   (sum_j 2^(s_j - M) v_j, M, sum_j 2^(s_j - M)).
//   After a cluster barrier, rank 0 reads the partials from its peers' shared memory and
//   combines them in split order, then the new key's (score s, 1, v_new):
//   y = sum 2^(M_s - M) O_s / sum 2^(M_s - M) L_s, rounded to bf16.
// fp32 arithmetic throughout.
template <int D>
__global__ void __launch_bounds__(32 * DA_WARPS)
    decode_attn_kernel(const __grid_constant__ DecodeAttn a, float scale_log2, int kps) {
  constexpr int LPK = D / 8;             // lanes per key row (16 B each)
  constexpr int KPI = 32 / LPK;           // key rows per load instruction of a warp: its key slots
  constexpr int KPL = 8 / KPI;            // keys per lane and step (8 keys per warp and step)
  constexpr int SLOTS = DA_WARPS * KPI;   // online-softmax slots of the CTA
  constexpr int HALF = D / 2;
  __shared__ float s_m[SLOTS], s_l[SLOTS], s_w[SLOTS];
  __shared__ float s_o[SLOTS][D];
  __shared__ float s_q[D];
  __shared__ __align__(16) bf16 s_kn[D];
  __shared__ __align__(16) bf16 s_vn[D];
  __shared__ float s_red[DA_WARPS];
  __shared__ float s_part[D + 2];   // the CTA's (O[D], M, L), read by the cluster's rank 0
  const int H = a.H, Hkv = a.Hkv;
  const int bh = blockIdx.x, split = blockIdx.y;
  const int b = bh / H, h = bh % H;
  const int g = h / (H / Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvcols = Hkv * D;
  const int pos = a.pos;
  const int jlo = a.window < 0 ? 0 : max(0, pos - a.window);
  const int j0 = jlo + split * kps, j1 = min(pos, j0 + kps);   // cached keys only
  const bool rank0 = split == 0;
  // The split's cached rows (complete before the preceding kernel started) start their way from
  // HBM into L2 now, while the preceding kernel still runs.  A position's keys (values) of all kv
  // heads are one contiguous row of the cache, so the H CTAs of (b, split) share the work: CTA h
  // prefetches every kv head's rows of its H-th of the split's positions, in at most two bulk
  // prefetches per tensor (two when the ring of slots wraps).
  if (tid < 2 && j1 > j0) {
    const int per = (j1 - j0 + H - 1) / H;
    const int p0 = j0 + h * per, p1 = min(j1, p0 + per);
    if (p0 < p1) {
      const bf16* base = (tid ? a.vc : a.kc) + static_cast<size_t>(b) * a.cap * kvcols;
      const uint32_t row_bytes = static_cast<uint32_t>(kvcols) * 2;
      const int s0 = p0 % a.cap, n = p1 - p0, first = min(n, a.cap - s0);
      bulk_prefetch_l2(base + static_cast<size_t>(s0) * kvcols, static_cast<uint32_t>(first) * row_bytes);
      if (n > first) bulk_prefetch_l2(base, static_cast<uint32_t>(n - first) * row_bytes);
    }
  }
  griddep_wait();   // the q|k|v products come from the preceding kernel
  griddep_launch();
  const float* r = a.raw + static_cast<size_t>(b) * a.ldraw;
  {
    // role 0: q head h; role 1 (rank 0 only): k and v of kv head g
    const int role = tid / HALF, j = tid % HALF;
    const bool act = role == 0 || (role == 1 && rank0);
    float c0 = 0.f, c1 = 0.f, ss = 0.f;
    float2 cs = make_float2(0.f, 0.f);
    if (act) {
      const int col = role == 0 ? h * D : (H + g) * D;
      c0 = r[col + j];
      c1 = r[col + j + HALF];
      cs = a.rope[static_cast<size_t>(j) * a.rope_ld + pos];
      ss = c0 * c0 + c1 * c1;
    }
    if (role < 2) {
      ss = warp_sum(ss);
      if (HALF > 32 && lane == 0) s_red[warp] = ss;   // warps 2 role, 2 role + 1
    }
    __syncthreads();
    if (act) {
      if (HALF > 32) ss = s_red[2 * role] + s_red[2 * role + 1];
      const float sc = rsqrtf(ss * (1.0f / D) + a.eps);
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
        const bf16 w0 = __float2bfloat16(v0), w1 = __float2bfloat16(v1);
        s_vn[j] = w0;
        s_vn[j + HALF] = w1;
        if (h % (H / Hkv) == 0) {   // one writer per kv head: the group's first q head
          const size_t slot = (static_cast<size_t>(b) * a.cap + pos % a.cap) * kvcols + static_cast<size_t>(g) * D;
          a.kc[slot + j] = y1;
          a.kc[slot + j + HALF] = y2;
          a.vc[slot + j] = w0;
          a.vc[slot + j + HALF] = w1;
        }
      }
    }
    __syncthreads();
  }
  // Key rows are read whole: LPK lanes per key, 16 B (8 elements) each, so one load instruction
  // of the warp covers KPI complete rows; a lane owns head-dimension elements [8 sub, 8 sub + 8)
  // of its key and accumulates the same elements of its slot's output.
  const int kq = lane / LPK, sub = lane % LPK;   // key within an instruction (the slot), lane's 16 B
  float qv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = s_q[sub * 8 + e];
  float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
  const size_t rowbase = static_cast<size_t>(b) * a.cap * kvcols + g * D + sub * 8;
#pragma unroll 2
  for (int jb = j0 + warp * 8; jb < j1; jb += 32 * DA_WARPS / 4) {   // 8 keys per warp and step
    uint4 kw[KPL], vw[KPL];   // the lane's 16 B of its KPL keys' key and value rows, loaded together
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int j = jb + i * KPI + kq;
      const size_t off = rowbase + static_cast<size_t>((j < j1 ? j : jb) % a.cap) * kvcols;
      kw[i] = __ldg(reinterpret_cast<const uint4*>(a.kc + off));
      vw[i] = __ldg(reinterpret_cast<const uint4*>(a.vc + off));
    }
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int j = jb + i * KPI + kq;
      const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kw[i]);
      float sc = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(k2[t]);
        sc = fmaf(qv[2 * t], f.x, sc);
        sc = fmaf(qv[2 * t + 1], f.y, sc);
      }
#pragma unroll
      for (int off2 = LPK / 2; off2 > 0; off2 >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off2);
      if (j < j1) {   // uniform across the key's LPK lanes
        const float mn = fmaxf(m, sc);
        const float corr = ex2_approx(m - mn);   // 0 on the slot's first key (m = -inf, sc finite)
        const float p = ex2_approx(sc - mn);
        l = fmaf(l, corr, p);
        const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vw[i]);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = __bfloat1622float2(v2[t]);
          o[2 * t] = fmaf(p, f.x, o[2 * t] * corr);
          o[2 * t + 1] = fmaf(p, f.y, o[2 * t + 1] * corr);
        }
        m = mn;
      }
    }
  }
  const int kslot = warp * KPI + kq;
  if (sub == 0) {
    s_m[kslot] = m;
    s_l[kslot] = l;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_o[kslot][sub * 8 + e] = o[e];
  __syncthreads();
  // the CTA's partial: the slots' weights 2^(m_w - M) once (an empty slot weighs 0), then sums
  if (warp == 0) {
    const float mw = lane < SLOTS ? s_m[lane] : -INFINITY;
    const float M = warp_max(mw);
    const float wv = mw == -INFINITY ? 0.f : exp2f(mw - M);
    if (lane < SLOTS) s_w[lane] = wv;
    const float L = warp_sum(lane < SLOTS ? s_l[lane] * wv : 0.f);
    if (lane == 0) {
      s_part[D] = M;
      s_part[D + 1] = L;
    }
  }
  __syncthreads();
  for (int d = tid; d < D; d += 32 * DA_WARPS) {
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < SLOTS; ++w) O = fmaf(s_o[w][d], s_w[w], O);
    s_part[d] = O;
  }
  // The cluster combines: rank 0 reads every CTA's partial from its shared memory in split
  // order, then adds the new key's; the second barrier keeps the peers' shared memory alive
  // until it has.
  cluster_sync();
  if (rank0) {
    // the new key's score q . k_new (base-2 units), a sum over the head dimension
    float dq = tid < D ? s_q[tid] * __bfloat162float(s_kn[tid]) : 0.f;
    dq = warp_sum(dq);
    if (lane == 0) s_red[warp] = dq;
    __syncthreads();
    float snew = 0.f;
#pragma unroll
    for (int w = 0; w < DA_WARPS; ++w) snew += s_red[w];
    const uint32_t base = smem_u32(s_part);
    float Ms[DA_SPLITS], f[DA_SPLITS];
    float Mx = snew;
#pragma unroll
    for (int s2 = 0; s2 < DA_SPLITS; ++s2) {
      Ms[s2] = ld_shared_cluster_f32(mapa_shared(base + D * 4, s2));
      Mx = fmaxf(Mx, Ms[s2]);
    }
    float L = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < DA_SPLITS; ++s2) {   // an empty split (M = -inf) weighs 0
      f[s2] = Ms[s2] == -INFINITY ? 0.f : exp2f(Ms[s2] - Mx);
      L = fmaf(ld_shared_cluster_f32(mapa_shared(base + (D + 1) * 4, s2)), f[s2], L);
    }
    const float fn = exp2f(snew - Mx);
    L += fn;
    for (int d = tid; d < D; d += 32 * DA_WARPS) {
      float O = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < DA_SPLITS; ++s2) O = fmaf(ld_shared_cluster_f32(mapa_shared(base + d * 4, s2)), f[s2], O);
      O = fmaf(__bfloat162float(s_vn[d]), fn, O);
      a.y[static_cast<size_t>(b) * a.ldy + h * D + d] = __float2bfloat16(O / L);
    }
  }
  cluster_sync();
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

cudaError_t launch_decode_attention(const DecodeAttn& a, cudaStream_t stream) {
  if (a.raw == nullptr || a.kc == nullptr || a.vc == nullptr || a.y == nullptr || a.rope == nullptr || a.B < 1 ||
      a.H < 1 || a.Hkv < 1 || a.H % a.Hkv != 0 || a.pos < 0 || a.pos >= a.rope_ld || a.cap < 1 ||
      a.ldy < a.H * a.D || (a.window < 0 ? a.cap <= a.pos : a.cap <= a.window && a.cap <= a.pos) ||
      (a.vgate && (a.ve == nullptr || a.tokens == nullptr)) ||
      a.ldraw < (a.H + a.Hkv) * a.D + a.Hkv * (a.vgate ? a.D + VGATE_ROWS : a.D))
    return cudaErrorInvalidValue;
  if (a.D != 64 && a.D != 128) return cudaErrorInvalidValue;
  const int jlo = a.window < 0 ? 0 : std::max(0, a.pos - a.window);
  const int kps = (a.pos - jlo + DA_SPLITS - 1) / DA_SPLITS;   // cached keys per split (some may be empty)
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;   // the splits of one (row, head)
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = DA_SPLITS;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.gridDim = dim3(a.B * a.H, DA_SPLITS);
  cfg.blockDim = dim3(32 * DA_WARPS);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = a.D == 128 ? cudaLaunchKernelEx(&cfg, decode_attn_kernel<128>, a, scale_log2, kps)
                                   : cudaLaunchKernelEx(&cfg, decode_attn_kernel<64>, a, scale_log2, kps);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace nc
