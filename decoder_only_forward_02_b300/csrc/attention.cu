// attention.cu -- causal grouped-query attention with a per-layer left window, on tcgen05.
//
//   y[b, i, h, :] = sum_j softmax_j(q[b,i,h] . k[b,j,g] / sqrt(D)) v[b,j,g],   g = h / (H/Hkv),
//   over keys max(0, i - W) <= j <= i (all j <= i when W < 0).
//
// "Nanochat在nanoGPT之上的新增功能", section 1 table: grouped-query attention (fewer kv heads
// than query heads) and per-layer sliding-window attention; the notes give the repeating
// three-short-one-long pattern with the last layer full.  "nanochat — 架构与原理", section 5:
// the reference's Blackwell path falls back to an attention without windows, so windows there
// cost full causal work; here key tiles outside the window are never loaded.
//
// One CTA per (128-query tile, head, batch row), two CTAs per SM (112 KB shared memory and
// 256 TMEM columns each).  Heaviest query tiles are dispatched first.
//   warp 0      TMA: Q tile once, then 64-key K and V tiles into a 2-stage ring.
//   warp 1      TMEM allocation; one lane issues S = Q K^T (128 x 64, fp32 in TMEM) and
//               O += P V (128 x D, fp32 in TMEM; V read MN-major straight from its
//               token-major layout).
//   warps 2..5  softmax, one thread per query row: read its S row from TMEM, mask (causal,
//               window, sequence end), online softmax in base 2 with the scale folded into
//               one FMA, P as bf16 into a 128-byte-swizzled shared tile (the A operand of
//               P V).  The running max moves only when a row's max grows by more than 2^8;
//               only then is that row of O rescaled in TMEM (after the previous P V is done).
//               Final: O / l -> bf16 -> y.
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace nc {
namespace {

constexpr int BQ = 128, BKV = 64, STAGES = 2, THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;   // S: columns [0, 64); O: [64, 64 + D)

struct __align__(8) AttnCtrl {
  uint64_t q_full;
  uint64_t kv_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full, s_free, p_full, o_done, drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct Lay {
  static constexpr int Q_BOX = BQ * 64 * 2;     // [128 rows][64 d] bf16, 16 KB
  static constexpr int KV_BOX = BKV * 64 * 2;   // [64 keys][64 d] bf16, 8 KB
  static constexpr int NB = D / 64;             // boxes along d
  static constexpr int Q_BYTES = NB * Q_BOX;
  static constexpr int K_BYTES = NB * KV_BOX;
  static constexpr int P_BYTES = BQ * BKV * 2;  // [128 rows][64 keys] bf16, 16 KB
  static constexpr int OFF_P = Q_BYTES;
  static constexpr int OFF_KV = OFF_P + P_BYTES;
  static constexpr int STAGE_BYTES = 2 * K_BYTES;  // K then V
  static constexpr int OFF_CTRL = OFF_KV + STAGES * STAGE_BYTES;
  static constexpr int TOTAL = OFF_CTRL + 256;
};

template <int D>
__global__ void __launch_bounds__(THREADS, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, int T, int H, int Hkv, int B, int window,
                   float scale_log2, bf16* __restrict__ y, int* status) {
  using L = Lay<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {   // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_error(status, NC_ERR_UNSUPPORTED);
    return;
  }
  AttnCtrl* ctl = reinterpret_cast<AttnCtrl*>(smem + L::OFF_CTRL);
  const uint32_t sQ = smem_u32(smem), sP = sQ + L::OFF_P, sKV = sQ + L::OFF_KV;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HB = H * B;
  const int nq = (T + BQ - 1) / BQ;
  const int qt = nq - 1 - static_cast<int>(blockIdx.x) / HB;   // heaviest tiles first
  const int hb = static_cast<int>(blockIdx.x) % HB;
  const int h = hb % H, b = hb / H;
  const int g = h / (H / Hkv);
  const int q0 = qt * BQ;
  const int q_last = min(q0 + BQ - 1, T - 1);
  const int k_lo = window < 0 ? 0 : max(0, q0 - window);
  const int j0 = k_lo / BKV;
  const int n = q_last / BKV - j0 + 1;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_full), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->kv_full[s]), 1);
      mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->s_full), 1);
    mbar_init(smem_u32(&ctl->s_free), 4);
    mbar_init(smem_u32(&ctl->p_full), 4);
    mbar_init(smem_u32(&ctl->o_done), 1);
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const uint32_t tS = tmem, tO = tmem + BKV;
  volatile int* abort = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint32_t qb = smem_u32(&ctl->q_full);
      mbar_arrive_expect_tx(qb, L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < L::NB; ++c) tma_load_2d(sQ + c * L::Q_BOX, &tmQ, qb, h * D + c * 64, b * T + q0);
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (j / STAGES) & 1;
        if (!mbar_wait(smem_u32(&ctl->kv_empty[s]), ph ^ 1, abort, status)) break;
        const uint32_t fb = smem_u32(&ctl->kv_full[s]);
        mbar_arrive_expect_tx(fb, L::STAGE_BYTES);
        const int row = b * T + (j0 + j) * BKV;
        const uint32_t sK = sKV + s * L::STAGE_BYTES, sV = sK + L::K_BYTES;
#pragma unroll
        for (int c = 0; c < L::NB; ++c) {
          tma_load_2d(sK + c * L::KV_BOX, &tmK, fb, g * D + c * 64, row);
          tma_load_2d(sV + c * L::KV_BOX, &tmV, fb, g * D + c * 64, row);
        }
        ++issued;
      }
      // every issued copy must land before the CTA may exit
      mbar_wait(qb, 0, nullptr, status);
      for (int j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j)
        mbar_wait(smem_u32(&ctl->kv_full[j % STAGES]), (j / STAGES) & 1, nullptr, status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BQ, BKV);
      constexpr uint32_t idO = idesc_bf16_f32_bmn(BQ, D);
      bool ok = mbar_wait(smem_u32(&ctl->q_full), 0, abort, status);
      auto issue_s = [&](int j) -> bool {
        const int s = j % STAGES;
        if (!mbar_wait(smem_u32(&ctl->kv_full[s]), (j / STAGES) & 1, abort, status)) return false;
        tc_fence_after();
        const uint32_t sK = sKV + s * L::STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sdesc_kmajor_sw128(sQ + (kk / 4) * L::Q_BOX + (kk % 4) * 32);
          const uint64_t bd = sdesc_kmajor_sw128(sK + (kk / 4) * L::KV_BOX + (kk % 4) * 32);
          umma_bf16(tS, a, bd, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&ctl->s_full));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n) {
          if (!mbar_wait(smem_u32(&ctl->s_free), j & 1, abort, status)) break;
          tc_fence_after();
          if (!issue_s(j + 1)) break;
        }
        if (!mbar_wait(smem_u32(&ctl->p_full), j & 1, abort, status)) break;
        tc_fence_after();
        const int s = j % STAGES;
        const uint32_t sV = sKV + s * L::STAGE_BYTES + L::K_BYTES;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const uint64_t a = sdesc_kmajor_sw128(sP + kk * 32);
          const uint64_t bd = sdesc_mnmajor_sw128(sV + kk * 16 * 128, L::KV_BOX);
          umma_bf16(tO, a, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&ctl->o_done));
        umma_commit(smem_u32(&ctl->kv_empty[s]));
      }
      umma_commit(smem_u32(&ctl->drain));
      mbar_wait(smem_u32(&ctl->drain), 0, nullptr, status);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int i = q0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float thr = 8.0f / scale_log2;   // raw-score growth that triggers a rescale (2^8)
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full), j & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tS + lane_off, r0);
      tmem_ld32(tS + lane_off + 32, r1);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free));

      const int key0 = (j0 + j) * BKV;
      // Tiles inside every row's visible range need no per-element mask: the last key is at
      // most the first query, the tile lies inside the sequence, and (with a window) its first
      // key is within the window of the last query.  The test is the same for the whole CTA.
      const bool interior = key0 + BKV - 1 <= q0 && key0 + BKV <= T &&
                            (window < 0 || key0 >= q0 + BQ - 1 - window);
      float s[BKV];
      if (interior) {
#pragma unroll
        for (int c = 0; c < BKV; ++c) s[c] = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
      } else {
        const int kmin = window < 0 ? 0 : i - window;
        const int kmax = min(i, T - 1);
#pragma unroll
        for (int c = 0; c < BKV; ++c) {
          const int key = key0 + c;
          const float v = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
          s[c] = (key <= kmax && key >= kmin) ? v : -INFINITY;
        }
      }
      // row max as 8 independent chains and a 3-level tree
      float mx[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx[q] = s[q];
#pragma unroll
      for (int c = 8; c < BKV; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_run + thr) {
        alpha = ex2_approx((m_run - mt) * scale_log2);   // 0 when m_run = -inf
        resc = m_run != -INFINITY;
        m_run = mt;
      }
      const float negm = (m_run == -INFINITY) ? 0.f : -m_run * scale_log2;
      uint32_t pk[BKV / 2];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};   // 4 independent partial sums
#pragma unroll
      for (int c = 0; c < BKV; c += 2) {
        const float p0 = ex2_approx(fmaf(s[c], scale_log2, negm));
        const float p1 = ex2_approx(fmaf(s[c + 1], scale_log2, negm));
        ps[(c >> 1) & 3] += p0 + p1;
        pk[c / 2] = pack_bf16(p0, p1);
      }
      const float sum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      l_run = l_run * alpha + sum;

      if (j > 0) {   // P V of the previous tile must be done before P and O are touched
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_done), (j - 1) & 1, abort, status));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
        const float a = resc ? alpha : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + ch * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
          tmem_st32(tO + lane_off + ch * 32, o);
        }
        tmem_st_wait();
      }
      uint8_t* prow = smem + L::OFF_P + row * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 v = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_done), (n - 1) & 1, abort, status));
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      bf16* dst = y + (static_cast<size_t>(b) * T + i) * (static_cast<size_t>(H) * D) + h * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + ch * 32, o);
        tmem_ld_wait(o);
        if (i < T) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[c8 * 8 + 0]) * inv, __uint_as_float(o[c8 * 8 + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(o[c8 * 8 + 2]) * inv, __uint_as_float(o[c8 * 8 + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(o[c8 * 8 + 4]) * inv, __uint_as_float(o[c8 * 8 + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(o[c8 * 8 + 6]) * inv, __uint_as_float(o[c8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + ch * 32 + c8 * 8) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H, int Hkv, int window,
                     bf16* y, int* status, cudaStream_t stream) {
  using Lt = Lay<D>;
  static cudaError_t attr =
      cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lt::TOTAL);
  if (attr != cudaSuccess) return attr;
  const uint64_t M = static_cast<uint64_t>(B) * T;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_2d(&tq, q, static_cast<uint64_t>(H) * D, M, static_cast<uint64_t>(H) * D * 2, 64, BQ) ||
      !make_tmap_bf16_2d(&tk, k, static_cast<uint64_t>(Hkv) * D, M, static_cast<uint64_t>(Hkv) * D * 2, 64, BKV) ||
      !make_tmap_bf16_2d(&tv, v, static_cast<uint64_t>(Hkv) * D, M, static_cast<uint64_t>(Hkv) * D * 2, 64, BKV))
    return cudaErrorInvalidValue;
  const int nq = (T + BQ - 1) / BQ;
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  attn_tc_kernel<D><<<nq * H * B, THREADS, Lt::TOTAL, stream>>>(tq, tk, tv, T, H, Hkv, B, window, scale_log2, y,
                                                                 status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H,
                             int Hkv, int D, int window, bf16* y, int* status, cudaStream_t stream) {
  if (D == 128) return launch_d<128>(q, k, v, B, T, H, Hkv, window, y, status, stream);
  if (D == 64) return launch_d<64>(q, k, v, B, T, H, Hkv, window, y, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nc
