// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   C[M, N] = epilogue(A[M, K] . B[N, K]^T),  A and B bf16, K contiguous (nn.Linear layout),
//   fp32 accumulation in tensor memory.
//
// Roles (320 threads, one CTA per SM, grid = min(tiles, SMs), static round-robin tiles):
//   warp 0       TMA producer: 128x64 A box + 256x64 B box per stage, 128-byte swizzle,
//                4-stage shared-memory ring guarded by full/empty mbarriers.
//   warp 1       allocates 512 TMEM columns (two 128x256 fp32 accumulators) and issues
//                tcgen05.mma 128x256x16 from one lane; tcgen05.commit frees each stage and
//                publishes each finished accumulator.
//   warps 2..9   epilogue: two warpgroups, each owns 128 accumulator columns; every thread
//                owns one output row (TMEM lane), reads its 128 columns with tcgen05.ld,
//                releases the accumulator, then applies the fused epilogue and stores.
// The double-buffered accumulator lets the epilogue of tile i overlap the MMAs of tile i+1.
//
// Fused epilogues (what each computes is defined on "Nanochat在nanoGPT之上的新增功能",
// section 1 feature table and notes):
//   EPI_RESID_F32    residual add of an output projection (attention c_proj, MLP c_proj)
//   EPI_RELU2_BF16   squared ReLU of the MLP up projection
//   EPI_SOFTCAP_F32  tanh soft-cap of the untied lm_head logits
//   EPI_QKV          split of the packed q|k|v projection; RoPE then per-head RMSNorm of q
//                    and k; on value-embedding layers v += gate * ve[token]
//   EPI_BF16         plain store (used by tests of the mainloop)
#include "internal.h"
#include "ptx.cuh"

#include <cstdio>
#include <mutex>

namespace nc {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 2 * BN;

struct __align__(8) Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int SMEM_BYTES = 1024 + STAGES * (A_BYTES + B_BYTES) + static_cast<int>(sizeof(Ctrl));

__device__ __forceinline__ void store_bf16x8(bf16* dst, const float* a) {
  uint4 p;
  p.x = pack_bf16(a[0], a[1]);
  p.y = pack_bf16(a[2], a[3]);
  p.z = pack_bf16(a[4], a[5]);
  p.w = pack_bf16(a[6], a[7]);
  *reinterpret_cast<uint4*>(dst) = p;
}

// Rotate pairs (d, d + D/2) by the position's angles, then RMS-normalise over the head.
template <int D>
__device__ __forceinline__ void rope_rmsnorm(float* x, const float2* rope_row, float eps) {
  const float4* rp = reinterpret_cast<const float4*>(rope_row);
#pragma unroll
  for (int d2 = 0; d2 < D / 4; ++d2) {
    const float4 cs = __ldg(rp + d2);
    const int d = 2 * d2;
    float x1 = x[d], x2 = x[d + D / 2];
    x[d] = x1 * cs.x + x2 * cs.y;
    x[d + D / 2] = -x1 * cs.y + x2 * cs.x;
    x1 = x[d + 1];
    x2 = x[d + 1 + D / 2];
    x[d + 1] = x1 * cs.z + x2 * cs.w;
    x[d + 1 + D / 2] = -x1 * cs.w + x2 * cs.z;
  }
  float ss = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d) ss = fmaf(x[d], x[d], ss);
  const float r = rsqrtf(ss * (1.0f / D) + eps);
#pragma unroll
  for (int d = 0; d < D; ++d) x[d] *= r;
}

// Epilogue for one thread: row m, columns [n0, n0 + 128).
template <int KIND, int D>
__device__ __forceinline__ void epilogue_row(float (&v)[128], int m, int n0, int M, int N,
                                             const GemmEpi& ep) {
  if (m >= M) return;
  if constexpr (KIND == EPI_BF16 || KIND == EPI_RELU2_BF16) {
    bf16* out = static_cast<bf16*>(ep.out) + static_cast<size_t>(m) * ep.ldo + n0;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if (n0 + c * 8 < N) {
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float t = v[c * 8 + j];
          if constexpr (KIND == EPI_RELU2_BF16) {
            t = fmaxf(t, 0.f);
            t = t * t;
          }
          a[j] = t;
        }
        store_bf16x8(out + c * 8, a);
      }
    }
  } else if constexpr (KIND == EPI_RESID_F32) {
    float* out = static_cast<float*>(ep.out) + static_cast<size_t>(m) * ep.ldo + n0;
    const float* res = ep.resid + static_cast<size_t>(m) * ep.ldr + n0;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if (n0 + c * 4 < N) {
        float4 r = *reinterpret_cast<const float4*>(res + c * 4);
        r.x += v[c * 4 + 0];
        r.y += v[c * 4 + 1];
        r.z += v[c * 4 + 2];
        r.w += v[c * 4 + 3];
        *reinterpret_cast<float4*>(out + c * 4) = r;
      }
    }
  } else if constexpr (KIND == EPI_SOFTCAP_F32) {
    float* out = static_cast<float*>(ep.out) + static_cast<size_t>(m) * ep.ldo + n0;
    const float cap = ep.cap, inv = 1.0f / ep.cap;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if (n0 + c * 4 < N) {
        float4 o;
        o.x = cap * tanhf(v[c * 4 + 0] * inv);
        o.y = cap * tanhf(v[c * 4 + 1] * inv);
        o.z = cap * tanhf(v[c * 4 + 2] * inv);
        o.w = cap * tanhf(v[c * 4 + 3] * inv);
        *reinterpret_cast<float4*>(out + c * 4) = o;
      }
    }
  } else if constexpr (KIND == EPI_QKV) {
    const int qcols = ep.H * D, kcols = ep.Hkv * D;
    const int pos = m % ep.T;
#pragma unroll
    for (int s = 0; s < 128 / D; ++s) {
      const int c = n0 + s * D;
      if (c >= N) continue;
      float* x = &v[s * D];
      bf16* dst;
      if (c < qcols + kcols) {
        rope_rmsnorm<D>(x, ep.rope + static_cast<size_t>(pos) * (D / 2), ep.eps);
        dst = (c < qcols) ? ep.q + static_cast<size_t>(m) * qcols + c
                          : ep.k + static_cast<size_t>(m) * kcols + (c - qcols);
      } else {
        const int hv = (c - qcols - kcols) / D;
        if (ep.gate != nullptr) {
          const float g = ep.gate[static_cast<size_t>(m) * ep.Hkv + hv];
          const int tok = ep.tokens[m];
          if (tok >= 0 && tok < ep.V) {
            const uint4* vr = reinterpret_cast<const uint4*>(
                ep.ve + static_cast<size_t>(tok) * kcols + static_cast<size_t>(hv) * D);
#pragma unroll
            for (int c8 = 0; c8 < D / 8; ++c8) {
              const uint4 u = __ldg(vr + c8);
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h2[j]);
                x[c8 * 8 + 2 * j] = fmaf(g, f.x, x[c8 * 8 + 2 * j]);
                x[c8 * 8 + 2 * j + 1] = fmaf(g, f.y, x[c8 * 8 + 2 * j + 1]);
              }
            }
          }
        }
        dst = ep.v + static_cast<size_t>(m) * kcols + (c - qcols - kcols);
      }
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8) store_bf16x8(dst + c8 * 8, x + c8 * 8);
    }
  }
}

template <int KIND, int D>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   int M, int N, int K, const __grid_constant__ GemmEpi ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + STAGES * (A_BYTES + B_BYTES));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n, kblocks = K / BK;
  int* status = ep.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), NUM_EPI_WARPS);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int mb = tile % num_m, nb = tile / num_m;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
          tma_load_2d(sA + s * A_BYTES, &tmA, fb, kb * BK, mb * BM);
          tma_load_2d(sB + s * B_BYTES, &tmB, fb, kb * BK, nb * BN);
          ++it;
        }
      }
      // Every issued load must land before the CTA may exit.
      for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
        mbar_wait(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1, nullptr, status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tc) {
        const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
        if (!mbar_wait(smem_u32(&ctl->tempty[a]), aph ^ 1, abort, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma_bf16(d_tmem, sdesc_kmajor_sw128(sA + s * A_BYTES + kk * 32),
                      sdesc_kmajor_sw128(sB + s * B_BYTES + kk * 32), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&ctl->empty[s]));
          ++it;
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctl->tfull[a]));
      }
      umma_commit(smem_u32(&ctl->drain));
      mbar_wait(smem_u32(&ctl->drain), 0, nullptr, status);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int group = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
      const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
      const bool ok = mbar_wait(smem_u32(&ctl->tfull[a]), aph, abort, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * BN + group * 128;
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(taddr + 0, r0);
      tmem_ld32(taddr + 32, r1);
      tmem_ld32(taddr + 64, r2);
      tmem_ld32(taddr + 96, r3);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      tmem_ld_wait(r2);
      tmem_ld_wait(r3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[a]));
      float v[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = __uint_as_float(r0[i]);
        v[32 + i] = __uint_as_float(r1[i]);
        v[64 + i] = __uint_as_float(r2[i]);
        v[96 + i] = __uint_as_float(r3[i]);
      }
      const int mb = tile % num_m, nb = tile / num_m;
      epilogue_row<KIND, D>(v, mb * BM + row, nb * BN + group * 128, M, N, ep);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int KIND, int D>
cudaError_t launch_kind(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K,
                        const GemmEpi& epi, int num_sms, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<KIND, D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  gemm_tc_kernel<KIND, D><<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, M, N, K, epi);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const bf16* A, const bf16* B, int M, int N, int K, const GemmEpi& epi,
                        int num_sms, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || K % BK != 0 || N % 32 != 0) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, A, K, M, static_cast<uint64_t>(K) * 2, BK, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&tb, B, K, N, static_cast<uint64_t>(K) * 2, BK, BN)) return cudaErrorInvalidValue;
  switch (epi.kind) {
    case EPI_BF16: return launch_kind<EPI_BF16, 0>(ta, tb, M, N, K, epi, num_sms, stream);
    case EPI_RESID_F32: return launch_kind<EPI_RESID_F32, 0>(ta, tb, M, N, K, epi, num_sms, stream);
    case EPI_RELU2_BF16: return launch_kind<EPI_RELU2_BF16, 0>(ta, tb, M, N, K, epi, num_sms, stream);
    case EPI_SOFTCAP_F32: return launch_kind<EPI_SOFTCAP_F32, 0>(ta, tb, M, N, K, epi, num_sms, stream);
    case EPI_QKV:
      if (epi.D == 128) return launch_kind<EPI_QKV, 128>(ta, tb, M, N, K, epi, num_sms, stream);
      if (epi.D == 64) return launch_kind<EPI_QKV, 64>(ta, tb, M, N, K, epi, num_sms, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nc
