// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   C[M, N] = epilogue(A[M, K] . B[N, K]^T),  A and B bf16, K contiguous (nn.Linear layout),
//   fp32 accumulation in tensor memory.
//
// CTA pairs (clusters of 2 on neighbouring SMs, one CTA per SM) compute 256x256 tiles with
// the pair form of tcgen05.mma: each CTA holds 128 rows of A and 128 of the 256 rows of B
// in its own shared memory and receives its 128 rows of the fp32 accumulator in its own
// TMEM, so each SM stages 32 KB instead of 48 KB per 64-deep k-block and the tensor cores read
// half of B from the peer.  Persistent grid: min(pair tiles, co-resident pairs); pair tiles
// are taken round-robin with the row-block index fastest (concurrent pairs share a weight tile).
// Roles (320 threads per CTA):
//   warp 0       TMA producer (both CTAs): its A box (128x64) and B half (128x64) per stage,
//                128-byte swizzle, 6-stage ring; both CTAs' copies complete on the leader
//                CTA's full barrier, which the leader arms with the pair's byte count.
//   warp 1       allocates 512 TMEM columns in both CTAs (two 128x256 fp32 accumulators);
//                in the leader one lane issues tcgen05.mma (M=256, N=256, K=16) for the pair;
//                pair commits free each stage in both CTAs and publish each finished
//                accumulator to both CTAs' epilogues.
//   warps 2..9   epilogue: two warpgroups, each owns 128 accumulator columns; every thread
//                owns one output row (TMEM lane).  A warp reads its 32 rows x 128 columns with
//                tcgen05.ld, releases the accumulator, applies the fused epilogue, writes
//                32-row x 128-byte chunks into its own 128-byte-swizzled shared slab and
//                stores each chunk with one TMA bulk-tensor store.
// The double-buffered accumulator lets the epilogue of tile i overlap the MMAs of tile i+1.
//
// Fused epilogues (what each computes is defined on "Nanochat在nanoGPT之上的新增功能",
// section 1 feature table and notes):
//   EPI_RESID_F32    residual add of an output projection (attention c_proj, MLP c_proj);
//                    the residual chunk is read with row-coalesced loads through the slab
//   EPI_RELU2_BF16   squared ReLU of the MLP up projection
//   EPI_SOFTCAP_F32  tanh soft-cap (+-cap) of the untied lm_head logits (hardware tanh)
//   EPI_QKV          split of the packed q|k|v projection; RoPE then per-head RMSNorm of q
//                    and k; on value-embedding layers v += gate * ve[token]
//   EPI_BF16         plain store (used by tests of the mainloop)
#include "internal.h"
#include "ptx.cuh"

#include <mutex>

namespace nc {
namespace {

constexpr int BM = 128;            // rows of A (and of D) held by each CTA of a pair
constexpr int PAIR_M = 2 * BM;     // rows of one pair tile
constexpr int BN = 256;            // columns of one pair tile
constexpr int B_ROWS = BN / 2;     // rows of B (columns of D) loaded by each CTA
constexpr int BK = 64, STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = B_ROWS * BK * 2;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int SLAB_BYTES = 32 * 128;   // per epilogue warp: 32 rows x 128 B

struct __align__(8) Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int OFF_SLAB = STAGES * (A_BYTES + B_BYTES);
constexpr int OFF_CTRL = OFF_SLAB + NUM_EPI_WARPS * SLAB_BYTES;
constexpr int SMEM_BYTES = 1024 + OFF_CTRL + static_cast<int>(sizeof(Ctrl));

// ---------------------------------------------------------------- slab helpers
// A slab holds a [32 rows][128 B] box in the TMA 128-byte swizzle: 16-byte chunk c of row r
// sits at chunk position c ^ (r % 8).

__device__ __forceinline__ uint4* slab_chunk(uint8_t* slab, int r, int c) {
  return reinterpret_cast<uint4*>(slab + r * 128 + ((c ^ (r & 7)) << 4));
}

// Before overwriting the slab: the previous TMA store must have finished reading it.
__device__ __forceinline__ void slab_acquire(int lane) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
}

// Publish the slab to the async proxy and store it as box (x, y) of `map`.
__device__ __forceinline__ void slab_store(uint32_t slab, const CUtensorMap* map, int x, int y, int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, slab, x, y);
    bulk_commit();
  }
}

// Row `lane` of the slab <- 8 x 16 B.
__device__ __forceinline__ void slab_put_row(uint8_t* slab, int lane, const uint4 (&x)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) *slab_chunk(slab, lane, c) = x[c];
}

__device__ __forceinline__ uint4 pack8_bf16(const float* a) {
  return make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]), pack_bf16(a[6], a[7]));
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

struct OutMaps {
  CUtensorMap o0, o1, o2;   // output (EPI_*), or q / k / v (EPI_QKV)
};

// Release an accumulator buffer to the pair's MMA thread (after this warp's last tcgen05.ld
// of it); `bar` is the leader CTA's barrier as a shared::cluster address.
__device__ __forceinline__ void release_acc(int lane, uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(bar);
}

// Epilogue of one warp: rows [m0w, m0w + 32) (this thread: row m0w + lane), accumulator
// columns [n0, n0 + 128) at TMEM address taddr (lane quarter already applied).
template <int KIND, int D>
__device__ __forceinline__ void epilogue_warp(uint32_t taddr, uint32_t tempty, int lane, int m0w, int n0, int M,
                                              int N, const GemmEpi& ep, const OutMaps& om, uint8_t* slab,
                                              uint32_t slab_s) {
  const int m = m0w + lane;
  if constexpr (KIND == EPI_RESID_F32 || KIND == EPI_SOFTCAP_F32) {
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      const int c0 = n0 + ch * 32;
      const bool live = c0 < N;   // warp-uniform (N % 32 == 0)
      uint32_t r[32];
      tmem_ld32(taddr + ch * 32, r);
      float4 rv[8];
      const int rsub = lane >> 3, csub = (lane & 7) * 4;
      if constexpr (KIND == EPI_RESID_F32) {
        // residual chunk [32 rows][32 cols]: each load instruction covers 4 whole rows
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int gm = m0w + k * 4 + rsub;
          rv[k] = (live && gm < M)
                      ? *reinterpret_cast<const float4*>(ep.resid + static_cast<size_t>(gm) * ep.ldr + c0 + csub)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      tmem_ld_wait(r);
      if (ch == 3) release_acc(lane, tempty);
      if (!live) continue;
      slab_acquire(lane);
      if constexpr (KIND == EPI_RESID_F32) {
#pragma unroll
        for (int k = 0; k < 8; ++k) *reinterpret_cast<float4*>(slab_chunk(slab, k * 4 + rsub, lane & 7)) = rv[k];
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float4* p = reinterpret_cast<float4*>(slab_chunk(slab, lane, c));
          float4 x = *p;
          x.x += __uint_as_float(r[c * 4 + 0]);
          x.y += __uint_as_float(r[c * 4 + 1]);
          x.z += __uint_as_float(r[c * 4 + 2]);
          x.w += __uint_as_float(r[c * 4 + 3]);
          *p = x;
        }
      } else {
        const float cap = ep.cap, inv = 1.0f / ep.cap;
        uint4 o[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          o[c] = make_uint4(__float_as_uint(cap * tanh_approx(__uint_as_float(r[c * 4 + 0]) * inv)),
                            __float_as_uint(cap * tanh_approx(__uint_as_float(r[c * 4 + 1]) * inv)),
                            __float_as_uint(cap * tanh_approx(__uint_as_float(r[c * 4 + 2]) * inv)),
                            __float_as_uint(cap * tanh_approx(__uint_as_float(r[c * 4 + 3]) * inv)));
        }
        slab_put_row(slab, lane, o);
      }
      slab_store(slab_s, &om.o0, c0, m0w, lane);
    }
  } else if constexpr (KIND == EPI_BF16 || KIND == EPI_RELU2_BF16) {
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {
      const int c0 = n0 + ch * 64;
      uint32_t r[32], r2[32];
      tmem_ld32(taddr + ch * 64, r);
      tmem_ld32(taddr + ch * 64 + 32, r2);
      tmem_ld_wait(r);
      tmem_ld_wait(r2);
      if (ch == 1) release_acc(lane, tempty);
      if (c0 >= N) continue;
      uint4 o[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = c * 8 + j;
          float t = __uint_as_float(e < 32 ? r[e] : r2[e - 32]);
          if constexpr (KIND == EPI_RELU2_BF16) {
            t = fmaxf(t, 0.f);
            t = t * t;
          }
          a[j] = t;
        }
        o[c] = pack8_bf16(a);
      }
      slab_acquire(lane);
      slab_put_row(slab, lane, o);
      slab_store(slab_s, &om.o0, c0, m0w, lane);
    }
  } else if constexpr (KIND == EPI_QKV) {
    float v[128];
    {
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(taddr + 0, r0);
      tmem_ld32(taddr + 32, r1);
      tmem_ld32(taddr + 64, r2);
      tmem_ld32(taddr + 96, r3);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      tmem_ld_wait(r2);
      tmem_ld_wait(r3);
      release_acc(lane, tempty);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = __uint_as_float(r0[i]);
        v[32 + i] = __uint_as_float(r1[i]);
        v[64 + i] = __uint_as_float(r2[i]);
        v[96 + i] = __uint_as_float(r3[i]);
      }
    }
    const int qcols = ep.H * D, kcols = ep.Hkv * D;
    const int pos = m % ep.T;
#pragma unroll
    for (int s = 0; s < 128 / D; ++s) {
      const int c = n0 + s * D;
      if (c >= N) break;
      float* x = &v[s * D];
      const CUtensorMap* map;
      int xcol;
      if (c < qcols + kcols) {
        rope_rmsnorm<D>(x, ep.rope + static_cast<size_t>(pos) * (D / 2), ep.eps);
        if (c < qcols) {
          map = &om.o0;
          xcol = c;
        } else {
          map = &om.o1;
          xcol = c - qcols;
        }
      } else {
        xcol = c - qcols - kcols;
        map = &om.o2;
        const int hv = xcol / D;
        if (ep.gate != nullptr && m < M) {
          const float g = ep.gate[static_cast<size_t>(m) * ep.Hkv + hv];
          const int tok = ep.tokens[m];
          if (tok >= 0 && tok < ep.V) {
            const uint4* vr = reinterpret_cast<const uint4*>(ep.ve + static_cast<size_t>(tok) * kcols +
                                                             static_cast<size_t>(hv) * D);
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
      }
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint4 o[8];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) o[c8] = pack8_bf16(x + cc * 64 + c8 * 8);
        slab_acquire(lane);
        slab_put_row(slab, lane, o);
        slab_store(slab_s, map, xcol + cc * 64, m0w, lane);
      }
    }
  }
}

template <int KIND, int D>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ OutMaps om, int M, int N, int K, const __grid_constant__ GemmEpi ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + OFF_CTRL);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();            // 0: pair leader (issues the MMAs)
  const int pair = static_cast<int>(blockIdx.x) >> 1, npairs = static_cast<int>(gridDim.x) >> 1;
  const int num_m = (M + PAIR_M - 1) / PAIR_M, num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n, kblocks = K / BK;
  int* status = ep.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), 2 * NUM_EPI_WARPS);
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
    tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        const int mb = tile % num_m, nb = tile / num_m;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&ctl->empty[s]), ph ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(smem_u32(&ctl->full[s]), 0);   // the leader's barrier
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), 2 * (A_BYTES + B_BYTES));
          tma_load_2d_pair(sA + s * A_BYTES, &tmA, fb, kb * BK, mb * PAIR_M + static_cast<int>(rank) * BM);
          tma_load_2d_pair(sB + s * B_BYTES, &tmB, fb, kb * BK, nb * BN + static_cast<int>(rank) * B_ROWS);
          ++it;
        }
      }
      // The leader's full barriers count both CTAs' copies: once its last phases completed,
      // every copy issued by the pair has landed (the peer exits only after the final sync).
      if (rank == 0) {
        for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_cluster(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1, nullptr, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(PAIR_M, BN);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs, ++tc) {
        const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
        if (!mbar_wait_cluster(smem_u32(&ctl->tempty[a]), aph ^ 1, abort, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&ctl->full[s]), ph, abort, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma_bf16_pair(d_tmem, sdesc_kmajor_sw128(sA + s * A_BYTES + kk * 32),
                           sdesc_kmajor_sw128(sB + s * B_BYTES + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&ctl->empty[s]), 0x3);
          ++it;
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&ctl->tfull[a]), 0x3);
      }
      umma_commit_pair(smem_u32(&ctl->drain), 0x1);
      mbar_wait(smem_u32(&ctl->drain), 0, nullptr, status);
    }
    __syncwarp();
  } else {
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int group = ew >> 2;
    uint8_t* slab = smem + OFF_SLAB + ew * SLAB_BYTES;
    const uint32_t slab_s = smem_u32(slab);
    uint32_t tc = 0;
    for (int tile = pair; tile < num_tiles; tile += npairs, ++tc) {
      const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
      const bool ok = mbar_wait_cluster(smem_u32(&ctl->tfull[a]), aph, abort, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * BN + group * 128;
      const int mb = tile % num_m, nb = tile / num_m;
      epilogue_warp<KIND, D>(taddr, mapa_shared(smem_u32(&ctl->tempty[a]), 0), lane,
                             mb * PAIR_M + static_cast<int>(rank) * BM + quarter * 32, nb * BN + group * 128, M, N,
                             ep, om, slab, slab_s);
    }
    if (lane == 0) bulk_wait<0>();   // stores complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();   // all MMAs done and all TMEM reads of both CTAs finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <int KIND, int D>
cudaError_t launch_kind(const CUtensorMap& ta, const CUtensorMap& tb, const OutMaps& om, int M, int N, int K,
                        const GemmEpi& epi, int num_sms, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_pairs = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<KIND, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * (num_sms / 2));
    if (cudaOccupancyMaxActiveClusters(&max_pairs, gemm_tc_kernel<KIND, D>, &q) != cudaSuccess || max_pairs < 1)
      max_pairs = num_sms / 2;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int tiles = ((M + PAIR_M - 1) / PAIR_M) * ((N + BN - 1) / BN);
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<KIND, D>, ta, tb, om, M, N, K, epi);
}

}  // namespace

cudaError_t launch_gemm(const bf16* A, const bf16* B, int M, int N, int K, const GemmEpi& epi,
                        int num_sms, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || K % BK != 0 || N % 32 != 0) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, A, K, M, static_cast<uint64_t>(K) * 2, BK, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_2d(&tb, B, K, N, static_cast<uint64_t>(K) * 2, BK, B_ROWS)) return cudaErrorInvalidValue;
  OutMaps om;
  const uint64_t Mu = static_cast<uint64_t>(M);
  bool ok = true;
  switch (epi.kind) {
    case EPI_RESID_F32:
    case EPI_SOFTCAP_F32:
      ok = make_tmap_2d(&om.o0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, epi.out, N, Mu, static_cast<uint64_t>(epi.ldo) * 4, 32, 32);
      break;
    case EPI_BF16:
    case EPI_RELU2_BF16:
      ok = make_tmap_bf16_2d(&om.o0, epi.out, N, Mu, static_cast<uint64_t>(epi.ldo) * 2, 64, 32);
      break;
    case EPI_QKV: {
      const uint64_t qc = static_cast<uint64_t>(epi.H) * epi.D, kc = static_cast<uint64_t>(epi.Hkv) * epi.D;
      ok = make_tmap_bf16_2d(&om.o0, epi.q, qc, Mu, qc * 2, 64, 32) &&
           make_tmap_bf16_2d(&om.o1, epi.k, kc, Mu, kc * 2, 64, 32) &&
           make_tmap_bf16_2d(&om.o2, epi.v, kc, Mu, kc * 2, 64, 32);
      break;
    }
    default: return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  switch (epi.kind) {
    case EPI_BF16: return launch_kind<EPI_BF16, 0>(ta, tb, om, M, N, K, epi, num_sms, stream);
    case EPI_RESID_F32: return launch_kind<EPI_RESID_F32, 0>(ta, tb, om, M, N, K, epi, num_sms, stream);
    case EPI_RELU2_BF16: return launch_kind<EPI_RELU2_BF16, 0>(ta, tb, om, M, N, K, epi, num_sms, stream);
    case EPI_SOFTCAP_F32: return launch_kind<EPI_SOFTCAP_F32, 0>(ta, tb, om, M, N, K, epi, num_sms, stream);
    case EPI_QKV:
      if (epi.D == 128) return launch_kind<EPI_QKV, 128>(ta, tb, om, M, N, K, epi, num_sms, stream);
      if (epi.D == 64) return launch_kind<EPI_QKV, 64>(ta, tb, om, M, N, K, epi, num_sms, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nc
