// quant.cu -- tensorwise e4m3 quantisation for the 8-bit linear layers.
//
// "Nanochat在nanoGPT之上的新增功能", section 1 feature table (FP8 training: dynamic tensor-level
// scaling, e4m3 in the forward) and "nanochat — 架构与原理", section 4 (a scaled matrix product with
// the quantisation inside).  Every linear layer's input activation and weight are quantised as
// whole tensors: s = 448 / max|v| (448 the largest finite e4m3 value; s = 1 for an all-zero
// tensor), q = e4m3(v * s) rounded to nearest even and saturating, and the product is divided by
// the two scales afterwards (the GEMM epilogue multiplies by the stored 1 / s values).
//
//   fp8_amax      one warp per row (grid-stride), per-block maxima of |v| (times the row's RMSNorm
//                 scale when the input is a normed residual stream) -> partial[FP8_AMAX_BLOCKS]
//   fp8_amax_rows the same per-block maxima of a row-scaled stream from its producer's per-row
//                 maxima over 32-column groups (the residual GEMM writes them), reading 1/32 of it
//   fp8_quantize  every block first reduces the partial maxima (the same fixed order in every
//                 block; a single word when the producer kept the maximum itself), then one warp per row converts 8 elements per lane-step to e4m3.  The
//                 scaled value is (v * 448) / amax, not v * (448 / amax): for bf16 v the product
//                 is exact, so a value that the exact scaling puts on a rounding tie of the e4m3
//                 grid (frequent: bf16 values have few significant bits) stays exactly on it and
//                 rounds to even, as in exact arithmetic.  The quotient takes one reciprocal per
//                 thread and a residual correction per element (q0 = p r, e = p - q0 a exactly by
//                 fma, q = q0 + e r), which returns the exact quotient whenever it is representable
//                 (every rounding tie is) and the correctly rounded one otherwise but for rare
//                 boundary cases; no per-element division.
// Both kernels keep four 16- or 32-byte loads per lane in flight (a row's chunks are loaded before
// they are reduced or converted).
// No atomics here; the producers' maxima are exact (order-independent): the scale and the codes are
// the same on every run.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_fp8.h>

namespace nc {
namespace {

constexpr int QT = 256;   // threads per block (8 warps)

__device__ __forceinline__ void load8(const void* src, int f32, size_t off, float (&v)[8]) {
  if (f32) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(src) + off);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(src) + off + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(src) + off);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  }
}

// The row's RMSNorm scale from its C / 128 partial sums of squares (1 without ssp).
__device__ __forceinline__ float row_scale(const float* ssp, int row, int C, float eps, int lane) {
  if (ssp == nullptr) return 1.f;
  const int ncg = C / SS_GROUP;
  float s = 0.f;
  for (int g = lane; g < ncg; g += 32) s += ssp[static_cast<size_t>(row) * ncg + g];
  s = warp_sum(s);
  return rsqrtf(s * (1.0f / C) + eps);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int UNR = 4;   // chunks of 8 elements per lane loaded before use

__global__ void __launch_bounds__(QT) fp8_amax_kernel(const void* __restrict__ src, int f32, int M, int C, int ld,
                                                      const float* __restrict__ ssp, float eps,
                                                      float* __restrict__ partial) {
  __shared__ float sh[QT / 32];
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = gridDim.x * (QT / 32);
  float mx = 0.f;
  for (int row = blockIdx.x * (QT / 32) + warp; row < M; row += nw) {
    const float rs = row_scale(ssp, row, C, eps, lane);
    float m = 0.f;
    for (int c0 = lane * 8; c0 < C; c0 += 256 * UNR) {
      float v[UNR][8];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (c0 + u * 256 < C) load8(src, f32, static_cast<size_t>(row) * ld + c0 + u * 256, v[u]);
        else
#pragma unroll
          for (int j = 0; j < 8; ++j) v[u][j] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[u][j]));
    }
    mx = fmaxf(mx, m * rs);
  }
  mx = warp_max(mx);
  if (lane == 0) sh[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < QT / 32; ++w) b = fmaxf(b, sh[w]);
    partial[blockIdx.x] = b;
  }
}

// The same per-block maxima as fp8_amax_kernel for a row-scaled fp32 stream, from its per-row,
// per-32-column maxima of |v| (written by the producer's epilogue): one warp per row.
__global__ void __launch_bounds__(QT) fp8_amax_rows_kernel(const float* __restrict__ rowmax, int M, int C,
                                                           const float* __restrict__ ssp, float eps,
                                                           float* __restrict__ partial) {
  __shared__ float sh[QT / 32];
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = gridDim.x * (QT / 32), ng = C / 32;
  float mx = 0.f;
  for (int row = blockIdx.x * (QT / 32) + warp; row < M; row += nw) {
    const float rs = row_scale(ssp, row, C, eps, lane);
    float m = 0.f;
    for (int gi = lane; gi < ng; gi += 32) m = fmaxf(m, rowmax[static_cast<size_t>(row) * ng + gi]);
    mx = fmaxf(mx, m * rs);
  }
  mx = warp_max(mx);
  if (lane == 0) sh[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < QT / 32; ++w) b = fmaxf(b, sh[w]);
    partial[blockIdx.x] = b;
  }
}

__global__ void __launch_bounds__(QT) fp8_quantize_kernel(const void* __restrict__ src, int f32, int M, int C, int ld,
                                                          const float* __restrict__ ssp, float eps,
                                                          const float* __restrict__ partial, int npart,
                                                          uint8_t* __restrict__ dst, int ld_dst, int group, int gap,
                                                          float* __restrict__ inv_scale) {
  __shared__ float sh[QT / 32];
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float a = 0.f;
  for (int i = threadIdx.x; i < npart; i += QT) a = fmaxf(a, partial[i]);
  a = warp_max(a);
  if (lane == 0) sh[warp] = a;
  __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int w = 0; w < QT / 32; ++w) amax = fmaxf(amax, sh[w]);
  const bool scaled = amax > 0.f;   // an all-zero tensor keeps scale 1
  if (blockIdx.x == 0 && threadIdx.x == 0) *inv_scale = scaled ? amax / 448.0f : 1.0f;
  const float den = scaled ? amax : 1.0f;
  const float rden = 1.0f / den;   // one reciprocal per thread
  const int nw = gridDim.x * (QT / 32);
  for (int row = blockIdx.x * (QT / 32) + warp; row < M; row += nw) {
    const float k = row_scale(ssp, row, C, eps, lane) * (scaled ? 448.0f : 1.0f);
    const int drow = group > 0 ? row + (row / group) * gap : row;
    for (int c0 = lane * 8; c0 < C; c0 += 256 * UNR) {
      float v[UNR][8];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        if (c0 + u * 256 < C) load8(src, f32, static_cast<size_t>(row) * ld + c0 + u * 256, v[u]);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (c0 + u * 256 >= C) break;
        float p[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // (v k) / den: q0 = p r, exact residual, one correction
          const float n = v[u][j] * k;
          const float q0 = n * rden;
          p[j] = fmaf(fmaf(-q0, den, n), rden, q0);
        }
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const __nv_fp8x2_storage_t lo =
              __nv_cvt_float2_to_fp8x2(make_float2(p[4 * h], p[4 * h + 1]), __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t hi =
              __nv_cvt_float2_to_fp8x2(make_float2(p[4 * h + 2], p[4 * h + 3]), __NV_SATFINITE, __NV_E4M3);
          w[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        *reinterpret_cast<uint2*>(dst + static_cast<size_t>(drow) * ld_dst + c0 + u * 256) = make_uint2(w[0], w[1]);
      }
    }
  }
}

template <typename K, typename... Args>
cudaError_t launch_q(K kernel, int grid, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(QT);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

bool q_args_ok(const void* src, int src_f32, int M, int C, int ld, const float* ssp) {
  const size_t esz = src_f32 ? 4 : 2;
  return src != nullptr && M >= 1 && C >= 8 && C % 8 == 0 && ld >= C && (ld * esz) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(src) % 16 == 0 && (ssp == nullptr || C % SS_GROUP == 0);
}

}  // namespace

cudaError_t launch_fp8_amax(const void* src, int src_f32, int M, int C, int ld, const float* ssp, float eps,
                            float* partial, cudaStream_t stream) {
  if (!q_args_ok(src, src_f32, M, C, ld, ssp) || partial == nullptr) return cudaErrorInvalidValue;
  return launch_q(fp8_amax_kernel, FP8_AMAX_BLOCKS, stream, src, src_f32, M, C, ld, ssp, eps, partial);
}

cudaError_t launch_fp8_amax_rows(const float* rowmax, int M, int C, const float* ssp, float eps, float* partial,
                                 cudaStream_t stream) {
  if (rowmax == nullptr || partial == nullptr || M < 1 || C < 32 || C % 32 != 0 ||
      (ssp != nullptr && C % SS_GROUP != 0))
    return cudaErrorInvalidValue;
  return launch_q(fp8_amax_rows_kernel, FP8_AMAX_BLOCKS, stream, rowmax, M, C, ssp, eps, partial);
}

cudaError_t launch_fp8_quantize(const void* src, int src_f32, int M, int C, int ld, const float* ssp, float eps,
                                const float* partial, int npart, uint8_t* dst, int ld_dst, int group, int gap,
                                float* inv_scale, cudaStream_t stream) {
  if (!q_args_ok(src, src_f32, M, C, ld, ssp) || partial == nullptr || npart < 1 || dst == nullptr ||
      inv_scale == nullptr ||
      ld_dst < C || ld_dst % 8 != 0 || reinterpret_cast<uintptr_t>(dst) % 8 != 0 || group < 0 || gap < 0)
    return cudaErrorInvalidValue;
  const int rows_per_block = QT / 32;
  int grid = (M + rows_per_block - 1) / rows_per_block;
  grid = grid < 4 * FP8_AMAX_BLOCKS ? grid : 4 * FP8_AMAX_BLOCKS;
  return launch_q(fp8_quantize_kernel, grid, stream, src, src_f32, M, C, ld, ssp, eps, partial, npart, dst, ld_dst,
                  group, gap, inv_scale);
}

}  // namespace nc
