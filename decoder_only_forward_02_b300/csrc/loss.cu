// loss.cu -- next-token cross-entropy from the partials of the fused lm_head (EPI_CE).
//
// "nanochat — 架构与原理", section 2 component table (the metrics row: bits per byte from the
// loss evaluation) and "NanoChat基础训练报告", section on the loss progression (training loss
// and validation bpb): the loss is the cross-entropy of the soft-capped logits against the
// next token, in nats; bits per byte divides the summed loss by ln 2 times the summed byte
// lengths of the target tokens (tokens of zero byte length, the special tokens, are left out).
//
//   ce_rows   one thread per row: S = sum over the G partial sums (group-major, so a warp
//             reads 32 consecutive rows of one group), loss = log S - z[target]; per block,
//             the sums needed by the statistics, reduced in a fixed order.
//   ce_stats  one block: the per-block sums, in a fixed order -> mean loss and bits per byte
//             (and 1 / rows counted, for the gradient pass).
// Both reductions run in fp64 and in a fixed order, so the statistics are bitwise repeatable.
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace nc {
namespace {

constexpr int CE_THREADS = 256;
constexpr int NSTAT = 4;   // per block: sum loss, rows counted, sum loss with bytes, sum bytes

// Fixed-order block sum of NSTAT doubles; the result is valid in thread 0.
__device__ __forceinline__ void block_sum(double (&v)[NSTAT], double (*sh)[CE_THREADS / 32]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < NSTAT; ++i)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_down_sync(0xffffffffu, v[i], o);
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < NSTAT; ++i) sh[i][warp] = v[i];
  __syncthreads();
  if (threadIdx.x == 0)
#pragma unroll
    for (int i = 0; i < NSTAT; ++i) {
      double t = 0.0;
      for (int w = 0; w < CE_THREADS / 32; ++w) t += sh[i][w];
      v[i] = t;
    }
}

__global__ void __launch_bounds__(CE_THREADS)
    ce_rows_kernel(const float* __restrict__ part, const float* __restrict__ zt, const int32_t* __restrict__ targets,
                   int M, int G, int V, const int32_t* __restrict__ token_bytes, float* __restrict__ loss,
                   double* __restrict__ block_stats, int* status, float* __restrict__ lse) {
  __shared__ double sh[NSTAT][CE_THREADS / 32];
  griddep_wait();   // the lm_head's partials are complete and visible
  griddep_launch();
  const int m = blockIdx.x * CE_THREADS + threadIdx.x;
  double v[NSTAT] = {0.0, 0.0, 0.0, 0.0};
  if (m < M) {
    const int t = targets[m];
    float l = 0.f, ls = 0.f;
    if (t >= 0 && t < V) {
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      int g = 0;
      for (; g + 4 <= G; g += 4)
#pragma unroll
        for (int u = 0; u < 4; ++u) s[u] += part[static_cast<size_t>(g + u) * M + m];
      for (; g < G; ++g) s[0] += part[static_cast<size_t>(g) * M + m];
      ls = logf((s[0] + s[1]) + (s[2] + s[3]));
      l = ls - zt[m];
      v[0] = l;
      v[1] = 1.0;
      if (token_bytes != nullptr) {
        const int nb = token_bytes[t];
        if (nb > 0) {
          v[2] = l;
          v[3] = nb;
        }
      }
    } else if (t >= V) {
      record_error(status, NC_ERR_TOKEN_RANGE);   // ignored like a negative target
    }
    if (loss != nullptr) loss[m] = l;
    if (lse != nullptr) lse[m] = ls;
  }
  block_sum(v, sh);
  if (threadIdx.x == 0)
#pragma unroll
    for (int i = 0; i < NSTAT; ++i) block_stats[static_cast<size_t>(blockIdx.x) * NSTAT + i] = v[i];
}

__global__ void __launch_bounds__(CE_THREADS)
    ce_stats_kernel(const double* __restrict__ block_stats, int nblocks, float* __restrict__ stats,
                    float* __restrict__ inv_count) {
  __shared__ double sh[NSTAT][CE_THREADS / 32];
  griddep_wait();
  griddep_launch();
  double v[NSTAT] = {0.0, 0.0, 0.0, 0.0};
  for (int b = threadIdx.x; b < nblocks; b += CE_THREADS)
#pragma unroll
    for (int i = 0; i < NSTAT; ++i) v[i] += block_stats[static_cast<size_t>(b) * NSTAT + i];
  block_sum(v, sh);
  if (threadIdx.x == 0) {
    stats[0] = v[1] > 0.0 ? static_cast<float>(v[0] / v[1]) : NAN;
    stats[1] = v[3] > 0.0 ? static_cast<float>(v[2] / (0.69314718055994530942 * v[3])) : NAN;
    if (inv_count != nullptr) *inv_count = v[1] > 0.0 ? static_cast<float>(1.0 / v[1]) : 0.f;
  }
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, int grid, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(CE_THREADS);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace

int ce_scratch_doubles(int M) { return NSTAT * ((M + CE_THREADS - 1) / CE_THREADS); }

cudaError_t launch_ce_finalize(const float* part, const float* zt, const int32_t* targets, int M, int G, int V,
                               const int32_t* token_bytes, float* loss, float* stats, double* scratch,
                               int* status, cudaStream_t stream, float* lse, float* inv_count) {
  if (part == nullptr || zt == nullptr || targets == nullptr || stats == nullptr || scratch == nullptr || M < 1 ||
      G < 1 || V < 1)
    return cudaErrorInvalidValue;
  const int nblocks = (M + CE_THREADS - 1) / CE_THREADS;
  cudaError_t e = launch_pdl(ce_rows_kernel, nblocks, stream, part, zt, targets, M, G, V, token_bytes, loss,
                             scratch, status, lse);
  if (e != cudaSuccess) return e;
  return launch_pdl(ce_stats_kernel, 1, stream, static_cast<const double*>(scratch), nblocks, stats, inv_count);
}

}  // namespace nc
