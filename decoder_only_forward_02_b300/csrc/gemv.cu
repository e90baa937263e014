// gemv.cu -- the products of a decode step: a few rows (one new token per batch row) times every
// weight matrix of the model, for sm_103a.
//
// "nanochat — 架构与原理", section 2 component table (the inference engine: KV cache, one token per
// step).  A decode step multiplies B rows by each weight once: B x K by K x N with B a handful,
// so the step reads every weight from HBM and does 2B flops per weight element -- a weight
// stream, not a contraction the tensor cores' tile machinery pays off on (a 256-row tcgen05 tile
// at 16 rows spends its launch on cluster set-up, tensor-memory allocation and the first operand
// round trip, and a few pair tiles cannot pull a weight from HBM fast enough).
//
// Work split: CTA (j, i) owns the weight rows [8j, 8j + 8) and the tokens [16i, 16i + 16); its
// warps split K.  A warp accumulates D[16 tokens][8 rows] in fp32 with mma.sync m16n8k16 (bf16
// operands): the tokens are the instruction's M side, the weight rows its N side.  Per 32-deep k
// step each lane loads 16 contiguous bytes of its weight row (four lanes cover 64 B of a row, a
// warp 8 rows) and 16 of each of its two token rows; the step's two instructions consume those
// bytes in the same permutation of k for both operands, which leaves the sum over k unchanged.
// The weight loads are issued before the kernel waits for its predecessor (the weights never
// change), so with programmatic dependent launch their latency overlaps the previous kernel.
// The warps' partial products are added in a fixed order (deterministic results), then one
// warp applies the epilogue to the CTA's 16 x 8 outputs:
//   GEMV_RAW          out_f32 = rs * acc                          (q|k|v before RoPE / norms)
//   GEMV_RESID        xr = x + acc; xm <- xr; x' = a xr + b Y; x <- x'; xb <- bf16(x');
//                     ssp_out[token][j] = sum of x'^2 over the CTA's 8 columns
//   GEMV_RELU2        h = bf16(relu(rs * acc)^2)                  (MLP up projection)
//   GEMV_SOFTCAP_F32  z = cap tanh(rs * acc / cap), fp32 or bf16  (lm_head)
// rs is the input's RMSNorm row scale, 1 / sqrt(sum of the row's partial sums of squares / ncols
// + eps), from the partials its producer wrote (the same formula as the full forward).
//
// Why mma.sync: the kernel is bound by the weight stream and the launch chain, not by arithmetic
// (2B flops per weight byte pair).  The warp-level instruction is used as a register-to-register
// dot-product unit: one instruction does 16 x 8 x 16 multiply-adds straight from the bf16 bytes
// the coalesced loads delivered, where CUDA cores would first convert every weight and token
// element to fp32 (a CUDA-core variant that did so was 2x slower per step).  tcgen05 would need
// the operands in shared memory, a tensor-memory allocation and at least 64 rows per CTA, all
// latency on a path whose every launch is on the critical chain.
#include "decode.h"
#include "ptx.cuh"

#include <algorithm>

namespace nc {
namespace {

constexpr int GV_ROWS = 8;    // weight rows per CTA (the MMA's N)
constexpr int GV_TOK = 16;    // tokens per CTA (the MMA's M)
constexpr int GV_SMAX = 6;    // 32-deep k steps a warp holds in registers at a time
constexpr int GV_RSP = 16;    // row-scale partials a thread loads at a time (8 threads per token)
constexpr int GV_MAXW = 16;   // warps per CTA at most

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg16(const bf16* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

template <int KIND>
__global__ void __launch_bounds__(32 * GV_MAXW)
    gemv_kernel(const bf16* __restrict__ A, int lda, int B, const bf16* __restrict__ W, int N, int K, int steps,
                const __grid_constant__ GemvEpi ep) {
  __shared__ float red[GV_MAXW - 1][32][4];
  __shared__ float rs_s[GV_TOK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.x * GV_ROWS, b0 = blockIdx.y * GV_TOK;
  const int ksteps = K / 32;
  const int s0 = warp * steps, s1 = min(ksteps, s0 + steps);   // this warp's k steps [s0, s1)
  // The lane's weight row n0 + g (N % 8 == 0: always a row of W), 16 B per step at k 32 s + 8 t.
  const bf16* wr = W + static_cast<size_t>(n0 + g) * K + 8 * t;
  uint4 w[GV_SMAX];
#pragma unroll
  for (int s = 0; s < GV_SMAX; ++s) w[s] = s0 + s < s1 ? ldg16(wr + (s0 + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
  griddep_wait();   // the activations and the row partials come from the preceding kernel
  griddep_launch();
  // The row scales' partial sums: threads 0..127, eight per token (token tid / 8 reads partials
  // tid % 8 + 8 j), loaded now and added up after the products (a fixed order).
  const int rt = threadIdx.x >> 3, rp = threadIdx.x & 7;
  const bool rsl = ep.ssp != nullptr && threadIdx.x < 8 * GV_TOK && b0 + rt < B;
  const float* rsp = rsl ? ep.ssp + static_cast<size_t>(b0 + rt) * ep.ssp_ld : nullptr;
  float pv[GV_RSP];
#pragma unroll
  for (int j = 0; j < GV_RSP; ++j) pv[j] = rsl && rp + 8 * j < ep.ssp_n ? rsp[rp + 8 * j] : 0.f;
  // The residual epilogue's inputs (warp 0 applies the epilogue), loaded before the products.
  const int n = n0 + 2 * t;
  float2 xres[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 yres[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if constexpr (KIND == GEMV_RESID) {
    if (warp == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = b0 + g + 8 * h;
        if (b < B) {
          const size_t o = static_cast<size_t>(b) * ep.ldx + n;
          xres[h] = *reinterpret_cast<const float2*>(ep.resid + o);
          if (ep.Y != nullptr) yres[h] = *reinterpret_cast<const float2*>(ep.Y + o);
        }
      }
    }
  }
  // The two token rows of the lane: b0 + g (the fragment's rows g) and b0 + g + 8 (rows g + 8).
  const bool va = b0 + g < B, vb = b0 + g + 8 < B;
  const bf16* ar = A + static_cast<size_t>(va ? b0 + g : 0) * lda + 8 * t;
  const bf16* br = A + static_cast<size_t>(vb ? b0 + g + 8 : 0) * lda + 8 * t;
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = s0; c < s1; c += GV_SMAX) {
    if (c != s0) {   // K beyond what the registers hold at once: the next chunk of weight steps
#pragma unroll
      for (int s = 0; s < GV_SMAX; ++s) w[s] = c + s < s1 ? ldg16(wr + (c + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint4 xa[GV_SMAX], xb[GV_SMAX];   // every token load of the chunk in flight at once
#pragma unroll
    for (int s = 0; s < GV_SMAX; ++s) {
      xa[s] = va && c + s < s1 ? ldg16(ar + (c + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
      xb[s] = vb && c + s < s1 ? ldg16(br + (c + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int s = 0; s < GV_SMAX; ++s) {
      if (c + s < s1) {   // uniform across the warp
        // k pairs (2t, 2t+1) and (2t+8, 2t+9) of the first instruction are the lane's bytes 0-3
        // and 4-7, of the second bytes 8-11 and 12-15, for the weight and the tokens alike
        mma_16816(d, xa[s].x, xb[s].x, xa[s].y, xb[s].y, w[s].x, w[s].y);
        mma_16816(d, xa[s].z, xb[s].z, xa[s].w, xb[s].w, w[s].z, w[s].w);
      }
    }
  }
  if (threadIdx.x < 8 * GV_TOK) {   // the row scales (warps 0..3: every CTA has at least four)
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < GV_RSP; ++j) ss += pv[j];
    for (int i0 = 8 * GV_RSP; i0 < ep.ssp_n; i0 += 8 * GV_RSP) {   // rows with more partials
#pragma unroll
      for (int j = 0; j < GV_RSP; ++j) pv[j] = rsl && i0 + rp + 8 * j < ep.ssp_n ? rsp[i0 + rp + 8 * j] : 0.f;
#pragma unroll
      for (int j = 0; j < GV_RSP; ++j) ss += pv[j];
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    if (rp == 0) rs_s[rt] = ep.ssp != nullptr ? rsqrtf(ss * ep.inv_ncols + ep.eps) : 1.f;
  }
  if (warp > 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp - 1][lane][i] = d[i];
  }
  __syncthreads();
  if (warp != 0) return;
  for (int w2 = 1; w2 < nw; ++w2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] += red[w2 - 1][lane][i];
  }
  // d[2h], d[2h+1]: token b0 + g + 8h, columns n, n + 1
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = b0 + g + 8 * h;
    const bool ok = b < B;
    const float rs = rs_s[g + 8 * h];
    const float v0 = d[2 * h], v1 = d[2 * h + 1];
    if constexpr (KIND == GEMV_RAW) {
      if (ok)
        *reinterpret_cast<float2*>(static_cast<float*>(ep.out) + static_cast<size_t>(b) * ep.ldo + n) =
            make_float2(v0 * rs, v1 * rs);
    } else if constexpr (KIND == GEMV_RELU2) {
      if (ok) {
        const float r0 = fmaxf(v0 * rs, 0.f), r1 = fmaxf(v1 * rs, 0.f);
        *reinterpret_cast<uint32_t*>(static_cast<bf16*>(ep.out) + static_cast<size_t>(b) * ep.ldo + n) =
            pack_bf16(r0 * r0, r1 * r1);
      }
    } else if constexpr (KIND == GEMV_SOFTCAP_F32 || KIND == GEMV_SOFTCAP_BF16) {
      if (ok) {
        const float sc = rs / ep.cap;
        const float z0 = ep.cap * tanh_approx(v0 * sc), z1 = ep.cap * tanh_approx(v1 * sc);
        if constexpr (KIND == GEMV_SOFTCAP_F32)
          __stcs(reinterpret_cast<float2*>(static_cast<float*>(ep.out) + static_cast<size_t>(b) * ep.ldo + n),
                 make_float2(z0, z1));
        else
          *reinterpret_cast<uint32_t*>(static_cast<bf16*>(ep.out) + static_cast<size_t>(b) * ep.ldo + n) =
              pack_bf16(z0, z1);
      }
    } else {   // GEMV_RESID
      float sq = 0.f;
      if (ok) {
        const size_t o = static_cast<size_t>(b) * ep.ldx + n;
        const float2 xv = xres[h];
        const float xr0 = v0 + xv.x, xr1 = v1 + xv.y;
        float x0, x1;
        if (ep.Y != nullptr) {
          const float2 yv = yres[h];
          x0 = fmaf(ep.a, xr0, ep.b * yv.x);
          x1 = fmaf(ep.a, xr1, ep.b * yv.y);
        } else {
          x0 = ep.a * xr0;
          x1 = ep.a * xr1;
        }
        if (ep.xm_out != nullptr) *reinterpret_cast<float2*>(ep.xm_out + o) = make_float2(xr0, xr1);
        if (ep.x_out != nullptr) *reinterpret_cast<float2*>(ep.x_out + o) = make_float2(x0, x1);
        *reinterpret_cast<uint32_t*>(ep.xb + static_cast<size_t>(b) * ep.ldb + n) = pack_bf16(x0, x1);
        sq = x0 * x0 + x1 * x1;
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);   // the token's 8 columns
      if (ok && t == 0) ep.ssp_out[static_cast<size_t>(b) * ep.ssp_out_ld + blockIdx.x] = sq;
    }
  }
}

// The lm_head of a decode step: far more 8-row blocks than the SMs hold at once.  Persistent
// CTAs take the row blocks rb = blockIdx.x + i * gridDim.x; the token rows are loaded once, and
// the next block's weight bytes are in flight while the current block's products and epilogue
// run.  Each warp's k steps fit in one register chunk (steps <= GV_SMAX).  Soft-capped logits.
template <int KIND>
__global__ void __launch_bounds__(32 * GV_MAXW)
    gemv_rows_kernel(const bf16* __restrict__ A, int lda, int B, const bf16* __restrict__ W, int N, int K,
                     int steps, const __grid_constant__ GemvEpi ep) {
  __shared__ float red[GV_MAXW - 1][32][4];
  __shared__ float rs_s[GV_TOK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int b0 = blockIdx.y * GV_TOK;
  const int ksteps = K / 32;
  const int s0 = warp * steps, s1 = min(ksteps, s0 + steps);
  const int nrb = N / GV_ROWS;
  int rb = blockIdx.x;
  uint4 w[GV_SMAX];
  {
    const bf16* wr = W + static_cast<size_t>(rb * GV_ROWS + g) * K + 8 * t;
#pragma unroll
    for (int s = 0; s < GV_SMAX; ++s)
      w[s] = rb < nrb && s0 + s < s1 ? ldg16(wr + (s0 + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
  }
  griddep_wait();   // the final stream's bf16 copy and its partial sums come from the preceding kernel
  griddep_launch();
  const int rt = threadIdx.x >> 3, rp = threadIdx.x & 7;
  const bool rsl = ep.ssp != nullptr && threadIdx.x < 8 * GV_TOK && b0 + rt < B;
  const float* rsp = rsl ? ep.ssp + static_cast<size_t>(b0 + rt) * ep.ssp_ld : nullptr;
  const bool va = b0 + g < B, vb = b0 + g + 8 < B;
  const bf16* ar = A + static_cast<size_t>(va ? b0 + g : 0) * lda + 8 * t;
  const bf16* br = A + static_cast<size_t>(vb ? b0 + g + 8 : 0) * lda + 8 * t;
  uint4 xa[GV_SMAX], xb[GV_SMAX];   // the token rows: loaded once for every row block
#pragma unroll
  for (int s = 0; s < GV_SMAX; ++s) {
    xa[s] = va && s0 + s < s1 ? ldg16(ar + (s0 + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
    xb[s] = vb && s0 + s < s1 ? ldg16(br + (s0 + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x < 8 * GV_TOK) {   // the row scales, as in gemv_kernel (rows of any length)
    float ss = 0.f;
    for (int i0 = 0; i0 < ep.ssp_n; i0 += 8 * GV_RSP) {
      float pv[GV_RSP];
#pragma unroll
      for (int j = 0; j < GV_RSP; ++j) pv[j] = rsl && i0 + rp + 8 * j < ep.ssp_n ? rsp[i0 + rp + 8 * j] : 0.f;
#pragma unroll
      for (int j = 0; j < GV_RSP; ++j) ss += pv[j];
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    if (rp == 0) rs_s[rt] = ep.ssp != nullptr ? rsqrtf(ss * ep.inv_ncols + ep.eps) : 1.f;
  }
  for (; rb < nrb; rb += gridDim.x) {   // uniform across the CTA
    const int nx = rb + gridDim.x;
    uint4 wn[GV_SMAX];   // the next block's weight bytes, in flight during this block
    {
      const bf16* wr = W + static_cast<size_t>((nx < nrb ? nx : rb) * GV_ROWS + g) * K + 8 * t;
#pragma unroll
      for (int s = 0; s < GV_SMAX; ++s)
        wn[s] = nx < nrb && s0 + s < s1 ? ldg16(wr + (s0 + s) * 32) : make_uint4(0u, 0u, 0u, 0u);
    }
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < GV_SMAX; ++s) {
      if (s0 + s < s1) {
        mma_16816(d, xa[s].x, xb[s].x, xa[s].y, xb[s].y, w[s].x, w[s].y);
        mma_16816(d, xa[s].z, xb[s].z, xa[s].w, xb[s].w, w[s].z, w[s].w);
      }
    }
    if (warp > 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) red[warp - 1][lane][i] = d[i];
    }
    __syncthreads();
    if (warp == 0) {
      for (int w2 = 1; w2 < nw; ++w2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += red[w2 - 1][lane][i];
      }
      const int n = rb * GV_ROWS + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = b0 + g + 8 * h;
        if (b < B) {
          const float sc = rs_s[g + 8 * h] / ep.cap;
          const float z0 = ep.cap * tanh_approx(d[2 * h] * sc), z1 = ep.cap * tanh_approx(d[2 * h + 1] * sc);
          if constexpr (KIND == GEMV_SOFTCAP_F32)
            __stcs(reinterpret_cast<float2*>(static_cast<float*>(ep.out) + static_cast<size_t>(b) * ep.ldo + n),
                   make_float2(z0, z1));
          else
            *reinterpret_cast<uint32_t*>(static_cast<bf16*>(ep.out) + static_cast<size_t>(b) * ep.ldo + n) =
                pack_bf16(z0, z1);
        }
      }
    }
    __syncthreads();   // red is refilled by the next block
#pragma unroll
    for (int s = 0; s < GV_SMAX; ++s) w[s] = wn[s];
  }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl2(Kern kernel, dim3 grid, int threads, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

bool al(const void* p, int bytes) { return reinterpret_cast<uintptr_t>(p) % bytes == 0; }

}  // namespace

cudaError_t launch_gemv(const bf16* A, int lda, int B, const bf16* W, int N, int K, const GemvEpi& ep,
                        cudaStream_t stream) {
  if (A == nullptr || W == nullptr || B < 1 || N < 8 || N % 8 != 0 || K < 32 || K % 32 != 0 || lda < K ||
      lda % 8 != 0 || !al(A, 16) || !al(W, 16) || (ep.ssp != nullptr && (ep.ssp_n < 1 || ep.ssp_ld < ep.ssp_n)))
    return cudaErrorInvalidValue;
  switch (ep.kind) {
    case GEMV_RAW:
    case GEMV_SOFTCAP_F32:
      if (ep.out == nullptr || !al(ep.out, 8) || ep.ldo < N || ep.ldo % 2 != 0) return cudaErrorInvalidValue;
      break;
    case GEMV_RELU2:
    case GEMV_SOFTCAP_BF16:
      if (ep.out == nullptr || !al(ep.out, 4) || ep.ldo < N || ep.ldo % 2 != 0) return cudaErrorInvalidValue;
      break;
    case GEMV_RESID:
      if (ep.resid == nullptr || ep.xb == nullptr || ep.ssp_out == nullptr || ep.ldx < N || ep.ldx % 2 != 0 ||
          ep.ldb < N || ep.ldb % 2 != 0 || ep.ssp_out_ld < N / GV_ROWS || !al(ep.resid, 8) || !al(ep.xb, 4) ||
          (ep.Y != nullptr && !al(ep.Y, 8)) || (ep.x_out != nullptr && !al(ep.x_out, 8)) ||
          (ep.xm_out != nullptr && !al(ep.xm_out, 8)))
        return cudaErrorInvalidValue;
      break;
    default: return cudaErrorInvalidValue;
  }
  const int ksteps = K / 32;
  const int nw = std::min(GV_MAXW, std::max(1, (ksteps + GV_SMAX - 1) / GV_SMAX));   // beyond 16 x 6: chunks
  // at least 4 warps: more loads in flight per CTA, and the row-scale sums use threads 0..127
  const int warps = std::min(GV_MAXW, std::max(4, nw));
  const int steps = (ksteps + warps - 1) / warps;
  const dim3 grid(N / GV_ROWS, (B + GV_TOK - 1) / GV_TOK);
  if ((ep.kind == GEMV_SOFTCAP_F32 || ep.kind == GEMV_SOFTCAP_BF16) && steps <= GV_SMAX) {
    // the lm_head: persistent CTAs, four per SM, when there are more row blocks than that
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorInvalidValue;
    const int ctas = 4 * sms;
    if (static_cast<int>(grid.x) > ctas) {
      const dim3 pgrid(ctas, grid.y);
      if (ep.kind == GEMV_SOFTCAP_F32)
        return launch_pdl2(gemv_rows_kernel<GEMV_SOFTCAP_F32>, pgrid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
      return launch_pdl2(gemv_rows_kernel<GEMV_SOFTCAP_BF16>, pgrid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
    }
  }
  switch (ep.kind) {
    case GEMV_RAW: return launch_pdl2(gemv_kernel<GEMV_RAW>, grid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
    case GEMV_RESID:
      return launch_pdl2(gemv_kernel<GEMV_RESID>, grid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
    case GEMV_RELU2:
      return launch_pdl2(gemv_kernel<GEMV_RELU2>, grid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
    case GEMV_SOFTCAP_F32:
      return launch_pdl2(gemv_kernel<GEMV_SOFTCAP_F32>, grid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
    default:
      return launch_pdl2(gemv_kernel<GEMV_SOFTCAP_BF16>, grid, 32 * warps, stream, A, lda, B, W, N, K, steps, ep);
  }
}

}  // namespace nc
