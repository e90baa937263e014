// internal.h -- launchers shared between the kernels and the model orchestration.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "nc.h"

namespace nc {

using bf16 = __nv_bfloat16;

enum EpiKind : int {
  EPI_BF16 = 0,         // out(bf16) = acc
  EPI_RESID = 1,        // residual stream update (see GemmEpi, "residual" fields)
  EPI_RELU2_BF16 = 2,   // out(bf16) = relu(rs * acc)^2
  EPI_SOFTCAP_F32 = 3,  // out(f32) = cap * tanh(rs * acc / cap)
  EPI_QKV = 4,          // q|k|v split, RoPE + RMSNorm on q and k, value-embedding gate on v
  EPI_CE = 5,           // cross-entropy partials of z = cap * tanh(rs * acc / cap), no logits
  EPI_SOFTCAP_BF16 = 6, // out(bf16) = cap * tanh(rs * acc / cap)
  EPI_F32 = 7,          // out(f32) = rs * acc
  EPI_CE_GRAD = 8,      // out(bf16) = gradient of the mean cross-entropy at the lm_head's pre-cap output
  EPI_DRELU2 = 9,       // out(bf16) = rs * acc * 2 sqrt(h)   (the squared ReLU's derivative)
};

// Columns covered by one partial sum of squares (one epilogue thread's share of a row).
constexpr int SS_GROUP = 128;

// Rows that follow each kv head's v rows in a value-embedding layer's packed q|k|v weight: the
// head's gate row, then zero rows (the MMA's N must be a multiple of 16), so that the head's
// GEMM tile, D + VGATE_ROWS columns wide, also yields the gate's pre-activation.
constexpr int VGATE_ROWS = 16;

struct GemmEpi {
  int kind = EPI_BF16;
  int* status = nullptr;
  // Limit of every bounded wait of the launch, and a test hook: the MMA issuer withholds the
  // "accumulator ready" signal of pair tile test_skip_tile (< 0: none), so that its epilogue's
  // wait runs out and the launch takes its abort path (see nc_op_test_wait_timeout).
  unsigned long long wait_ns = 2000000000ull;
  int test_skip_tile = -1;

  // Operand layouts.  0: K contiguous, A[M][K] and B[N][K] (nn.Linear weights and activations);
  // 1: M (or N) contiguous, A stored as [K][M], B as [K][N] -- the transposed operands of the
  // backward's products (a weight gradient contracts over tokens, an input gradient multiplies
  // by the weight itself).  Both stored densely (row pitch = the contiguous extent).
  int a_mn = 0, b_mn = 0;

  // 8-bit operands: A and B e4m3 (one byte per element, K-contiguous, K % 16 == 0), the tensor
  // cores' kind::f8f6f4; the accumulator is dequantised by multiplying it by fp8_sa[0] (the input's
  // 1 / scale) times fp8_sw[j] (the weight's), j = 0 except for EPI_QKV, where the q, k and v
  // column ranges use fp8_sw[0], [1], [2].  The row scale of ssp_in does not apply (the quantised
  // input already carries its RMSNorm).
  int fp8 = 0;
  const float* fp8_sa = nullptr;
  const float* fp8_sw = nullptr;

  // Row scale of the consuming epilogues (RELU2, SOFTCAP, QKV, F32, CE_GRAD, DRELU2): rs[m] = 1 / sqrt(sum_g
  // ssp[m, g] / ncols + eps), ssp fp32 [M, ncg] partial sums of squares; ssp == null -> rs = 1.
  const float* ssp_in = nullptr;
  int ncg = 0;            // partial sums per row (ncols / SS_GROUP)
  float inv_ncols = 0.f;  // 1 / ncols
  float eps = 1e-6f;

  // EPI_BF16 / EPI_RELU2_BF16 / EPI_SOFTCAP_F32 / EPI_SOFTCAP_BF16 / EPI_F32 / EPI_CE_GRAD / EPI_DRELU2
  void* out = nullptr;
  int ldo = 0;
  float cap = 15.f;

  // 8-bit producers of the next quantisation's maximum: EPI_RESID on the 8-bit path writes
  // rowmax_out[m * (N / 32) + n / 32] = max |x'| over columns [n, n + 32) when set; EPI_RELU2_BF16
  // on the 8-bit path raises *amax_out (fp32 bits compared as unsigned: the values are >= 0) to the
  // largest h it stores (after its bf16 rounding) when set.  Both are exact maxima, the same
  // numbers a pass over the stored tensor would find.
  float* rowmax_out = nullptr;
  float* amax_out = nullptr;

  // EPI_RESID (launch_gemm_resid; N = ncols of the stream, N % 128 == 0):
  //   xr = resid + acc;  xm_out <- xr (if set);  x' = a * xr + b * Y (Y may be null);
  //   x_out <- x' (if set, may alias resid);  xb <- bf16(x');
  //   ssp_out[m, g] = sum of x'^2 over columns [128 g, 128 g + 128).
  const float* resid = nullptr;
  float a = 1.f, b = 0.f;
  const float* Y = nullptr;
  float* x_out = nullptr;
  float* xm_out = nullptr;
  bf16* xb = nullptr;
  float* ssp_out = nullptr;

  // EPI_QKV
  bf16* q = nullptr;
  bf16* k = nullptr;
  bf16* v = nullptr;
  int H = 0, Hkv = 0, D = 0, T = 1;
  int rope_ld = 0;                // row length (positions) of the rotary table
  const float2* rope = nullptr;   // [D/2][rope_ld] (cos, sin), position fastest
  // vgate != 0 (a value-embedding layer): B holds the q and k rows, then for each kv head its D v
  // rows followed by its gate row and VGATE_ROWS - 1 zero rows; v += gate * ve[token] with
  // gate = gate_scale * sigmoid(rs * (x . gate row)).
  int vgate = 0;
  float gate_scale = 1.f;
  // With gpre set, a value-embedding head's gate pre-activation is read from gpre[m * gpre_ld + g]
  // (already scaled by the row's RMSNorm) instead of the tile's gate column: the 8-bit path keeps
  // the gate's dot product in bf16 (its packed gate rows are zero).
  const float* gpre = nullptr;
  int gpre_ld = 0;
  const bf16* ve = nullptr;       // [V, Hkv*D]
  const int32_t* tokens = nullptr;
  int V = 0;

  // EPI_CE (uses ssp_in / cap): for each row m and 128-column group g (g = col / 128),
  //   ce_part[g * M + m] = sum over the group's columns of exp(z[m, col])   (group-major);
  //   ce_zt[m] = z[m, targets[m]], written by the group holding the target column (rows whose
  //   target lies outside [0, N) are not written).
  const int32_t* targets = nullptr;
  float* ce_part = nullptr;
  float* ce_zt = nullptr;

  // EPI_CE_GRAD (uses ssp_in / cap / targets): with z = cap * tanh(u / cap), u = rs * acc,
  //   out[m, n] = rs * inv_count * (exp(z - ce_lse[m]) - [n == targets[m]]) * (1 - (z / cap)^2)
  // -- d(mean loss)/du times the row's RMSNorm scale, which the weight gradient needs -- and 0 on
  // rows whose target lies outside [0, N).  ce_lse[m] = log sum_n exp(z[m, n]); inv_count: one
  // float in device memory, 1 / (rows counted).
  const float* ce_lse = nullptr;
  const float* inv_count = nullptr;
  // EPI_DRELU2 (uses ssp_in): h_in bf16 [M, ldo] holds relu(u)^2 of the forward, so relu(u) =
  // sqrt(h) and out = rs * acc * 2 sqrt(h).
  const bf16* h_in = nullptr;

  // EPI_F32 split over K (launch_gemm sets these from split_ws / gemm_ksplit): the k-blocks are cut
  // into ksplit consecutive ranges, each computed by its own tiles into the fp32 slab
  // split_ws + s * M * ldo, then added in the order s = 0, 1, ... into out by a second kernel, so
  // the result does not depend on which tiles ran first.
  int ksplit = 1;
  float* split_ws = nullptr;
};

// How many K ranges an EPI_F32 product of this shape is split into: enough that its tiles fill
// the CTA pairs of the device (a weight gradient has few output tiles and a long K), at least one
// 64-deep k-block per range, at most 16.  1 when the output tiles alone fill half the pairs.
int gemm_ksplit(int M, int N, int K, int num_sms);
// Bytes of split_ws such a product needs (0 when it is not split).
size_t gemm_split_ws_bytes(int M, int N, int K, int ldo, int num_sms);


// Records `e` as the calling thread's last CUDA error (read by nc_last_cuda_error) and maps it
// to a status: NC_OK for cudaSuccess, NC_ERR_CUDA otherwise.
nc_status cuda_status(cudaError_t e);
const char* last_cuda_error_name();

// One-time per-device set-up of a kernel (its shared-memory attribute, its occupancy), done with
// that device current, so that a process running models on several GPUs sets each one up.
constexpr int MAX_DEVICES = 64;

// Kernel state for the current device (states[dev]), initialised on first use on that device by
// init(State&) -> cudaError_t; a failed init is retried on the next call.
template <typename State, typename Init>
cudaError_t per_device(State (&states)[MAX_DEVICES], bool (&ready)[MAX_DEVICES], std::mutex& mu, Init init,
                       State** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev]) {
    const cudaError_t e = init(states[dev]);
    if (e != cudaSuccess) return e;
    ready[dev] = true;
  }
  *out = &states[dev];
  return cudaSuccess;
}

// Launch attribute that lets a kernel's CTAs start while the previous kernel on the stream
// drains (each kernel waits for its predecessor before touching memory: griddep_wait()).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Encodes a 2-D TMA descriptor through the driver entry point (no link-time libcuda), with
// 128-byte swizzling unless swizzle128 is false (then the box is a dense row-major array in shared
// memory).  inner/outer are extents in elements, row stride in bytes.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                  bool swizzle128 = true);

inline bool make_tmap_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, inner, outer, row_stride_bytes,
                      box_inner, box_outer);
}

// C[M, N] = epi(A[M, K] . B[N, K]^T); A, B bf16, K contiguous unless epi.a_mn / epi.b_mn.
// An EPI_F32 product with epi.split_ws set (>= gemm_split_ws_bytes) is split over K as described
// at GemmEpi::ksplit (two launches); without split_ws it runs unsplit.
// Requires N % 32 == 0, 16-byte aligned rows (K % 8 == 0 for a K-contiguous operand, M % 8 or
// N % 8 == 0 for an MN-contiguous one); K may be ragged (the last k-block is zero-filled).
cudaError_t launch_gemm(const bf16* A, const bf16* B, int M, int N, int K, const GemmEpi& epi,
                        int num_sms, cudaStream_t stream);

// Residual-stream update of an output projection (EPI_RESID fields of `epi`), computed as the
// transposed product W . A^T so that the epilogue's loads and stores of the stream are coalesced
// from registers: xr = resid + A[M, K] . W[N, K]^T, then the updates listed at GemmEpi.
// Requires K % 64 == 0, N % 128 == 0, 16-byte aligned rows of A and W.
cudaError_t launch_gemm_resid(const bf16* A, const bf16* W, int M, int N, int K, const GemmEpi& epi,
                              int num_sms, cudaStream_t stream);

// x0 = smear(wte[tokens]); x = a * x0; xb = bf16(x); ssp[m, g] = sum of x^2 over column group g.
cudaError_t launch_embed_smear(const int32_t* tokens, int B, int T, const bf16* wte, int V, int C,
                               const bf16* smear_gate, int c_s, int embed_norm, float eps, float a,
                               float* x0, float* x, bf16* xb, float* ssp, int* status, cudaStream_t stream);

// table[i][t] = (cos, sin)(t * base^(-2i/D)), i < D/2, t < T (position fastest).
cudaError_t launch_rope_table(float2* table, int T, int D, float base, cudaStream_t stream);

// Cross-entropy from the EPI_CE partials: per row S = sum_g part[g * M + m] over G groups;
// loss[m] = log S - zt[m] for targets in [0, V), 0 for ignored rows (target < 0; other targets
// outside [0, V) record NC_ERR_TOKEN_RANGE and are ignored).  stats[0] = mean loss over the
// counted rows, stats[1] = bits per byte (sum of the losses of rows whose target has a nonzero
// byte count, over ln 2 times the sum of those byte counts; NaN without token_bytes or bytes).
// scratch holds ce_scratch_doubles(M) doubles.  loss may be null.
// lse (optional) receives log S per counted row (0 on ignored rows) and inv_count (optional, one
// float) 1 / (rows counted), 0 when none is counted: the inputs of EPI_CE_GRAD.
int ce_scratch_doubles(int M);
cudaError_t launch_ce_finalize(const float* part, const float* zt, const int32_t* targets, int M, int G, int V,
                               const int32_t* token_bytes, float* loss, float* stats, double* scratch,
                               int* status, cudaStream_t stream, float* lse = nullptr,
                               float* inv_count = nullptr);

// ---- 8-bit (e4m3) tensorwise quantisation: q = e4m3(v * s), s = 448 / max|v| over the whole tensor
// (1 when it is all zero), round to nearest even, saturating at +-448.  v = src[m, c], times the
// row's RMSNorm scale rs[m] = 1 / sqrt(sum_g ssp[m, g] / C + eps) when ssp is given.  Two launches:
// fp8_amax writes per-block maxima to partial[FP8_AMAX_BLOCKS]; fp8_quantize reduces partial[0 ..
// npart) in every block, writes q [M, ld_dst] and inv_scale[0] = 1 / s.  Rows of src are `ld`
// elements apart; dst row r goes to r + (r / group) * gap (group = 0: no remap), for the packed
// q|k|v weight's v heads.  fp8_amax_rows computes the same per-block maxima of a row-scaled stream
// from its producer's per-row maxima of |v| over 32-column groups (rowmax [M][C/32], written by
// the residual GEMM's epilogue), without reading the stream: max over rows of rs[m] * max|v[m, :]|
// is the same number either way (multiplication by rs > 0 keeps the order of rounded products).
constexpr int FP8_AMAX_BLOCKS = 592;
cudaError_t launch_fp8_amax(const void* src, int src_f32, int M, int C, int ld, const float* ssp, float eps,
                            float* partial, cudaStream_t stream);
cudaError_t launch_fp8_amax_rows(const float* rowmax, int M, int C, const float* ssp, float eps, float* partial,
                                 cudaStream_t stream);
cudaError_t launch_fp8_quantize(const void* src, int src_f32, int M, int C, int ld, const float* ssp, float eps,
                                const float* partial, int npart, uint8_t* dst, int ld_dst, int group, int gap,
                                float* inv_scale, cudaStream_t stream);

// Backward of the weightless RMSNorm xn = rs * x (rs = 1 / sqrt(mean x^2 + eps), from the partial
// sums ssp [M, C / 128]) given G = rs * dL/dxn:  dx = G - rs^2 * x * mean(G * x)  (+ add, if set).
// dx goes to dx_f32 (if set) and as bf16 to dx_b16 (if set); rows of C fp32 elements, C % 128 == 0.
cudaError_t launch_rms_backward(const float* G, const float* x, const float* ssp, const float* add, int M, int C,
                                float eps, float* dx_f32, bf16* dx_b16, cudaStream_t stream);

// y[M, H*D] = windowed causal GQA attention of q [M, H*D], k/v [M, Hkv*D].
cudaError_t launch_attention(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H,
                             int Hkv, int D, int window, bf16* y, int* status, cudaStream_t stream);

}  // namespace nc
