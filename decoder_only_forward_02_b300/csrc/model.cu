// model.cu -- the C ABI declared in include/nc.h: validation, weight packing, workspace
// layout and the per-layer launch sequence of the forward pass.
//
// Launch sequence for one forward ("Nanochat在nanoGPT之上的新增功能", section 1 table and
// notes; each block is pre-norm attention, then pre-norm MLP).  RMSNorm has no weight, so each
// norm is split: the kernel that writes the residual stream also writes its bf16 copy and
// per-row partial sums of squares, and the GEMM that consumes it scales its accumulator rows
// by 1 / rms.
//   embed: x0 = smear(wte[tok]); x = (lr_0 + l0_0) x0 (+ bf16 copy, partial sums)
//   per layer i:
//     QKV GEMM  (row scale, RoPE, QK-norm; on VE layers the gate rows packed after each kv head's
//               v rows give the gate, and v += gate * ve)
//     attention
//     out-proj GEMM: x += y Wo^T (+ bf16 copy, partial sums)
//     fc GEMM   (row scale, ReLU^2)
//     proj GEMM: x += h Wproj^T; after layer L/2-1 that result is also the backout cache;
//                then x = lr_{i+1} x + l0_{i+1} x0 for the next block, or after the last layer
//                x - lb * x_mid (final norm's input)
//   lm_head GEMM (row scale, soft-cap)
#include "decode.h"
#include "internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

namespace nc {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
}  // namespace

nc_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NC_OK;
  g_last_cuda_error = e;
  return NC_ERR_CUDA;
}

const char* last_cuda_error_name() { return cudaGetErrorName(g_last_cuda_error); }

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                  bool swizzle128) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace nc

using nc::bf16;

namespace {

constexpr size_t ALIGN = 256;
inline size_t align_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct TimedLaunch {
  int cls;
  cudaEvent_t a, b;
};

struct Layout {
  size_t x0, x, xm, xb, q, k, v, y, h, ssp;
  // 8-bit path only (zero-sized otherwise): quantised activations (the normed stream, the
  // attention output, the MLP hidden layer), the bf16 gate pre-activations [M, 32], the amax
  // scratch and the 1 / scale of each quantised activation
  size_t a8, y8, h8, gpre, qpart, qscale, rowmax, hmax;
  size_t end;
};

// Where the last block's MLP down projection writes the lm_head's input when the backward runs:
// its own buffers, so that the last block's MLP input (x, xb, ssp) survives the forward.
struct TailOut {
  float* xf;     // fp32 [M, C] x after the final backout (the final RMSNorm's input)
  nc::bf16* xbf; // its bf16 copy (the lm_head's operand)
  float* sspf;   // its partial sums of squares
};

using nc::VGATE_ROWS;

}  // namespace

struct nc_model {
  nc_config cfg{};
  std::vector<int> window;
  std::vector<unsigned char> has_ve;
  std::vector<float> lr, l0;
  float lb = 0.f;
  const bf16* wte = nullptr;
  const bf16* smear = nullptr;
  const bf16* lm = nullptr;
  std::vector<const bf16*> wo, wfc, wproj, ve;
  bf16* wqkv = nullptr;     // packed per layer: [q rows | k rows | v rows (+ gate rows on VE layers)][C]
  std::vector<size_t> qkv_off;   // element offset of each layer's packed weight
  // 8-bit weights (fp8 configs): e4m3 q|k|v at the same element offsets as wqkv, per-layer
  // W_o, W_fc, W_proj and W_lm; bf16 gate matrices [GATE_PAD][C] per layer; 1 / scale per weight
  uint8_t* wqkv8 = nullptr;
  uint8_t* wo8 = nullptr;
  uint8_t* wfc8 = nullptr;
  uint8_t* wproj8 = nullptr;
  uint8_t* lm8 = nullptr;
  bf16* wg = nullptr;
  float* wscale = nullptr;
  float2* rope = nullptr;   // [D/2][seq_len_ctx] (cos, sin), position fastest
  int* status = nullptr;    // device status word
  int device = 0;           // the device current at creation (where packed_buf lives)
  int num_sms = 148;
  bool timing = false;
  std::vector<TimedLaunch> pending;
  std::vector<cudaEvent_t> free_events;
  double acc_ms[NC_K_COUNT] = {};
  int acc_n[NC_K_COUNT] = {};

  int C() const { return cfg.n_embd; }
  // rows of layer i's packed q|k|v weight
  int Nqkv(int i) const {
    return (cfg.n_head + 2 * cfg.n_kv_head) * cfg.head_dim + (has_ve[i] ? cfg.n_kv_head * VGATE_ROWS : 0);
  }
};

namespace {

nc_status validate_config(const nc_config* c) {
  if (c == nullptr) return NC_ERR_INVALID_ARG;
  if (c->n_layer < 1 || c->n_embd < 1 || c->n_head < 1 || c->n_kv_head < 1 || c->head_dim < 1 ||
      c->mlp_hidden < 1 || c->vocab_size < 1 || c->seq_len_ctx < 1)
    return NC_ERR_INVALID_ARG;
  if (c->window_left == nullptr || c->has_ve == nullptr) return NC_ERR_INVALID_ARG;
  if (c->n_embd != c->n_head * c->head_dim) return NC_ERR_INVALID_ARG;
  if (c->n_head % c->n_kv_head != 0) return NC_ERR_INVALID_ARG;
  if (c->smear_gate_channels < 0 || c->smear_gate_channels > c->n_embd) return NC_ERR_INVALID_ARG;
  if (c->ve_gate_channels < 0 || c->ve_gate_channels > c->n_embd) return NC_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.f) || !(c->softcap > 0.f) || !(c->rope_base > 0.f)) return NC_ERR_INVALID_ARG;
  if (c->logits_bf16 != 0 && c->logits_bf16 != 1) return NC_ERR_INVALID_ARG;
  if (c->fp8 != 0 && c->fp8 != 1) return NC_ERR_INVALID_ARG;
  if (c->fp8 && c->mlp_hidden % 128 != 0) return NC_ERR_UNSUPPORTED;   // the 8-bit down projection's K
  if (c->head_dim != 64 && c->head_dim != 128) return NC_ERR_UNSUPPORTED;
  if (c->n_embd % 128 != 0 || c->n_embd > 2048) return NC_ERR_UNSUPPORTED;
  if (c->mlp_hidden % 64 != 0 || c->vocab_size % 64 != 0) return NC_ERR_UNSUPPORTED;
  if (c->smear_gate_channels % 4 != 0 || c->ve_gate_channels % 8 != 0) return NC_ERR_UNSUPPORTED;
  return NC_OK;
}

size_t qkv_rows_total(const nc_config* c) {
  size_t rows = 0;
  for (int i = 0; i < c->n_layer; ++i)
    rows += (c->n_head + 2 * c->n_kv_head) * c->head_dim + (c->has_ve[i] ? c->n_kv_head * VGATE_ROWS : 0);
  return rows;
}

// The 8-bit weights after the bf16 packed q|k|v (fp8 configs only), byte offsets from the start of
// the packed buffer: e4m3 q|k|v in the bf16 one's row layout (gate rows zero), per layer W_o, W_fc,
// W_proj, then W_lm; per layer a bf16 [GATE_PAD, C] matrix of the value-embedding gate rows (the
// gate's dot product stays bf16); 1 / scale of every quantised weight ([6 L + 1] floats: q, k, v,
// o, fc, proj per layer, then the lm_head); the amax scratch of the weight quantisation.
constexpr int GATE_PAD = 32;
struct Fp8Pack {
  size_t qkv8, wo8, wfc8, wproj8, lm8, wg, wscale, part, end;
};

Fp8Pack fp8_pack_for(const nc_config* c, size_t start) {
  const size_t C = c->n_embd, HD = static_cast<size_t>(c->n_head) * c->head_dim, F = c->mlp_hidden;
  const size_t L = c->n_layer;
  Fp8Pack p{};
  size_t off = start;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  p.qkv8 = take(qkv_rows_total(c) * C);
  p.wo8 = take(L * C * HD);
  p.wfc8 = take(L * F * C);
  p.wproj8 = take(L * C * F);
  p.lm8 = take(static_cast<size_t>(c->vocab_size) * C);
  p.wg = take(L * GATE_PAD * C * sizeof(bf16));
  p.wscale = take((6 * L + 1) * sizeof(float));
  p.part = take(nc::FP8_AMAX_BLOCKS * sizeof(float));
  p.end = off;
  return p;
}

size_t packed_bf16_end(const nc_config* c) {
  const size_t status = ALIGN;
  const size_t rope = align_up(static_cast<size_t>(c->seq_len_ctx) * (c->head_dim / 2) * sizeof(float2));
  return status + rope + align_up(qkv_rows_total(c) * c->n_embd * sizeof(bf16));
}

size_t packed_bytes_for(const nc_config* c) {
  const size_t end = packed_bf16_end(c);
  return c->fp8 ? fp8_pack_for(c, end).end : end;
}

// Quantises one weight tensor [rows, cols] (bf16) to e4m3 at its own tensorwise scale, into dst
// (rows remapped as launch_fp8_quantize describes), 1 / scale into *inv.
cudaError_t quantize_weight(const void* src, int rows, int cols, uint8_t* dst, int group, int gap, float* inv,
                            float* part, cudaStream_t stream) {
  cudaError_t e = nc::launch_fp8_amax(src, 0, rows, cols, cols, nullptr, 0.f, part, stream);
  if (e == cudaSuccess)
    e = nc::launch_fp8_quantize(src, 0, rows, cols, cols, nullptr, 0.f, part, nc::FP8_AMAX_BLOCKS, dst, cols, group,
                                gap, inv, stream);
  return e;
}

// The 8-bit copies of every linear layer's weight and the bf16 gate matrices (fp8 configs).
cudaError_t pack_fp8(nc_model* m, const nc_weights* w, uint8_t* base, cudaStream_t stream) {
  const nc_config* c = &m->cfg;
  const Fp8Pack p = fp8_pack_for(c, packed_bf16_end(c));
  const int L = c->n_layer, C = c->n_embd, D = c->head_dim, F = c->mlp_hidden;
  const int qd = c->n_head * D, kd = c->n_kv_head * D;
  const size_t c_g = c->ve_gate_channels ? c->ve_gate_channels : C;
  m->wqkv8 = base + p.qkv8;
  m->wo8 = base + p.wo8;
  m->wfc8 = base + p.wfc8;
  m->wproj8 = base + p.wproj8;
  m->lm8 = base + p.lm8;
  m->wg = reinterpret_cast<bf16*>(base + p.wg);
  m->wscale = reinterpret_cast<float*>(base + p.wscale);
  float* part = reinterpret_cast<float*>(base + p.part);
  cudaError_t e = cudaMemsetAsync(m->wqkv8, 0, p.wo8 - p.qkv8, stream);   // gate rows stay zero
  if (e == cudaSuccess) e = cudaMemsetAsync(m->wg, 0, p.wscale - p.wg, stream);
  for (int i = 0; i < L && e == cudaSuccess; ++i) {
    uint8_t* q8 = m->wqkv8 + m->qkv_off[i];
    float* s = m->wscale + 6 * i;
    const bool ve = m->has_ve[i] != 0;
    e = quantize_weight(w->wq[i], qd, C, q8, 0, 0, s + 0, part, stream);
    if (e == cudaSuccess) e = quantize_weight(w->wk[i], kd, C, q8 + static_cast<size_t>(qd) * C, 0, 0, s + 1, part, stream);
    if (e == cudaSuccess)   // v heads: D rows each, followed by VGATE_ROWS (zero) rows on value-embedding layers
      e = quantize_weight(w->wv[i], kd, C, q8 + static_cast<size_t>(qd + kd) * C, ve ? D : 0, ve ? VGATE_ROWS : 0,
                          s + 2, part, stream);
    if (e == cudaSuccess)
      e = quantize_weight(w->wo[i], C, qd, m->wo8 + static_cast<size_t>(i) * C * qd, 0, 0, s + 3, part, stream);
    if (e == cudaSuccess)
      e = quantize_weight(w->wfc[i], F, C, m->wfc8 + static_cast<size_t>(i) * F * C, 0, 0, s + 4, part, stream);
    if (e == cudaSuccess)
      e = quantize_weight(w->wproj[i], C, F, m->wproj8 + static_cast<size_t>(i) * C * F, 0, 0, s + 5, part, stream);
    for (int g = 0; ve && g < c->n_kv_head && e == cudaSuccess; ++g)   // gate row g: first c_g columns
      e = cudaMemcpyAsync(m->wg + (static_cast<size_t>(i) * GATE_PAD + g) * C,
                          static_cast<const bf16*>(w->ve_gate[i]) + g * c_g, c_g * 2, cudaMemcpyDeviceToDevice,
                          stream);
  }
  if (e == cudaSuccess)
    e = quantize_weight(w->lm_head, c->vocab_size, C, m->lm8, 0, 0, m->wscale + 6 * L, part, stream);
  return e;
}

Layout layout_for(const nc_model* m, int B, int T) {
  const nc_config& c = m->cfg;
  const size_t M = static_cast<size_t>(B) * T;
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L.x0 = take(M * c.n_embd * 4);
  L.x = take(M * c.n_embd * 4);
  L.xm = take(c.use_backout ? M * c.n_embd * 4 : 0);
  L.xb = take(M * c.n_embd * 2);
  L.q = take(M * c.n_head * c.head_dim * 2);
  L.k = take(M * c.n_kv_head * c.head_dim * 2);
  L.v = take(M * c.n_kv_head * c.head_dim * 2);
  L.y = take(M * c.n_head * c.head_dim * 2);
  L.h = take(M * c.mlp_hidden * 2);
  L.ssp = take(M * (c.n_embd / nc::SS_GROUP) * 4);
  const size_t f8 = c.fp8 ? 1 : 0;
  L.a8 = take(f8 * M * c.n_embd);
  L.y8 = take(f8 * M * c.n_head * c.head_dim);
  L.h8 = take(f8 * M * c.mlp_hidden);
  L.gpre = take(f8 * M * 32 * 4);
  L.qpart = take(f8 * nc::FP8_AMAX_BLOCKS * 4);
  L.qscale = take(f8 * 8 * 4);
  L.rowmax = take(f8 * M * (c.n_embd / 32) * 4);
  L.hmax = take(f8 * c.n_layer * 4);
  L.end = off;
  return L;
}

cudaEvent_t take_event(nc_model* m) {
  if (!m->free_events.empty()) {
    cudaEvent_t e = m->free_events.back();
    m->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Runs `launch` and, with timing on, brackets it with an event pair on `stream`.
template <typename F>
cudaError_t timed(nc_model* m, int cls, cudaStream_t stream, F&& launch) {
  if (!m->timing) return launch();
  TimedLaunch t{cls, take_event(m), take_event(m)};
  cudaEventRecord(t.a, stream);
  cudaError_t e = launch();
  cudaEventRecord(t.b, stream);
  m->pending.push_back(t);
  return e;
}

void flush_timing(nc_model* m) {
  for (auto& t : m->pending) {
    float ms = 0.f;
    cudaEventSynchronize(t.b);
    if (cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      m->acc_ms[t.cls] += ms;
      m->acc_n[t.cls] += 1;
    }
    m->free_events.push_back(t.a);
    m->free_events.push_back(t.b);
  }
  m->pending.clear();
}

}  // namespace

extern "C" {

const char* nc_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "ok";
    case NC_ERR_INVALID_ARG: return "invalid argument";
    case NC_ERR_UNSUPPORTED: return "unsupported configuration";
    case NC_ERR_WORKSPACE: return "buffer smaller than required";
    case NC_ERR_CUDA: return "CUDA runtime error";
    case NC_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case NC_ERR_TOKEN_RANGE: return "token id out of range";
    default: return "unknown status";
  }
}

const char* nc_last_cuda_error(void) { return nc::last_cuda_error_name(); }

const char* nc_kernel_class_name(nc_kernel_class k) {
  static const char* names[NC_K_COUNT] = {"embed_smear",   "qkv_rope_qknorm_ve", "attention",  "oproj_residual",
                                          "fc_relu2",      "proj_residual",      "lmhead_softcap", "cross_entropy",
                                          "lmhead_grad",   "mlp_grad",           "oproj_grad",     "rmsnorm_grad",
                                          "fp8_quantize"};
  return (k >= 0 && k < NC_K_COUNT) ? names[k] : "unknown";
}

nc_status nc_model_packed_bytes(const nc_config* cfg, size_t* bytes) {
  if (bytes == nullptr) return NC_ERR_INVALID_ARG;
  nc_status s = validate_config(cfg);
  if (s != NC_OK) return s;
  *bytes = packed_bytes_for(cfg);
  return NC_OK;
}

nc_status nc_model_create(const nc_config* cfg, const nc_weights* w, void* packed_buf,
                          size_t packed_bytes, void* stream_, nc_model** out) {
  if (out == nullptr) return NC_ERR_INVALID_ARG;
  *out = nullptr;
  nc_status s = validate_config(cfg);
  if (s != NC_OK) return s;
  if (w == nullptr || packed_buf == nullptr) return NC_ERR_INVALID_ARG;
  if (!aligned(packed_buf, ALIGN)) return NC_ERR_INVALID_ARG;
  if (packed_bytes < packed_bytes_for(cfg)) return NC_ERR_WORKSPACE;
  const int L = cfg->n_layer;
  if (w->wte == nullptr || w->lm_head == nullptr || w->wq == nullptr || w->wk == nullptr ||
      w->wv == nullptr || w->wo == nullptr || w->wfc == nullptr || w->wproj == nullptr ||
      w->resid_lambdas == nullptr || w->x0_lambdas == nullptr)
    return NC_ERR_INVALID_ARG;
  if (cfg->use_smear && w->smear_gate == nullptr) return NC_ERR_INVALID_ARG;
  for (int i = 0; i < L; ++i) {
    const void* ptrs[] = {w->wq[i], w->wk[i], w->wv[i], w->wo[i], w->wfc[i], w->wproj[i]};
    for (const void* p : ptrs)
      if (p == nullptr || !aligned(p, 16)) return NC_ERR_INVALID_ARG;
    if (cfg->has_ve[i]) {
      if (w->ve_table == nullptr || w->ve_gate == nullptr || w->ve_table[i] == nullptr ||
          w->ve_gate[i] == nullptr || !aligned(w->ve_table[i], 16) || !aligned(w->ve_gate[i], 2))
        return NC_ERR_INVALID_ARG;
    }
  }
  if (!aligned(w->wte, 16) || !aligned(w->lm_head, 16)) return NC_ERR_INVALID_ARG;
  if (cfg->use_smear && !aligned(w->smear_gate, 8)) return NC_ERR_INVALID_ARG;

  nc_model* m = new (std::nothrow) nc_model();
  if (m == nullptr) return NC_ERR_INVALID_ARG;
  m->cfg = *cfg;
  m->window.assign(cfg->window_left, cfg->window_left + L);
  m->has_ve.assign(cfg->has_ve, cfg->has_ve + L);
  m->cfg.window_left = m->window.data();
  m->cfg.has_ve = m->has_ve.data();
  m->lr.assign(w->resid_lambdas, w->resid_lambdas + L);
  m->l0.assign(w->x0_lambdas, w->x0_lambdas + L);
  m->lb = w->backout_lambda;
  m->wte = static_cast<const bf16*>(w->wte);
  m->lm = static_cast<const bf16*>(w->lm_head);
  m->smear = cfg->use_smear ? static_cast<const bf16*>(w->smear_gate) : nullptr;
  for (int i = 0; i < L; ++i) {
    m->wo.push_back(static_cast<const bf16*>(w->wo[i]));
    m->wfc.push_back(static_cast<const bf16*>(w->wfc[i]));
    m->wproj.push_back(static_cast<const bf16*>(w->wproj[i]));
    m->ve.push_back(cfg->has_ve[i] ? static_cast<const bf16*>(w->ve_table[i]) : nullptr);
  }
  uint8_t* base = static_cast<uint8_t*>(packed_buf);
  m->status = reinterpret_cast<int*>(base);
  m->rope = reinterpret_cast<float2*>(base + ALIGN);
  m->wqkv = reinterpret_cast<bf16*>(
      base + ALIGN + align_up(static_cast<size_t>(cfg->seq_len_ctx) * (cfg->head_dim / 2) * sizeof(float2)));

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  m->device = dev;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t C = cfg->n_embd, D = cfg->head_dim, qd = static_cast<size_t>(cfg->n_head) * D,
               kd = static_cast<size_t>(cfg->n_kv_head) * D;
  const size_t c_g = cfg->ve_gate_channels ? cfg->ve_gate_channels : C;
  size_t off = 0;
  for (int i = 0; i < L; ++i) {
    m->qkv_off.push_back(off);
    off += static_cast<size_t>(m->Nqkv(i)) * C;
  }
  for (int i = 0; i < L && e == cudaSuccess; ++i) {
    bf16* dst = m->wqkv + m->qkv_off[i];
    e = cudaMemcpyAsync(dst, w->wq[i], qd * C * 2, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dst + qd * C, w->wk[i], kd * C * 2, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) break;
    bf16* v0 = dst + (qd + kd) * C;
    if (!cfg->has_ve[i]) {
      e = cudaMemcpyAsync(v0, w->wv[i], kd * C * 2, cudaMemcpyDeviceToDevice, stream);
      continue;
    }
    // per kv head g: its D v rows, its gate row (the first c_g columns, zeros after), 15 zero rows
    const size_t head_rows = D + VGATE_ROWS;
    e = cudaMemsetAsync(v0, 0, static_cast<size_t>(cfg->n_kv_head) * head_rows * C * 2, stream);
    for (int g = 0; g < cfg->n_kv_head && e == cudaSuccess; ++g) {
      bf16* hd = v0 + g * head_rows * C;
      e = cudaMemcpyAsync(hd, static_cast<const bf16*>(w->wv[i]) + g * D * C, D * C * 2, cudaMemcpyDeviceToDevice,
                          stream);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(hd + D * C, static_cast<const bf16*>(w->ve_gate[i]) + g * c_g, c_g * 2,
                            cudaMemcpyDeviceToDevice, stream);
    }
  }
  if (e == cudaSuccess && cfg->fp8) e = pack_fp8(m, w, base, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(m->status, 0, sizeof(int), stream);
  if (e == cudaSuccess)
    e = nc::launch_rope_table(m->rope, cfg->seq_len_ctx, cfg->head_dim, cfg->rope_base, stream);
  if (e != cudaSuccess) {
    delete m;
    return nc::cuda_status(e);
  }
  *out = m;
  return NC_OK;
}

nc_status nc_workspace_bytes(const nc_model* m, int B, int T, size_t* bytes) {
  if (m == nullptr || bytes == nullptr || B < 1 || T < 1) return NC_ERR_INVALID_ARG;
  if (T > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  *bytes = layout_for(m, B, T).end;
  return NC_OK;
}

nc_status nc_workspace_bytes_host(const nc_model* m, int B, int T, size_t* bytes) {
  size_t base = 0;
  nc_status s = nc_workspace_bytes(m, B, T, &base);
  if (s != NC_OK) return s;
  const size_t M = static_cast<size_t>(B) * T;
  *bytes = base + align_up(M * 4) + align_up(M * m->cfg.vocab_size * (m->cfg.logits_bf16 ? 2 : 4));
  return NC_OK;
}

}  // extern "C"

namespace {

// The calling thread's current device is the model's (checked before any device work).
bool on_model_device(const nc_model* m) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return dev == m->device;
}

// Argument checks shared by the forward entry points (before any device work).
nc_status check_forward_args(const nc_model* m, const int32_t* tokens, int B, int T, const void* workspace) {
  if (m == nullptr || tokens == nullptr || workspace == nullptr) return NC_ERR_INVALID_ARG;
  if (!on_model_device(m)) return NC_ERR_INVALID_ARG;
  if (B < 1 || T < 1) return NC_ERR_INVALID_ARG;
  if (T > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * T > (1LL << 30)) return NC_ERR_UNSUPPORTED;
  if (!aligned(workspace, ALIGN) || !aligned(tokens, 4)) return NC_ERR_INVALID_ARG;
  return NC_OK;
}

// Epilogue fields of a GEMM whose input is the residual stream's RMSNorm (row scale from ssp).
void set_consumer(nc::GemmEpi& e, const nc_model* m, float* ssp) {
  e.ssp_in = ssp;
  e.ncg = m->C() / nc::SS_GROUP;
  e.inv_ncols = 1.0f / static_cast<float>(m->C());
  e.eps = m->cfg.rms_eps;
  e.status = m->status;
}

// KV cache of the prefill / decode path: per layer, keys then values, each [B][cap][Hkv*D]
// bf16, cap = T_max on full layers and min(T_max, W + 1) on a layer with window W (position j in
// slot j % cap).
int kv_cap(const nc_model* m, int layer, int T_max) {
  const int w = m->window[layer];
  return w < 0 ? T_max : std::min(T_max, w + 1);
}

size_t kv_tensor_bytes(const nc_model* m, int B, int cap) {
  return align_up(static_cast<size_t>(B) * cap * m->cfg.n_kv_head * m->cfg.head_dim * sizeof(bf16));
}

size_t kv_cache_bytes(const nc_model* m, int B, int T_max) {
  size_t n = 0;
  for (int i = 0; i < m->cfg.n_layer; ++i) n += 2 * kv_tensor_bytes(m, B, kv_cap(m, i, T_max));
  return n;
}

// Where a forward writes its keys and values and which attention it runs.
struct KvCtx {
  uint8_t* cache = nullptr;
  int T_max = 0;
};

// The embedding and every block, up to the final backout: leaves the lm_head's input (before
// its RMSNorm) as xb with its partial sums of squares in ssp.  With kv, each layer's keys and
// values also go to the cache (prefill: the positions the layer's window can still see; decode:
// the new position), and a decode step attends over the cache.
cudaError_t run_blocks(nc_model* m, const int32_t* tokens, int B, int T, const Layout& Lo, uint8_t* ws,
                       cudaStream_t stream, const KvCtx* kv = nullptr, const TailOut* tail = nullptr) {
  const nc_config& c = m->cfg;
  const int M = B * T, C = c.n_embd, H = c.n_head, Hkv = c.n_kv_head, D = c.head_dim;
  const int F = c.mlp_hidden, V = c.vocab_size, L = c.n_layer;
  const int ncg = C / nc::SS_GROUP;
  float* x0 = reinterpret_cast<float*>(ws + Lo.x0);
  float* x = reinterpret_cast<float*>(ws + Lo.x);
  float* xm = reinterpret_cast<float*>(ws + Lo.xm);
  bf16* xb = reinterpret_cast<bf16*>(ws + Lo.xb);
  bf16* q = reinterpret_cast<bf16*>(ws + Lo.q);
  bf16* k = reinterpret_cast<bf16*>(ws + Lo.k);
  bf16* v = reinterpret_cast<bf16*>(ws + Lo.v);
  bf16* y = reinterpret_cast<bf16*>(ws + Lo.y);
  bf16* h = reinterpret_cast<bf16*>(ws + Lo.h);
  float* ssp = reinterpret_cast<float*>(ws + Lo.ssp);
  const int c_s = c.smear_gate_channels ? c.smear_gate_channels : C;
  const int mid = L / 2 - 1;
  uint8_t* kv_next = kv != nullptr ? kv->cache : nullptr;   // the current layer's keys, then values

  // Residual-stream update of an output projection: x += acc, bf16 copy and partial sums.
  auto resid = [&](nc::GemmEpi& e) {
    e.kind = nc::EPI_RESID;
    e.resid = x;
    e.x_out = x;
    e.xb = xb;
    e.ssp_out = ssp;
    e.ncg = ncg;
    e.status = m->status;
  };

  // 8-bit path: every linear layer's input is quantised as one tensor over the batch (its amax,
  // then its e4m3 codes; the normed stream from the fp32 x with its RMSNorm row scale), and its
  // GEMM runs on the e4m3 copies of input and weight, dequantised in the epilogue.
  const bool f8 = c.fp8 != 0;
  uint8_t* a8 = ws + Lo.a8;
  uint8_t* y8 = ws + Lo.y8;
  uint8_t* h8 = ws + Lo.h8;
  float* gpre = reinterpret_cast<float*>(ws + Lo.gpre);
  float* qpart = reinterpret_cast<float*>(ws + Lo.qpart);
  float* qscale = reinterpret_cast<float*>(ws + Lo.qscale);   // 1 / scale: [0] q|k|v input, [1] y, [2] fc input, [3] h
  // The maximum comes from a pass over the tensor, from the producer's per-row maxima of the fp32
  // stream (the residual GEMMs write them on this path), or as one word the producer raised (the
  // fc's squared ReLU); the same number each way.
  float* rowmax = reinterpret_cast<float*>(ws + Lo.rowmax);
  float* hmax = reinterpret_cast<float*>(ws + Lo.hmax);   // [L]: each block's fc output maximum
  auto quant = [&](const void* src, int f32, int cols, const float* row_ssp, uint8_t* dst, float* inv) {
    cudaError_t r = timed(m, NC_K_QUANT, stream, [&] {
      return nc::launch_fp8_amax(src, f32, M, cols, cols, row_ssp, c.rms_eps, qpart, stream);
    });
    if (r == cudaSuccess)
      r = timed(m, NC_K_QUANT, stream, [&] {
        return nc::launch_fp8_quantize(src, f32, M, cols, cols, row_ssp, c.rms_eps, qpart, nc::FP8_AMAX_BLOCKS, dst,
                                       cols, 0, 0, inv, stream);
      });
    return r;
  };
  auto quant_stream = [&](uint8_t* dst, float* inv) {   // the normed fp32 stream x, from rowmax
    cudaError_t r = timed(m, NC_K_QUANT, stream, [&] {
      return nc::launch_fp8_amax_rows(rowmax, M, C, ssp, c.rms_eps, qpart, stream);
    });
    if (r == cudaSuccess)
      r = timed(m, NC_K_QUANT, stream, [&] {
        return nc::launch_fp8_quantize(x, 1, M, C, C, ssp, c.rms_eps, qpart, nc::FP8_AMAX_BLOCKS, dst, C, 0, 0, inv,
                                       stream);
      });
    return r;
  };
  auto as8 = [](const void* p) { return static_cast<const bf16*>(p); };   // e4m3 operands travel as untyped bytes

  cudaError_t e = f8 ? cudaMemsetAsync(hmax, 0, static_cast<size_t>(L) * sizeof(float), stream) : cudaSuccess;
  if (e == cudaSuccess)
    e = timed(m, NC_K_EMBED, stream, [&] {
      return nc::launch_embed_smear(tokens, B, T, m->wte, V, C, m->smear, c_s, c.embed_norm, c.rms_eps,
                                    m->lr[0] + m->l0[0], x0, x, xb, ssp, m->status, stream);
    });
  for (int i = 0; i < L && e == cudaSuccess; ++i) {
    const bool ve = m->has_ve[i] != 0;
    nc::GemmEpi qe;
    set_consumer(qe, m, ssp);
    qe.kind = nc::EPI_QKV;
    qe.q = q;
    qe.k = k;
    qe.v = v;
    qe.H = H;
    qe.Hkv = Hkv;
    qe.D = D;
    qe.T = T;
    qe.rope = m->rope;
    qe.rope_ld = c.seq_len_ctx;
    qe.vgate = ve ? 1 : 0;
    qe.gate_scale = c.ve_gate_scale;
    qe.ve = m->ve[i];
    qe.tokens = tokens;
    qe.V = V;
    if (f8) {
      e = i == 0 ? quant(x, 1, C, ssp, a8, qscale + 0) : quant_stream(a8, qscale + 0);
      if (e == cudaSuccess && ve) {   // the value-embedding gates' dot products, bf16: rs * (xb . W_g^T)
        nc::GemmEpi ge;
        set_consumer(ge, m, ssp);
        ge.kind = nc::EPI_F32;
        ge.out = gpre;
        ge.ldo = 32;
        e = timed(m, NC_K_QKV, stream, [&] {
          return nc::launch_gemm(xb, m->wg + static_cast<size_t>(i) * GATE_PAD * C, M, GATE_PAD, C, ge, m->num_sms,
                                 stream);
        });
      }
      if (e != cudaSuccess) break;
      qe.ssp_in = nullptr;
      qe.fp8 = 1;
      qe.fp8_sa = qscale + 0;
      qe.fp8_sw = m->wscale + 6 * i;
      qe.gpre = ve ? gpre : nullptr;
      qe.gpre_ld = 32;
    }
    e = timed(m, NC_K_QKV, stream, [&] {
      return f8 ? nc::launch_gemm(as8(a8), as8(m->wqkv8 + m->qkv_off[i]), M, m->Nqkv(i), C, qe, m->num_sms, stream)
                : nc::launch_gemm(xb, m->wqkv + m->qkv_off[i], M, m->Nqkv(i), C, qe, m->num_sms, stream);
    });
    if (e != cudaSuccess) break;
    if (kv != nullptr) {
      const int cap = kv_cap(m, i, kv->T_max);
      bf16* kc = reinterpret_cast<bf16*>(kv_next);
      bf16* vc = reinterpret_cast<bf16*>(kv_next + kv_tensor_bytes(m, B, cap));
      kv_next += 2 * kv_tensor_bytes(m, B, cap);
      e = timed(m, NC_K_ATTN, stream, [&] {
        const int first = std::max(0, T - cap);
        return nc::launch_kv_append(k, v, B, T, first, T - first, 0, Hkv * D, kc, vc, cap, stream);
      });
      if (e != cudaSuccess) break;
    }
    e = timed(m, NC_K_ATTN, stream, [&] {
      return nc::launch_attention(q, k, v, B, T, H, Hkv, D, m->window[i], y, m->status, stream);
    });
    if (e != cudaSuccess) break;
    nc::GemmEpi oe;
    resid(oe);
    if (f8) {
      e = quant(y, 0, H * D, nullptr, y8, qscale + 1);
      if (e != cudaSuccess) break;
      oe.fp8 = 1;
      oe.rowmax_out = rowmax;   // the fc input's maximum
      oe.fp8_sa = qscale + 1;
      oe.fp8_sw = m->wscale + 6 * i + 3;
    }
    e = timed(m, NC_K_OPROJ, stream, [&] {
      return f8 ? nc::launch_gemm_resid(as8(y8), as8(m->wo8 + static_cast<size_t>(i) * C * H * D), M, C, H * D, oe,
                                        m->num_sms, stream)
                : nc::launch_gemm_resid(y, m->wo[i], M, C, H * D, oe, m->num_sms, stream);
    });
    if (e != cudaSuccess) break;
    nc::GemmEpi fe;
    set_consumer(fe, m, ssp);
    fe.kind = nc::EPI_RELU2_BF16;
    fe.out = h;
    fe.ldo = F;
    if (f8) {
      e = quant_stream(a8, qscale + 2);
      if (e != cudaSuccess) break;
      fe.ssp_in = nullptr;
      fe.fp8 = 1;
      fe.amax_out = hmax + i;   // the down projection's input maximum
      fe.fp8_sa = qscale + 2;
      fe.fp8_sw = m->wscale + 6 * i + 4;
    }
    e = timed(m, NC_K_FC, stream, [&] {
      return f8 ? nc::launch_gemm(as8(a8), as8(m->wfc8 + static_cast<size_t>(i) * F * C), M, F, C, fe, m->num_sms,
                                  stream)
                : nc::launch_gemm(xb, m->wfc[i], M, F, C, fe, m->num_sms, stream);
    });
    if (e != cudaSuccess) break;
    nc::GemmEpi pe;
    resid(pe);
    if (c.use_backout && i == mid) pe.xm_out = xm;
    if (i + 1 < L) {   // the next block's residual mix
      pe.a = m->lr[i + 1];
      pe.b = m->l0[i + 1];
      pe.Y = x0;
    } else {           // final: backout, then only the lm_head's inputs are needed
      pe.x_out = nullptr;
      if (c.use_backout) {
        pe.a = 1.f;
        pe.b = -m->lb;
        pe.Y = mid < 0 ? x0 : xm;
      }
      if (tail != nullptr) {   // keep the last block's MLP input for the backward
        pe.x_out = tail->xf;
        pe.xb = tail->xbf;
        pe.ssp_out = tail->sspf;
      }
      if (f8) pe.x_out = x;   // the lm_head's input is quantised from the fp32 stream
    }
    if (f8) {
      e = timed(m, NC_K_QUANT, stream, [&] {
        return nc::launch_fp8_quantize(h, 0, M, F, F, nullptr, c.rms_eps, hmax + i, 1, h8, F, 0, 0, qscale + 3,
                                       stream);
      });
      if (e != cudaSuccess) break;
      pe.fp8 = 1;
      pe.rowmax_out = rowmax;   // the next block's q|k|v input (or the lm_head's) maximum
      pe.fp8_sa = qscale + 3;
      pe.fp8_sw = m->wscale + 6 * i + 5;
    }
    e = timed(m, NC_K_PROJ, stream, [&] {
      return f8 ? nc::launch_gemm_resid(as8(h8), as8(m->wproj8 + static_cast<size_t>(i) * C * F), M, C, F, pe,
                                        m->num_sms, stream)
                : nc::launch_gemm_resid(h, m->wproj[i], M, C, F, pe, m->num_sms, stream);
    });
  }
  return e;
}

// Loss-path buffers placed after the forward's layout: the cross-entropy partials
// [ceil(V/128)][M], the target logits [M] and the reduction scratch.
struct LossLayout {
  size_t part, zt, scratch, end;
};

LossLayout loss_layout_for(const nc_model* m, const Layout& Lo, int B, int T) {
  const size_t M = static_cast<size_t>(B) * T;
  const size_t G = (m->cfg.vocab_size + 127) / 128;
  LossLayout L{};
  L.part = Lo.end;
  L.zt = L.part + align_up(G * M * 4);
  L.scratch = L.zt + align_up(M * 4);
  L.end = L.scratch + align_up(static_cast<size_t>(nc::ce_scratch_doubles(static_cast<int>(M))) * sizeof(double));
  return L;
}

// Backward buffers placed after the loss path's: the final stream and its bf16 copy and partials
// (TailOut), the per-row log-sum-exp and 1 / rows counted, the lm_head's output gradient
// dlt bf16 [M, V], the pre-norm input gradient G fp32 [M, C] (reused for both norms), the
// gradient at the last block's output (fp32 and bf16), the MLP's hidden gradient du bf16 [M, F]
// and the gradient at the last block's MLP input (bf16).
struct TailLayout {
  size_t xf, xbf, sspf, lse, invc, dlt, G, dxl, dxlb, du, dxa, split, end;
};

TailLayout tail_layout_for(const nc_model* m, const LossLayout& LL, int B, int T) {
  const nc_config& c = m->cfg;
  const size_t M = static_cast<size_t>(B) * T, C = c.n_embd;
  TailLayout L{};
  size_t off = LL.end;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L.xf = take(M * C * 4);
  L.xbf = take(M * C * 2);
  L.sspf = take(M * (C / nc::SS_GROUP) * 4);
  L.lse = take(M * 4);
  L.invc = take(4);
  L.dlt = take(M * c.vocab_size * 2);
  L.G = take(M * C * 4);
  L.dxl = take(M * C * 4);
  L.dxlb = take(M * C * 2);
  L.du = take(M * c.mlp_hidden * 2);
  L.dxa = take(M * C * 2);
  // the K-range slabs of the weight gradients split over tokens (one product at a time)
  const int Mi = static_cast<int>(M), Ci = static_cast<int>(C), F = c.mlp_hidden, HD = c.n_head * c.head_dim;
  size_t split = nc::gemm_split_ws_bytes(c.vocab_size, Ci, Mi, Ci, m->num_sms);
  split = std::max(split, nc::gemm_split_ws_bytes(Ci, F, Mi, F, m->num_sms));
  split = std::max(split, nc::gemm_split_ws_bytes(F, Ci, Mi, Ci, m->num_sms));
  split = std::max(split, nc::gemm_split_ws_bytes(Ci, HD, Mi, HD, m->num_sms));
  L.split = take(split);
  L.end = off;
  return L;
}

}  // namespace

extern "C" {

namespace {

// Bytes of one logit in the caller's output.
size_t logit_bytes(const nc_model* m) { return m->cfg.logits_bf16 ? 2 : 4; }

// The lm_head's operands: the bf16 final stream xb with the final RMSNorm as the epilogue's row
// scale, or on the 8-bit path the e4m3 quantisation of the normed final stream (from the fp32 x)
// and the e4m3 W_lm, dequantised in the epilogue.
cudaError_t lm_head_operands(nc_model* m, uint8_t* ws, const Layout& Lo, int M, cudaStream_t stream, nc::GemmEpi& le,
                             const bf16** A, const bf16** W) {
  float* ssp = reinterpret_cast<float*>(ws + Lo.ssp);
  set_consumer(le, m, ssp);
  if (!m->cfg.fp8) {
    *A = reinterpret_cast<const bf16*>(ws + Lo.xb);
    *W = m->lm;
    return cudaSuccess;
  }
  const int C = m->C();
  const float* x = reinterpret_cast<const float*>(ws + Lo.x);
  float* qpart = reinterpret_cast<float*>(ws + Lo.qpart);
  float* inv = reinterpret_cast<float*>(ws + Lo.qscale) + 4;
  uint8_t* a8 = ws + Lo.a8;
  // the maximum from the last down projection's per-row maxima of x
  const float* rowmax = reinterpret_cast<const float*>(ws + Lo.rowmax);
  cudaError_t e = timed(m, NC_K_QUANT, stream, [&] {
    return nc::launch_fp8_amax_rows(rowmax, M, C, ssp, m->cfg.rms_eps, qpart, stream);
  });
  if (e == cudaSuccess)
    e = timed(m, NC_K_QUANT, stream, [&] {
      return nc::launch_fp8_quantize(x, 1, M, C, C, ssp, m->cfg.rms_eps, qpart, nc::FP8_AMAX_BLOCKS, a8, C, 0, 0, inv,
                                     stream);
    });
  le.ssp_in = nullptr;
  le.fp8 = 1;
  le.fp8_sa = inv;
  le.fp8_sw = m->wscale + 6 * m->cfg.n_layer;
  *A = reinterpret_cast<const bf16*>(a8);
  *W = reinterpret_cast<const bf16*>(m->lm8);
  return e;
}

// The lm_head with the final RMSNorm and the soft-cap, writing fp32 or bf16 logits [M, V] as the
// config asks.
cudaError_t launch_lm_head(nc_model* m, uint8_t* ws, const Layout& Lo, int M, void* logits, cudaStream_t stream) {
  nc::GemmEpi le;
  const bf16 *A = nullptr, *W = nullptr;
  cudaError_t e = lm_head_operands(m, ws, Lo, M, stream, le, &A, &W);
  if (e != cudaSuccess) return e;
  le.kind = m->cfg.logits_bf16 ? nc::EPI_SOFTCAP_BF16 : nc::EPI_SOFTCAP_F32;
  le.out = logits;
  le.ldo = m->cfg.vocab_size;
  le.cap = m->cfg.softcap;
  return timed(m, NC_K_LMHEAD, stream, [&] {
    return nc::launch_gemm(A, W, M, m->cfg.vocab_size, m->C(), le, m->num_sms, stream);
  });
}

}  // namespace

nc_status nc_forward(nc_model* m, const int32_t* tokens, int B, int T, void* logits,
                     void* workspace, size_t ws_bytes, void* stream_) {
  nc_status s = check_forward_args(m, tokens, B, T, workspace);
  if (s != NC_OK) return s;
  if (logits == nullptr || !aligned(logits, 16)) return NC_ERR_INVALID_ARG;
  const Layout Lo = layout_for(m, B, T);
  if (ws_bytes < Lo.end) return NC_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = run_blocks(m, tokens, B, T, Lo, ws, stream);
  if (e == cudaSuccess)
    e = launch_lm_head(m, ws, Lo, B * T, logits, stream);
  return nc::cuda_status(e);
}

nc_status nc_workspace_bytes_loss(const nc_model* m, int B, int T, size_t* bytes) {
  if (m == nullptr || bytes == nullptr || B < 1 || T < 1) return NC_ERR_INVALID_ARG;
  if (T > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * T > (1LL << 30)) return NC_ERR_UNSUPPORTED;
  *bytes = loss_layout_for(m, layout_for(m, B, T), B, T).end;
  return NC_OK;
}

nc_status nc_forward_loss(nc_model* m, const int32_t* tokens, const int32_t* targets, int B, int T,
                          const int32_t* token_bytes, float* loss, float* stats, void* workspace,
                          size_t ws_bytes, void* stream_) {
  nc_status s = check_forward_args(m, tokens, B, T, workspace);
  if (s != NC_OK) return s;
  if (targets == nullptr || stats == nullptr || !aligned(targets, 4) || !aligned(stats, 4) ||
      (loss != nullptr && !aligned(loss, 4)) || (token_bytes != nullptr && !aligned(token_bytes, 4)))
    return NC_ERR_INVALID_ARG;
  const Layout Lo = layout_for(m, B, T);
  const LossLayout LL = loss_layout_for(m, Lo, B, T);
  if (ws_bytes < LL.end) return NC_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int M = B * T, V = m->cfg.vocab_size;
  float* part = reinterpret_cast<float*>(ws + LL.part);
  float* zt = reinterpret_cast<float*>(ws + LL.zt);
  cudaError_t e = run_blocks(m, tokens, B, T, Lo, ws, stream);
  if (e == cudaSuccess) {
    nc::GemmEpi le;
    const bf16 *A = nullptr, *W = nullptr;
    e = lm_head_operands(m, ws, Lo, M, stream, le, &A, &W);
    le.kind = nc::EPI_CE;
    le.cap = m->cfg.softcap;
    le.targets = targets;
    le.ce_part = part;
    le.ce_zt = zt;
    if (e == cudaSuccess)
      e = timed(m, NC_K_LMHEAD, stream, [&] { return nc::launch_gemm(A, W, M, V, m->C(), le, m->num_sms, stream); });
  }
  if (e == cudaSuccess)
    e = timed(m, NC_K_LOSS, stream, [&] {
      return nc::launch_ce_finalize(part, zt, targets, M, (V + 127) / 128, V, token_bytes, loss, stats,
                                    reinterpret_cast<double*>(ws + LL.scratch), m->status, stream);
    });
  return nc::cuda_status(e);
}

nc_status nc_workspace_bytes_grad_tail(const nc_model* m, int B, int T, size_t* bytes) {
  if (m == nullptr || bytes == nullptr || B < 1 || T < 1) return NC_ERR_INVALID_ARG;
  if (m->cfg.fp8) return NC_ERR_UNSUPPORTED;   // the backward runs on the bf16 path
  if (T > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * T > (1LL << 30)) return NC_ERR_UNSUPPORTED;
  const Layout Lo = layout_for(m, B, T);
  *bytes = tail_layout_for(m, loss_layout_for(m, Lo, B, T), B, T).end;
  return NC_OK;
}

nc_status nc_forward_loss_grad_tail(nc_model* m, const int32_t* tokens, const int32_t* targets, int B, int T,
                                    const int32_t* token_bytes, float* stats, float* grad_lm_head,
                                    float* grad_wproj, float* grad_wfc, float* grad_wo, void* workspace,
                                    size_t ws_bytes, void* stream_) {
  nc_status s = check_forward_args(m, tokens, B, T, workspace);
  if (s != NC_OK) return s;
  if (m->cfg.fp8) return NC_ERR_UNSUPPORTED;
  if (targets == nullptr || stats == nullptr || !aligned(targets, 4) || !aligned(stats, 4) ||
      (token_bytes != nullptr && !aligned(token_bytes, 4)))
    return NC_ERR_INVALID_ARG;
  for (const float* g : {grad_lm_head, grad_wproj, grad_wfc, grad_wo})
    if (g == nullptr || !aligned(g, 16)) return NC_ERR_INVALID_ARG;
  const Layout Lo = layout_for(m, B, T);
  const LossLayout LL = loss_layout_for(m, Lo, B, T);
  const TailLayout TL = tail_layout_for(m, LL, B, T);
  if (ws_bytes < TL.end) return NC_ERR_WORKSPACE;
  const nc_config& c = m->cfg;
  const int M = B * T, V = c.vocab_size, C = c.n_embd, F = c.mlp_hidden, HD = c.n_head * c.head_dim;
  const int last = c.n_layer - 1;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  auto b16 = [&](size_t off) { return reinterpret_cast<nc::bf16*>(ws + off); };
  const TailOut tail{f32(TL.xf), b16(TL.xbf), f32(TL.sspf)};
  float* part = f32(LL.part);
  float* zt = f32(LL.zt);

  // forward, keeping the last block's MLP input (x, xb, ssp) and its h and y
  cudaError_t e = run_blocks(m, tokens, B, T, Lo, ws, stream, nullptr, &tail);
  if (e == cudaSuccess) {   // loss: cross-entropy partials, then log-sum-exp, 1 / count, mean loss
    nc::GemmEpi le;
    set_consumer(le, m, tail.sspf);
    le.kind = nc::EPI_CE;
    le.cap = c.softcap;
    le.targets = targets;
    le.ce_part = part;
    le.ce_zt = zt;
    e = timed(m, NC_K_LMHEAD, stream, [&] { return nc::launch_gemm(tail.xbf, m->lm, M, V, C, le, m->num_sms, stream); });
  }
  if (e == cudaSuccess)
    e = timed(m, NC_K_LOSS, stream, [&] {
      return nc::launch_ce_finalize(part, zt, targets, M, (V + 127) / 128, V, token_bytes, nullptr, stats,
                                    reinterpret_cast<double*>(ws + LL.scratch), m->status, stream, f32(TL.lse),
                                    f32(TL.invc));
    });
  // the lm_head's output gradient (the logits recomputed), then its input and weight gradients
  auto gemm = [&](int cls, const nc::bf16* A, const nc::bf16* Bm, int Mg, int Ng, int Kg, nc::GemmEpi& ge) {
    ge.status = m->status;
    return timed(m, cls, stream, [&] { return nc::launch_gemm(A, Bm, Mg, Ng, Kg, ge, m->num_sms, stream); });
  };
  if (e == cudaSuccess) {
    nc::GemmEpi ge;
    set_consumer(ge, m, tail.sspf);
    ge.kind = nc::EPI_CE_GRAD;
    ge.cap = c.softcap;
    ge.targets = targets;
    ge.ce_lse = f32(TL.lse);
    ge.inv_count = f32(TL.invc);
    ge.out = b16(TL.dlt);
    ge.ldo = V;
    e = gemm(NC_K_LMHEAD_GRAD, tail.xbf, m->lm, M, V, C, ge);
  }
  if (e == cudaSuccess) {   // G = dlt . W_lm   (W_lm [V][C]: N-contiguous B)
    nc::GemmEpi ge;
    ge.kind = nc::EPI_F32;
    ge.b_mn = 1;
    ge.out = f32(TL.G);
    ge.ldo = C;
    e = gemm(NC_K_LMHEAD_GRAD, b16(TL.dlt), m->lm, M, C, V, ge);
  }
  if (e == cudaSuccess) {   // dW_lm = dlt^T . xbf   (both token-major)
    nc::GemmEpi ge;
    ge.kind = nc::EPI_F32;
    ge.a_mn = 1;
    ge.b_mn = 1;
    ge.out = grad_lm_head;
    ge.split_ws = f32(TL.split);
    ge.ldo = C;
    e = gemm(NC_K_LMHEAD_GRAD, b16(TL.dlt), tail.xbf, V, C, M, ge);
  }
  // the final RMSNorm's backward: the gradient at the last block's output (the backout
  // subtracts a stream that does not depend on the last block)
  if (e == cudaSuccess)
    e = timed(m, NC_K_RMS_GRAD, stream, [&] {
      return nc::launch_rms_backward(f32(TL.G), tail.xf, tail.sspf, nullptr, M, C, c.rms_eps, f32(TL.dxl),
                                     b16(TL.dxlb), stream);
    });
  const nc::bf16* h = b16(Lo.h);
  const nc::bf16* xb = b16(Lo.xb);
  float* ssp = f32(Lo.ssp);
  if (e == cudaSuccess) {   // du' = rs . (dxl . W_proj) * 2 sqrt(h)   (W_proj [C][F]: N-contiguous B)
    nc::GemmEpi ge;
    set_consumer(ge, m, ssp);
    ge.kind = nc::EPI_DRELU2;
    ge.b_mn = 1;
    ge.h_in = h;
    ge.out = b16(TL.du);
    ge.ldo = F;
    e = gemm(NC_K_MLP_GRAD, b16(TL.dxlb), m->wproj[last], M, F, C, ge);
  }
  if (e == cudaSuccess) {   // dW_proj = dxl^T . h
    nc::GemmEpi ge;
    ge.kind = nc::EPI_F32;
    ge.a_mn = 1;
    ge.b_mn = 1;
    ge.out = grad_wproj;
    ge.split_ws = f32(TL.split);
    ge.ldo = F;
    e = gemm(NC_K_MLP_GRAD, b16(TL.dxlb), h, C, F, M, ge);
  }
  if (e == cudaSuccess) {   // dW_fc = du'^T . xb   (du' carries the MLP input's row scale)
    nc::GemmEpi ge;
    ge.kind = nc::EPI_F32;
    ge.a_mn = 1;
    ge.b_mn = 1;
    ge.out = grad_wfc;
    ge.split_ws = f32(TL.split);
    ge.ldo = C;
    e = gemm(NC_K_MLP_GRAD, b16(TL.du), xb, F, C, M, ge);
  }
  if (e == cudaSuccess) {   // G = du' . W_fc   (W_fc [F][C]: N-contiguous B)
    nc::GemmEpi ge;
    ge.kind = nc::EPI_F32;
    ge.b_mn = 1;
    ge.out = f32(TL.G);
    ge.ldo = C;
    e = gemm(NC_K_MLP_GRAD, b16(TL.du), m->wfc[last], M, C, F, ge);
  }
  // the MLP input's RMSNorm backward plus the residual path: the gradient at the stream after the
  // attention's output projection, then that projection's weight gradient
  if (e == cudaSuccess)
    e = timed(m, NC_K_RMS_GRAD, stream, [&] {
      return nc::launch_rms_backward(f32(TL.G), f32(Lo.x), ssp, f32(TL.dxl), M, C, c.rms_eps, nullptr, b16(TL.dxa),
                                     stream);
    });
  if (e == cudaSuccess) {   // dW_o = dxa^T . y
    nc::GemmEpi ge;
    ge.kind = nc::EPI_F32;
    ge.a_mn = 1;
    ge.b_mn = 1;
    ge.out = grad_wo;
    ge.split_ws = f32(TL.split);
    ge.ldo = HD;
    e = gemm(NC_K_OPROJ_GRAD, b16(TL.dxa), b16(Lo.y), C, HD, M, ge);
  }
  return nc::cuda_status(e);
}

nc_status nc_kv_cache_bytes(const nc_model* m, int B, int T_max, size_t* bytes) {
  if (m == nullptr || bytes == nullptr || B < 1 || T_max < 1) return NC_ERR_INVALID_ARG;
  // the 8-bit path's scales span the whole batch of a call, so a decode step could not reproduce
  // the full forward: the cache paths run bf16 only
  if (m->cfg.fp8) return NC_ERR_UNSUPPORTED;
  if (T_max > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  *bytes = kv_cache_bytes(m, B, T_max);
  return NC_OK;
}

nc_status nc_prefill(nc_model* m, const int32_t* tokens, int B, int T, void* kv_cache, size_t cache_bytes,
                     int T_max, void* logits, void* workspace, size_t ws_bytes, void* stream_) {
  nc_status s = check_forward_args(m, tokens, B, T, workspace);
  if (s != NC_OK) return s;
  if (m->cfg.fp8) return NC_ERR_UNSUPPORTED;
  if (logits == nullptr || !aligned(logits, 16) || kv_cache == nullptr || !aligned(kv_cache, ALIGN))
    return NC_ERR_INVALID_ARG;
  if (T_max < T) return NC_ERR_INVALID_ARG;
  if (T_max > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  if (cache_bytes < kv_cache_bytes(m, B, T_max)) return NC_ERR_WORKSPACE;
  const Layout Lo = layout_for(m, B, T);
  if (ws_bytes < Lo.end) return NC_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  KvCtx kv;
  kv.cache = static_cast<uint8_t*>(kv_cache);
  kv.T_max = T_max;
  cudaError_t e = run_blocks(m, tokens, B, T, Lo, ws, stream, &kv);
  if (e == cudaSuccess)
    e = launch_lm_head(m, ws, Lo, B * T, logits, stream);
  return nc::cuda_status(e);
}

namespace {

// Buffers of a decode step that the forward's layout does not have: after Lo.end, the pair
// tokens [B][2] int32, the q|k|v products [B][max Nqkv] fp32 and the partial sums of squares
// [B][C / 8] fp32 that the residual products write.
struct DecodeLayout {
  size_t pair, raw, ssp8, end;
  int ldraw;
};

DecodeLayout decode_layout(const nc_model* m, int B) {
  DecodeLayout d;
  int nq = 0;
  for (int i = 0; i < m->cfg.n_layer; ++i) nq = std::max(nq, m->Nqkv(i));
  d.ldraw = nq;
  d.pair = layout_for(m, B, 2).end;
  d.raw = d.pair + align_up(2 * static_cast<size_t>(B) * 4);
  d.ssp8 = d.raw + align_up(static_cast<size_t>(B) * nq * 4);
  d.end = d.ssp8 + align_up(static_cast<size_t>(B) * (m->cfg.n_embd / 8) * 4);
  return d;
}

// One decode step (one new token per batch row at position pos), "nanochat — 架构与原理" section 2
// (engine: KV cache, one token at a time).  The embedding runs on the pairs (token at pos - 1,
// token at pos), so that its smear sees the previous token; everything after it runs on the B
// second rows only (row 2b + 1 of the pair buffers): per layer the q|k|v product, its RoPE /
// QK-norm / value-embedding epilogue with the cache append and the attention over the cache (one
// launch), then the out-projection, fc and down-projection products with their
// residual, squared-ReLU and mixing epilogues; finally the lm_head straight into `logits`.
cudaError_t run_decode(nc_model* m, const int32_t* pair, const int32_t* tokens, int B, int pos, uint8_t* cache,
                       int T_max, void* logits, uint8_t* ws, cudaStream_t stream) {
  const nc_config& c = m->cfg;
  const int C = c.n_embd, H = c.n_head, Hkv = c.n_kv_head, D = c.head_dim, F = c.mlp_hidden, V = c.vocab_size;
  const int L = c.n_layer, HD = H * D, ncg = C / nc::SS_GROUP, n8 = C / 8;
  const Layout Lo = layout_for(m, B, 2);
  const DecodeLayout dl = decode_layout(m, B);
  // the second row of each pair: row 2b + 1, pitch two rows
  float* x0 = reinterpret_cast<float*>(ws + Lo.x0) + C;
  float* x = reinterpret_cast<float*>(ws + Lo.x) + C;
  float* xm = reinterpret_cast<float*>(ws + Lo.xm) + C;
  bf16* xb = reinterpret_cast<bf16*>(ws + Lo.xb) + C;
  bf16* y = reinterpret_cast<bf16*>(ws + Lo.y);   // the attention writes row 2b + 1 of its pair
  bf16* h = reinterpret_cast<bf16*>(ws + Lo.h);   // dense [B][F]
  float* ssp0 = reinterpret_cast<float*>(ws + Lo.ssp) + ncg;
  float* raw = reinterpret_cast<float*>(ws + dl.raw);
  float* ssp8 = reinterpret_cast<float*>(ws + dl.ssp8);
  const int c_s = c.smear_gate_channels ? c.smear_gate_channels : C;
  const int mid = L / 2 - 1;
  const float inv_c = 1.0f / static_cast<float>(C);
  uint8_t* kv_next = cache;

  auto scale_from = [&](nc::GemvEpi& g, bool first) {   // the input's RMSNorm partials
    g.ssp = first ? ssp0 : ssp8;
    g.ssp_ld = first ? 2 * ncg : n8;
    g.ssp_n = first ? ncg : n8;
    g.inv_ncols = inv_c;
    g.eps = c.rms_eps;
  };
  auto resid = [&](nc::GemvEpi& g) {
    g.kind = nc::GEMV_RESID;
    g.resid = x;
    g.x_out = x;
    g.ldx = 2 * C;
    g.xb = xb;
    g.ldb = 2 * C;
    g.ssp_out = ssp8;
    g.ssp_out_ld = n8;
  };

  cudaError_t e = timed(m, NC_K_EMBED, stream, [&] {
    return nc::launch_embed_smear(pair, B, 2, m->wte, V, C, m->smear, c_s, c.embed_norm, c.rms_eps,
                                  m->lr[0] + m->l0[0], reinterpret_cast<float*>(ws + Lo.x0),
                                  reinterpret_cast<float*>(ws + Lo.x), reinterpret_cast<bf16*>(ws + Lo.xb),
                                  reinterpret_cast<float*>(ws + Lo.ssp), m->status, stream);
  });
  for (int i = 0; i < L && e == cudaSuccess; ++i) {
    const int cap = kv_cap(m, i, T_max);
    bf16* kc = reinterpret_cast<bf16*>(kv_next);
    bf16* vc = reinterpret_cast<bf16*>(kv_next + kv_tensor_bytes(m, B, cap));
    kv_next += 2 * kv_tensor_bytes(m, B, cap);
    nc::GemvEpi qe;
    qe.kind = nc::GEMV_RAW;
    scale_from(qe, i == 0);
    qe.out = raw;
    qe.ldo = dl.ldraw;
    e = timed(m, NC_K_QKV, stream, [&] {
      return nc::launch_gemv(xb, 2 * C, B, m->wqkv + m->qkv_off[i], m->Nqkv(i), C, qe, stream);
    });
    if (e != cudaSuccess) break;
    e = timed(m, NC_K_ATTN, stream, [&] {
      nc::DecodeAttn da;
      da.raw = raw;
      da.ldraw = dl.ldraw;
      da.B = B;
      da.H = H;
      da.Hkv = Hkv;
      da.D = D;
      da.vgate = m->has_ve[i] ? 1 : 0;
      da.gate_scale = c.ve_gate_scale;
      da.ve = m->ve[i];
      da.tokens = tokens;
      da.V = V;
      da.rope = m->rope;
      da.rope_ld = c.seq_len_ctx;
      da.pos = pos;
      da.eps = c.rms_eps;
      da.kc = kc;
      da.vc = vc;
      da.cap = cap;
      da.window = m->window[i];
      da.y = y + HD;
      da.ldy = 2 * HD;
      return nc::launch_decode_attention(da, stream);
    });
    if (e != cudaSuccess) break;
    nc::GemvEpi oe;
    resid(oe);
    e = timed(m, NC_K_OPROJ, stream, [&] { return nc::launch_gemv(y + HD, 2 * HD, B, m->wo[i], C, HD, oe, stream); });
    if (e != cudaSuccess) break;
    nc::GemvEpi fe;
    fe.kind = nc::GEMV_RELU2;
    scale_from(fe, false);
    fe.out = h;
    fe.ldo = F;
    e = timed(m, NC_K_FC, stream, [&] { return nc::launch_gemv(xb, 2 * C, B, m->wfc[i], F, C, fe, stream); });
    if (e != cudaSuccess) break;
    nc::GemvEpi pe;
    resid(pe);
    if (c.use_backout && i == mid) pe.xm_out = xm;
    if (i + 1 < L) {   // the next block's residual mix
      pe.a = m->lr[i + 1];
      pe.b = m->l0[i + 1];
      pe.Y = x0;
    } else {           // final: backout; the lm_head needs only xb and the partials
      pe.x_out = nullptr;
      if (c.use_backout) {
        pe.a = 1.f;
        pe.b = -m->lb;
        pe.Y = mid < 0 ? x0 : xm;
      }
    }
    e = timed(m, NC_K_PROJ, stream, [&] { return nc::launch_gemv(h, F, B, m->wproj[i], C, F, pe, stream); });
  }
  if (e == cudaSuccess) {
    nc::GemvEpi le;
    le.kind = logit_bytes(m) == 2 ? nc::GEMV_SOFTCAP_BF16 : nc::GEMV_SOFTCAP_F32;
    scale_from(le, L == 0);
    le.out = logits;
    le.ldo = V;
    le.cap = c.softcap;
    e = timed(m, NC_K_LMHEAD, stream, [&] { return nc::launch_gemv(xb, 2 * C, B, m->lm, V, C, le, stream); });
  }
  return e;
}

}  // namespace

nc_status nc_workspace_bytes_decode(const nc_model* m, int B, size_t* bytes) {
  if (m == nullptr || bytes == nullptr || B < 1) return NC_ERR_INVALID_ARG;
  if (m->cfg.fp8) return NC_ERR_UNSUPPORTED;
  if (m->cfg.seq_len_ctx < 2) return NC_ERR_UNSUPPORTED;
  *bytes = decode_layout(m, B).end;
  return NC_OK;
}

nc_status nc_decode_step(nc_model* m, const int32_t* prev_tokens, const int32_t* tokens, int B, int pos,
                         void* kv_cache, size_t cache_bytes, int T_max, void* logits, void* workspace,
                         size_t ws_bytes, void* stream_) {
  if (m == nullptr || prev_tokens == nullptr || tokens == nullptr || logits == nullptr || kv_cache == nullptr ||
      workspace == nullptr || B < 1)
    return NC_ERR_INVALID_ARG;
  if (!on_model_device(m)) return NC_ERR_INVALID_ARG;
  if (m->cfg.fp8) return NC_ERR_UNSUPPORTED;
  if (!aligned(prev_tokens, 4) || !aligned(tokens, 4) || !aligned(logits, 16) || !aligned(kv_cache, ALIGN) ||
      !aligned(workspace, ALIGN))
    return NC_ERR_INVALID_ARG;
  if (pos < 1 || pos >= T_max) return NC_ERR_INVALID_ARG;
  if (T_max > m->cfg.seq_len_ctx) return NC_ERR_UNSUPPORTED;
  if (cache_bytes < kv_cache_bytes(m, B, T_max)) return NC_ERR_WORKSPACE;
  size_t need = 0;
  nc_status s = nc_workspace_bytes_decode(m, B, &need);
  if (s != NC_OK) return s;
  if (ws_bytes < need) return NC_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* pair = reinterpret_cast<int32_t*>(ws + decode_layout(m, B).pair);   // [B][2] (prev, token)
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // Each row becomes the pair (previous token, new token) for the embedding, whose smear reads
  // the previous token's embedding; the rest of the step runs on the second rows.
  cudaError_t e = cudaMemcpy2DAsync(pair, 8, prev_tokens, 4, 4, B, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpy2DAsync(pair + 1, 8, tokens, 4, 4, B, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = run_decode(m, pair, tokens, B, pos, static_cast<uint8_t*>(kv_cache), T_max, logits, ws, stream);
  return nc::cuda_status(e);
}

nc_status nc_forward_host(nc_model* m, const int32_t* tokens_host, int B, int T, void* logits_host,
                          void* workspace, size_t ws_bytes, void* stream_) {
  if (m == nullptr || tokens_host == nullptr || logits_host == nullptr || workspace == nullptr)
    return NC_ERR_INVALID_ARG;
  size_t need = 0;
  nc_status s = nc_workspace_bytes_host(m, B, T, &need);
  if (s != NC_OK) return s;
  if (ws_bytes < need) return NC_ERR_WORKSPACE;
  if (!aligned(workspace, ALIGN)) return NC_ERR_INVALID_ARG;
  size_t base = 0;
  nc_workspace_bytes(m, B, T, &base);
  const size_t M = static_cast<size_t>(B) * T;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* tok_dev = reinterpret_cast<int32_t*>(ws + base);
  void* logits_dev = ws + base + align_up(M * 4);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  s = nc::cuda_status(cudaMemcpyAsync(tok_dev, tokens_host, M * 4, cudaMemcpyHostToDevice, stream));
  if (s != NC_OK) return s;
  s = nc_forward(m, tok_dev, B, T, logits_dev, workspace, base, stream_);
  if (s != NC_OK) return s;
  s = nc::cuda_status(
      cudaMemcpyAsync(logits_host, logits_dev, M * m->cfg.vocab_size * logit_bytes(m), cudaMemcpyDeviceToHost, stream));
  if (s != NC_OK) return s;
  return nc::cuda_status(cudaStreamSynchronize(stream));
}

nc_status nc_get_status(nc_model* m, void* stream_) {
  if (m == nullptr) return NC_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int h = 0;
  nc_status s = nc::cuda_status(cudaStreamSynchronize(stream));
  if (s == NC_OK) s = nc::cuda_status(cudaMemcpy(&h, m->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (s == NC_OK) s = nc::cuda_status(cudaMemset(m->status, 0, sizeof(int)));
  if (s != NC_OK) return s;
  return static_cast<nc_status>(h);
}

void nc_model_destroy(nc_model* m) {
  if (m == nullptr) return;
  flush_timing(m);
  for (cudaEvent_t e : m->free_events) cudaEventDestroy(e);
  delete m;
}

nc_status nc_timing_enable(nc_model* m, int enable) {
  if (m == nullptr) return NC_ERR_INVALID_ARG;
  m->timing = enable != 0;
  return NC_OK;
}

nc_status nc_timing_read(nc_model* m, nc_kernel_class k, double* total_ms, int* launches) {
  if (m == nullptr || total_ms == nullptr || launches == nullptr || k < 0 || k >= NC_K_COUNT)
    return NC_ERR_INVALID_ARG;
  flush_timing(m);
  *total_ms = m->acc_ms[k];
  *launches = m->acc_n[k];
  m->acc_ms[k] = 0.0;
  m->acc_n[k] = 0;
  return NC_OK;
}

int nc_forward_launch_count(const nc_model* m) {
  if (m == nullptr) return 0;
  if (!m->cfg.fp8) return 2 + 5 * m->cfg.n_layer;
  // 8-bit: per block four quantisations (two launches each, but one for the fc output, whose
  // maximum the fc epilogue keeps) and the gate product on value-embedding layers; the lm_head's
  // input quantisation
  int ve = 0;
  for (int i = 0; i < m->cfg.n_layer; ++i) ve += m->has_ve[i] ? 1 : 0;
  return 2 + 5 * m->cfg.n_layer + 7 * m->cfg.n_layer + ve + 2;
}

int nc_kv_launch_count(const nc_model* m) {
  if (m == nullptr) return 0;
  return 2 + 5 * m->cfg.n_layer;   // a decode step: per layer q|k|v, attention (with the cache
                                   // append), out-projection, fc, down projection
}

int nc_forward_loss_launch_count(const nc_model* m) {
  if (m == nullptr) return 0;
  return nc_forward_launch_count(m) + 2;   // + the two cross-entropy reduction kernels
}

int nc_grad_tail_launch_count(const nc_model* m) {
  if (m == nullptr) return 0;
  // the loss path, then the lm_head's output, input and weight gradients, two RMSNorm backwards,
  // four MLP gradient products and the attention output projection's weight gradient
  return nc_forward_loss_launch_count(m) + 3 + 2 + 4 + 1;
}

}  // extern "C"
