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
// are taken round-robin with the column-block index fastest, so the pairs running at the same
// time share one row block of A (read from DRAM once) and the weights stay in L2.
// Roles (384 threads = 12 warps per CTA; warpgroup 0 runs at 56 registers per thread and the two
// epilogue warpgroups at 224, moved with setmaxnreg within the launch's 384 x 168):
//   warp 0       TMA producer (both CTAs): its A box (128x64) and B half (128x64) per stage,
//                128-byte swizzle, a 4- to 7-stage ring (the depth depends on how much shared
//                memory the epilogue kind keeps: Cfg::STAGES); both CTAs' copies complete on
//                the leader CTA's full barrier, which the leader arms with the pair's byte count.
//   warp 1       allocates 512 TMEM columns in both CTAs (two 128x256 fp32 accumulators);
//                in the leader one lane issues tcgen05.mma (M=256, N=256, K=16) for the pair;
//                pair commits free each stage in both CTAs and publish each finished
//                accumulator to both CTAs' epilogues.
//   warps 2, 3   idle (they complete warpgroup 0 for the register reallocation).
//   warps 4..11  epilogue: two warpgroups, each owns 128 accumulator columns; every thread
//                owns one output row (TMEM lane).  A warp reads its 32 rows with tcgen05.ld and
//                applies the fused epilogue; depending on the kind it stores 32-row x 128-byte
//                boxes with TMA from two alternating 128-byte-swizzled shared buffers, stores
//                row-coalesced from one staging buffer, stores whole sectors straight from the
//                registers (fp32 outputs), or stores nothing (cross-entropy).
// The double-buffered accumulator lets the epilogue of tile i overlap the MMAs of tile i+1.
//
// Fused epilogues (the operations are those of "Nanochat在nanoGPT之上的新增功能", section 1
// feature table and notes; RMSNorm has no weight, so norm(x) W^T = diag(1/rms(x)) (x W^T) and
// the normalisation of a GEMM's input becomes a per-row scale of its accumulator):
//   EPI_RELU2_BF16   squared ReLU of the MLP up projection, input RMSNorm as a row scale
//   EPI_SOFTCAP_F32  tanh soft-cap (+-cap) of the untied lm_head logits, final RMSNorm as a row
//                    scale (hardware tanh); EPI_SOFTCAP_BF16 the same logits rounded to bf16
//   EPI_CE           the lm_head with soft-cap and cross-entropy: per row and 128-column group,
//                    the sum of exp(logit) and the target's logit; no logits are stored
//   EPI_QKV          split of the packed q|k|v projection, input RMSNorm as a row scale; RoPE
//                    then per-head RMSNorm of q and k; on value-embedding layers each kv head's
//                    v rows are followed in the packed weight by its gate row (and 15 zero rows),
//                    so the head's tile (N = D + 16) also yields the gate's pre-activation
//                    x . w_gate and the epilogue adds gate * ve[token] with
//                    gate = scale * sigmoid(rs * (x . w_gate)) -- the gate is a contraction, so it
//                    runs on the tensor cores with the projection it belongs to
//   EPI_BF16         plain store (used by tests of the mainloop)
// and the backward of the loss and the MLP (the gradient of the mean next-token cross-entropy,
// "NanoChat基础训练报告", loss progression table: the training loss):
//   EPI_F32          rs * acc in fp32: weight gradients and input gradients before their RMSNorm
//   EPI_CE_GRAD      the lm_head recomputed with the forward's row scale and soft-cap, written as
//                    rs * (softmax(z) - onehot(target)) * (1 - (z/cap)^2) / (rows counted) in bf16:
//                    the gradient at its pre-cap output, with the row scale the weight gradient needs
//   EPI_DRELU2       rs * acc * 2 sqrt(h): the squared ReLU's derivative, from the forward's h
//
// Operand layouts: A and B are K-contiguous (nn.Linear weights, token-major activations) unless
// GemmEpi::a_mn / b_mn mark one as MN-contiguous (stored [K][M] or [K][N]), as the backward's
// products need: a weight gradient dW = G^T X contracts over tokens, so both of its operands are
// token-major [K][rows]; an input gradient dX = G W multiplies by the weight itself, [K][N].  An
// MN-contiguous stage is two TMA boxes [64 k][64 rows] with 128-byte swizzle, described to the
// MMA with the MN-major descriptor (8-row groups 1024 B apart, 64-row blocks 8 KB apart) and the
// instruction descriptor's transpose bit for that operand.  K may be ragged: TMA fills the k
// positions past the end with zeros.
// The residual-stream updates of the output projections are in gemm_resid.cu.
#include "internal.h"
#include "ptx.cuh"

#include <mutex>

namespace nc {
namespace {

constexpr int BM = 128;            // rows of A (and of D) held by each CTA of a pair
constexpr int PAIR_M = 2 * BM;     // rows of one pair tile
constexpr int BN = 256;            // columns of one pair tile
constexpr int B_ROWS = BN / 2;     // rows of B (columns of D) loaded by each CTA
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = B_ROWS * BK * 2;
constexpr int MN_BLOCK = 64 * BK * 2;   // an MN-contiguous operand's [64 k][64 rows] box (8 KB)
static_assert(A_BYTES == 2 * MN_BLOCK && B_BYTES == 2 * MN_BLOCK, "two MN boxes per operand stage");
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                    // epilogue warps 4..11 (warpgroups 1 and 2)
constexpr int THREADS = 32 * (EPI_WARP0 + NUM_EPI_WARPS);
// Register split (launch: 384 threads x 168): warpgroup 0 (TMA producer, MMA issuer, two idle
// warps) drops to 56, the two epilogue warpgroups rise to 224: 128*56 + 256*224 = 384*168.
constexpr int REGS_CTRL = 56, REGS_EPI = 224;
static_assert(128 * REGS_CTRL + 256 * REGS_EPI <= THREADS * 168, "register split exceeds the launch allocation");
constexpr int MAX_NCG = 16;                     // column groups of a row (n_embd <= 2048)
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int SLAB_BUF = 32 * 128;       // one staging buffer: 32 rows x 128 B
constexpr int SLAB_BYTES = 2 * SLAB_BUF; // two per epilogue warp, used alternately


// Shared memory per epilogue kind.  Kinds whose epilogue stores with TMA keep two staging
// buffers per warp (a store drains from one while the next is filled) and a 5-stage operand
// ring; the bf16 epilogues that store row-coalesced use one buffer, and the space saved
// deepens their ring to 6 stages (operand latency is what starves the MMA).  The fp32 outputs
// (stored from registers) and the cross-entropy epilogue (no tile stored) keep no staging
// buffers and a 7-stage ring.
template <int KIND, int D>
struct Cfg {
  // fp32 outputs and the cross-entropy partials need no staging; the other kinds stored by
  // plain instructions stage one [32 rows][128 B] buffer per warp, the TMA-stored ones two
  static constexpr bool NO_SLAB = KIND == EPI_CE || KIND == EPI_SOFTCAP_F32 || KIND == EPI_F32;
  static constexpr bool LSU_STORE = KIND == EPI_RELU2_BF16 || KIND == EPI_SOFTCAP_BF16 || KIND == EPI_CE_GRAD ||
                                    KIND == EPI_DRELU2;
  static constexpr int STAGES = NO_SLAB ? 7 : (LSU_STORE ? 6 : 5);
  static constexpr int SLAB_WARP = NO_SLAB ? 0 : (LSU_STORE ? SLAB_BUF : SLAB_BYTES);   // staging bytes per warp
  static constexpr int OFF_SLAB = STAGES * (A_BYTES + B_BYTES);
  static constexpr int OFF_CTRL = OFF_SLAB + NUM_EPI_WARPS * SLAB_WARP;
  struct __align__(8) Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
  };
  static constexpr int SMEM_BYTES = 1024 + OFF_CTRL + static_cast<int>(sizeof(Ctrl));
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// ---------------------------------------------------------------- staging slabs
// A buffer holds a [32 rows][128 B] box in the TMA 128-byte swizzle: 16-byte chunk c of row r
// sits at chunk position c ^ (r % 8).  Each epilogue warp owns two buffers and alternates
// between them, one per TMA store, so a store can be in flight while the next is staged.

__device__ __forceinline__ uint4* slab_chunk(uint8_t* buf, int r, int c) {
  return reinterpret_cast<uint4*>(buf + r * 128 + ((c ^ (r & 7)) << 4));
}

struct Slab {
  uint8_t* base;
  uint32_t base_s;
  uint32_t n;   // stores issued so far (warp-uniform)

  __device__ __forceinline__ uint8_t* buf() const { return base + (n & 1u) * SLAB_BUF; }
  // The buffer the k-th store from now (k = 0 or 1) will be issued from.
  __device__ __forceinline__ uint8_t* buf_ahead(int k) const { return base + ((n + k) & 1u) * SLAB_BUF; }
  // Before writing both buffers: every earlier store has finished reading its buffer.
  __device__ __forceinline__ void acquire_both(int lane) const {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }
  // Before writing the current buffer: the store issued from it two stores ago must have
  // finished reading it (the most recent store, from the other buffer, may still run).
  __device__ __forceinline__ void acquire(int lane) const {
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
  }
  // Publish the current buffer to the async proxy and store it as box (x, y) of `map`.
  __device__ __forceinline__ void store(const CUtensorMap* map, int x, int y, int lane) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, base_s + (n & 1u) * SLAB_BUF, x, y);
      bulk_commit();
    }
    ++n;
  }
  // Row `lane` of the current buffer <- 8 x 16 B.
  __device__ __forceinline__ void put_row(int lane, const uint4 (&x)[8]) const {
#pragma unroll
    for (int c = 0; c < 8; ++c) *slab_chunk(buf(), lane, c) = x[c];
  }
};

__device__ __forceinline__ uint4 pack8_bf16(const float* a) {
  return make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]), pack_bf16(a[6], a[7]));
}

__device__ __forceinline__ float sigmoid_fast(float z) { return 1.0f / (1.0f + __expf(-z)); }

struct OutMaps {
  CUtensorMap o0, o1, o2;   // EPI_QKV: q, k, v;  else: o0 = out
};

// Release an accumulator buffer to the pair's MMA thread (after this warp's last tcgen05.ld
// of it); `bar` is the leader CTA's barrier as a shared::cluster address.  The arrive is relaxed:
// the MMA thread reads nothing this warp wrote to memory, and a release would first wait for
// every global store the warp has issued (the lm_head's logits: 6% of its time).
__device__ __forceinline__ void release_acc(int lane, uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster_relaxed(bar);
}

// ---------------------------------------------------------------- tile order
// Pair tiles are walked in groups of `grp` row blocks: inside a group the row block is the
// fastest index, then the column block.  grp = 1 walks the column blocks of one row block
// together (the pairs of a wave share a row block of A); grp = num_m walks the row blocks of one
// column block together (they share a block of B); a value in between shares B among grp pairs
// and keeps the concurrently written output rows grp blocks tall.
// A negative grp walks the same order backwards (last tile first), with group size -grp.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int grp, int& mb, int& nb) {
  if (grp < 0) {
    tile = num_m * num_n - 1 - tile;
    grp = -grp;
  }
  const int per_group = grp * num_n;
  const int group = tile / per_group, local = tile % per_group;
  const int rows = min(grp, num_m - group * grp);   // the last group may be shorter
  mb = group * grp + local % rows;
  nb = local / rows;
}

// ---------------------------------------------------------------- column tiles
// Column tile nb of a launch: its first column (a row of B), its width (the MMA's N) and, for a
// value-embedding head's tile of the q|k|v projection, that kv head (else -1).  Without gate rows
// every tile is BN wide (the epilogue skips columns at or beyond `end`).  With them, the q|k
// columns are cut into BN-wide tiles (the last one narrower) and each kv head gets one tile of
// its D v rows and VGATE_ROWS gate rows.
struct ColTile {
  int col0, width, end, vhead;
};

template <int KIND>
__device__ __forceinline__ ColTile col_tile(int nb, int N, const GemmEpi& ep) {
  ColTile t;
  t.vhead = -1;
  if (KIND == EPI_QKV && ep.vgate) {
    const int qk = (ep.H + ep.Hkv) * ep.D, nqk = (qk + BN - 1) / BN;
    if (nb >= nqk) {
      t.vhead = nb - nqk;
      t.width = ep.D + VGATE_ROWS;
      t.col0 = qk + t.vhead * t.width;
      t.end = t.col0 + t.width;
      return t;
    }
    t.col0 = nb * BN;
    t.width = min(BN, qk - t.col0);
    t.end = t.col0 + t.width;
    return t;
  }
  t.col0 = nb * BN;
  t.width = BN;
  t.end = N;
  return t;
}

__host__ __device__ __forceinline__ int num_col_tiles(int kind, int N, int H, int Hkv, int D, int vgate) {
  if (kind == EPI_QKV && vgate) return ((H + Hkv) * D + BN - 1) / BN + Hkv;
  return (N + BN - 1) / BN;
}

// ---------------------------------------------------------------- per-tile prologue
// Row data an epilogue needs that does not depend on the accumulator (the RMSNorm partial sums,
// the token id).  Its loads are issued one tile ahead, while the epilogue of the previous tile
// runs, and reduced just before the tile's epilogue, so their latency is off the epilogue's
// critical path.
struct PreRaw {
  float ss[MAX_NCG];
  int tok;
  float lse;
};

struct EpiPre {
  float rs = 1.f;              // input RMSNorm row scale (8-bit: the dequantisation; EPI_QKV: of the q columns)
  float rs_k = 1.f, rs_v = 1.f;   // EPI_QKV: the same for the k and v columns (they differ on the 8-bit path)
  int tok = -1;                // EPI_QKV: token id of the row on a value-embedding head's tile, else -1;
                               // EPI_CE, EPI_CE_GRAD: the row's target
  float lse = 0.f;             // EPI_CE_GRAD: log sum exp of the row's logits
};

template <int KIND>
__device__ __forceinline__ void pre_issue(PreRaw& raw, int lane, int m0w, int M, const GemmEpi& ep,
                                          const ColTile& ct) {
  const int m = m0w + lane;
  if (m >= M) return;
  if (ep.ssp_in != nullptr) {
    const float* p = ep.ssp_in + static_cast<size_t>(m) * ep.ncg;
#pragma unroll
    for (int g = 0; g < MAX_NCG; ++g)
      if (g < ep.ncg) raw.ss[g] = p[g];
  }
  if constexpr (KIND == EPI_CE || KIND == EPI_CE_GRAD) raw.tok = ep.targets[m];
  if constexpr (KIND == EPI_CE_GRAD) raw.lse = ep.ce_lse[m];
  if constexpr (KIND == EPI_QKV) raw.tok = ct.vhead >= 0 ? ep.tokens[m] : -1;
  if constexpr (KIND == EPI_DRELU2) {   // the tile's h rows (both column halves), into L2 a tile ahead
    const bf16* hr = ep.h_in + static_cast<size_t>(m) * ep.ldo + ct.col0;
    for (int l = 0; l < 4 && ct.col0 + l * 64 < ct.end; ++l) prefetch_l2(hr + l * 64);   // ct.end = N
  }
}

template <int KIND>
__device__ __forceinline__ EpiPre pre_finish(const PreRaw& raw, int lane, int m0w, int M, const GemmEpi& ep,
                                             const ColTile& ct) {
  EpiPre p;
  const int m = m0w + lane;
  if (m >= M) return p;
  if constexpr (KIND == EPI_CE || KIND == EPI_CE_GRAD) p.tok = raw.tok;
  if constexpr (KIND == EPI_CE_GRAD) p.lse = raw.lse;
  if (ep.fp8) {   // dequantisation: the input's and the weight's 1 / scale (q, k, v ranges of the packed weight)
    const float sa = __ldg(ep.fp8_sa);
    p.rs = sa * __ldg(ep.fp8_sw);
    if constexpr (KIND == EPI_QKV) {   // q, k and v weights each have their own scale
      p.rs_k = sa * __ldg(ep.fp8_sw + 1);
      p.rs_v = sa * __ldg(ep.fp8_sw + 2);
    }
  } else {
    if (ep.ssp_in != nullptr) {
      float ss = 0.f;
#pragma unroll
      for (int g = 0; g < MAX_NCG; ++g)
        if (g < ep.ncg) ss += raw.ss[g];
      p.rs = rsqrtf(ss * ep.inv_ncols + ep.eps);
    }
    p.rs_k = p.rs_v = p.rs;
  }
  if constexpr (KIND == EPI_QKV) {
    if (ct.vhead >= 0) {
      p.tok = (raw.tok >= 0 && raw.tok < ep.V) ? raw.tok : -1;
      if (p.tok >= 0) {   // the head's slice of the token's value-embedding row, into L2
        const bf16* row = ep.ve + static_cast<size_t>(p.tok) * ep.Hkv * ep.D + static_cast<size_t>(ct.vhead) * ep.D;
        for (int l = 0; l < ep.D * 2 / 128; ++l) prefetch_l2(row + l * 64);
      }
    }
  }
  return p;
}

// ---------------------------------------------------------------- epilogues
// One warp: rows [m0w, m0w + 32) (this thread: row m0w + lane), accumulator columns
// [n0, n0 + 128) at TMEM address taddr (lane quarter applied).  Each releases the accumulator
// after its last tcgen05.ld.

// Row-coalesced stores of the staged [32 rows][128 B] box to rows m0w.. of `out` (row pitch
// ld_bytes), starting at byte column col_bytes; rows at or beyond M are skipped.  Streaming
// (evict-first) stores when `stream` is set.
__device__ __forceinline__ void lsu_store_box(const uint8_t* buf, void* out, size_t ld_bytes, int m0w, size_t col_bytes,
                                              int M, int lane, bool stream) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int row = k * 4 + (lane >> 3), q = lane & 7;
    const uint4 v = *slab_chunk(const_cast<uint8_t*>(buf), row, q);
    if (m0w + row < M) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + static_cast<size_t>(m0w + row) * ld_bytes +
                                            col_bytes + q * 16);
      if (stream) __stcs(dst, v);
      else *dst = v;
    }
  }
}

// bf16 outputs of 64-column boxes: plain (TMA store), relu(rs * acc)^2 (MLP up projection, squared
// ReLU), cap * tanh(rs * acc / cap) (the lm_head's soft-capped logits in bf16), the cross-entropy
// gradient at the lm_head's pre-cap output (EPI_CE_GRAD) or the squared ReLU's backward
// rs * acc * 2 sqrt(h) (EPI_DRELU2); all but the first are stored row-coalesced from the single
// staging buffer, the logits with streaming stores.
enum Bf16Mode { BF16_PLAIN = 0, BF16_RELU2 = 1, BF16_SOFTCAP = 2, BF16_CEGRAD = 3, BF16_DRELU2 = 4 };

template <int MODE, bool AMAX = false>
__device__ __forceinline__ void epi_bf16(uint32_t taddr, uint32_t tempty, int lane, int m0w, int n0, int M, int N,
                                         const GemmEpi& ep, const OutMaps& om, Slab& sl, const EpiPre& pre) {
  const float rs = pre.rs, rs2 = 2.f * pre.rs;
  float hmax = 0.f;   // AMAX (squared ReLU, 8-bit path): the largest value this warp stores
  const float cap = ep.cap, sc = rs / cap;
  const int m = m0w + lane;
  // EPI_CE_GRAD: exp(z - lse) = 2^(log2(e) * (cap * th - lse)); rows without a counted target
  // get scale 0.  The exponential and tanh are the approximations the cross-entropy pass used.
  float gscale = 0.f, l2e_cap = 0.f, lse_l2 = 0.f;
  if constexpr (MODE == BF16_CEGRAD) {
    const bool counted = m < M && pre.tok >= 0 && pre.tok < N;
    gscale = counted ? rs * __ldg(ep.inv_count) : 0.f;
    l2e_cap = cap * 1.4426950408889634f;
    lse_l2 = pre.lse * 1.4426950408889634f;
  }
#pragma unroll 1
  for (int ch = 0; ch < 2; ++ch) {
    const int c0 = n0 + ch * 64;
    if (c0 >= N) break;
    uint32_t r[32], r2[32];
    tmem_ld32(taddr + ch * 64, r);
    tmem_ld32(taddr + ch * 64 + 32, r2);
    uint4 hv[8];
    if constexpr (MODE == BF16_DRELU2) {
      // The forward's relu(u)^2 of the warp's 32 rows x 64 columns, read row-coalesced (each load
      // instruction covers four whole 128-byte rows), then handed to the owning lanes through the
      // staging buffer: lane l holds chunk l % 8 of rows 4 k + l / 8.
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int row = k * 4 + (lane >> 3), q = lane & 7;
        const bool in = m0w + row < M && c0 + q * 8 < N;
        hv[k] = in ? __ldg(reinterpret_cast<const uint4*>(ep.h_in + static_cast<size_t>(m0w + row) * ep.ldo + c0) + q)
                   : make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();   // every lane is done reading the previous box from the staging buffer
#pragma unroll
      for (int k = 0; k < 8; ++k) *slab_chunk(sl.buf(), k * 4 + (lane >> 3), lane & 7) = hv[k];
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 8; ++c) hv[c] = *slab_chunk(sl.buf(), lane, c);
    }
    tmem_ld_wait(r);
    tmem_ld_wait(r2);
    const int tcol = pre.tok - c0;   // EPI_CE_GRAD: the target's column within this box
    uint4 o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float a[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = c * 8 + j;
        float t = __uint_as_float(e < 32 ? r[e] : r2[e - 32]);
        if constexpr (MODE == BF16_PLAIN) {
          t = t * rs;   // 1 without a row scale; the 8-bit path's dequantisation
        } else if constexpr (MODE == BF16_RELU2) {
          t = fmaxf(t * rs, 0.f);
          t = t * t;
          if constexpr (AMAX) hmax = fmaxf(hmax, t);   // rows and columns past the ends are 0
        } else if constexpr (MODE == BF16_SOFTCAP) {
          t = cap * tanh_approx(t * sc);
        } else if constexpr (MODE == BF16_CEGRAD) {
          const float th = tanh_approx(t * sc);
          const float p = ex2_approx(fmaf(th, l2e_cap, -lse_l2));
          t = (p - (e == tcol ? 1.f : 0.f)) * fmaf(-th, th, 1.f) * gscale;
        } else if constexpr (MODE == BF16_DRELU2) {
          const __nv_bfloat162 h2 = reinterpret_cast<const __nv_bfloat162*>(&hv[c])[j >> 1];
          const float hval = (j & 1) ? __high2float(h2) : __low2float(h2);
          t = t * rs2 * sqrt_approx(hval);
        }
        a[j] = t;
      }
      o[c] = pack8_bf16(a);
    }
    if constexpr (MODE != BF16_PLAIN) {
      constexpr bool stream = MODE == BF16_SOFTCAP;
      __syncwarp();   // every lane is done reading the previous box
      sl.put_row(lane, o);
      __syncwarp();
      if (c0 + 64 <= N) {
        lsu_store_box(sl.buf(), ep.out, static_cast<size_t>(ep.ldo) * 2, m0w, static_cast<size_t>(c0) * 2, M, lane,
                      stream);
      } else {   // ragged last box: 32 valid columns (N % 32 == 0)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int row = k * 4 + (lane >> 3), q = lane & 7;
          const uint4 v = *slab_chunk(sl.buf(), row, q);
          if (m0w + row < M && c0 + q * 8 < N)
            *reinterpret_cast<uint4*>(static_cast<bf16*>(ep.out) + static_cast<size_t>(m0w + row) * ep.ldo + c0 + q * 8) = v;
        }
      }
    } else {
      sl.acquire(lane);
      sl.put_row(lane, o);
      sl.store(&om.o0, c0, m0w, lane);
    }
  }
  release_acc(lane, tempty);
  if constexpr (AMAX) {   // bf16 rounding keeps the order: the rounded maximum is the maximum stored
    hmax = warp_max(hmax);
    if (lane == 0 && ep.amax_out != nullptr)
      atomicMax(reinterpret_cast<unsigned int*>(ep.amax_out), __float_as_uint(__bfloat162float(__float2bfloat16(hmax))));
  }
}

// fp32 outputs: cap * tanh(rs * acc / cap) (logit soft-cap of the lm_head, streaming stores) or
// rs * acc (EPI_F32: the backward's weight and input gradients).  The accumulator is read in the
// 16x256b shape, in which four consecutive threads hold 8 consecutive columns of one row, so
// each 8-byte store instruction writes whole 32-byte sectors (8 rows x 32 B) straight from the
// registers: no staging through shared memory, whose bytes go to a deeper operand ring instead.
template <bool SOFTCAP>
__device__ __forceinline__ void epi_f32out(uint32_t taddr, uint32_t tempty, int lane, int m0w, int n0, int M,
                                           int N, const GemmEpi& ep, const EpiPre& pre, void* out) {
  const float cap = ep.cap;
  const int rq = lane >> 2, cq = lane & 3;
  // the row scales of this thread's four rows m0w + 16 h + 8 e + lane / 4 (lane l holds row m0w + l's)
  float sc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float r = __shfl_sync(0xffffffffu, pre.rs, (i >> 1) * 16 + (i & 1) * 8 + rq);
    sc[i] = SOFTCAP ? r / cap : r;
  }
  uint8_t* const obase = static_cast<uint8_t*>(out);
  const size_t ld_bytes = static_cast<size_t>(ep.ldo) * 4;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    const int c0 = n0 + ch * 32;
    if (c0 >= N) break;
    uint32_t r[2][16];
    tmem_ld16x256_x4(taddr + ch * 32, r[0]);               // lanes 0..15 of the warp's quarter
    tmem_ld16x256_x4(taddr + (16u << 16) + ch * 32, r[1]);   // lanes 16..31
    tmem_ld_wait(r[0]);
    tmem_ld_wait(r[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = m0w + h * 16 + e * 8 + rq;
        if (row >= M) continue;
        uint8_t* const orow = obase + static_cast<size_t>(row) * ld_bytes;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v0 = __uint_as_float(r[h][4 * j + 2 * e]) * sc[2 * h + e];
          float v1 = __uint_as_float(r[h][4 * j + 2 * e + 1]) * sc[2 * h + e];
          if (SOFTCAP) {
            v0 = cap * tanh_approx(v0);
            v1 = cap * tanh_approx(v1);
          }
          float2* dst = reinterpret_cast<float2*>(orow + static_cast<size_t>(c0 + 8 * j + 2 * cq) * 4);
          if (SOFTCAP) __stcs(dst, make_float2(v0, v1));   // written once, never re-read
          else *dst = make_float2(v0, v1);
        }
      }
    }
  }
  release_acc(lane, tempty);
}

// Cross-entropy partials of the soft-capped lm_head, with no logits stored: per row, the sum
// of exp(z) over the warp's 128 columns, z = cap * tanh(rs * acc / cap), and z at the row's
// target column when the target lies in them.  |z| < cap bounds every term by e^cap, so the sum
// needs no running maximum (cap = 15: under 2^22 per column, far inside fp32 for any vocabulary
// this kernel can address).  The target's z is the same rounded value that entered the sum.
__device__ __forceinline__ void epi_ce(uint32_t taddr, uint32_t tempty, int lane, int m0w, int n0, int M, int N,
                                       const GemmEpi& ep, const EpiPre& pre) {
  const float cap = ep.cap;
  const float sc = pre.rs / cap;
  const float l2e_cap = cap * 1.4426950408889634f;   // exp(cap * t) = 2^(log2(e) * cap * t)
  const int tcol = pre.tok - n0;                      // the target's column among the warp's 128
  float s0 = 0.f, s1 = 0.f, zt = 0.f;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    const int c0 = n0 + ch * 32;
    if (c0 >= N) break;
    uint32_t r[32];
    tmem_ld32(taddr + ch * 32, r);
    tmem_ld_wait(r);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      s0 += ex2_approx(tanh_approx(__uint_as_float(r[j]) * sc) * l2e_cap);
      s1 += ex2_approx(tanh_approx(__uint_as_float(r[j + 1]) * sc) * l2e_cap);
    }
    const int tj = tcol - ch * 32;
    if (static_cast<unsigned>(tj) < 32u) {   // rare: this chunk holds the row's target
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) a = j == tj ? __uint_as_float(r[j]) : a;
      zt = cap * tanh_approx(a * sc);
    }
  }
  release_acc(lane, tempty);
  const int m = m0w + lane;
  if (m < M && n0 < N) {
    ep.ce_part[static_cast<size_t>(n0 / 128) * M + m] = s0 + s1;
    if (tcol >= 0 && tcol < 128 && pre.tok < N) ep.ce_zt[m] = zt;
  }
}

// Packed q|k|v projection: q and k heads are rotated (RoPE) and RMS-normalised per head; v heads
// (of a layer without value embeddings) are stored as they are.  rs (the block's input RMSNorm)
// scales every column; for q and k the head norm is taken from the unrotated accumulator, since
// the rotation keeps each head's norm.  Columns at or beyond `end` belong to no output.
template <int D>
__device__ __forceinline__ void epi_qkv(uint32_t taddr, uint32_t tempty, int lane, int m0w, int n0, int end, int M,
                                        const GemmEpi& ep, const OutMaps& om, Slab& sl, const EpiPre& pre) {
  const int m = m0w + lane;
  const int qcols = ep.H * D, kcols = ep.Hkv * D;
  const int pos = m < M ? m % ep.T : 0;
  // A head is D/64 boxes of [32 rows][64 columns] bf16: results go straight into the staging
  // buffers (box b in the buffer of the b-th store from now), then the boxes are stored.
#pragma unroll
  for (int s = 0; s < 128 / D; ++s) {
    const int c = n0 + s * D;
    if (c >= end) break;
    const uint32_t tb = taddr + s * D;
    const CUtensorMap* map;
    int xcol;
    // the head's scale: the input RMSNorm, or on the 8-bit path the q, k or v weight's dequantisation
    const float rs = c < qcols ? pre.rs : (c < qcols + kcols ? pre.rs_k : pre.rs_v);
    sl.acquire_both(lane);
    if (c < qcols + kcols) {
      if (c < qcols) {
        map = &om.o0;
        xcol = c;
      } else {
        map = &om.o1;
        xcol = c - qcols;
      }
      // the rotation table rows do not depend on the accumulator: load them first
      const float2* rope = ep.rope + pos;
      float2 cs[D / 2];
#pragma unroll
      for (int j = 0; j < D / 2; ++j) cs[j] = __ldg(rope + static_cast<size_t>(j) * ep.rope_ld);
      float ss = 0.f;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tb + ch * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) ss = fmaf(__uint_as_float(r[j]), __uint_as_float(r[j]), ss);
      }
      const float sc = rs * rsqrtf(rs * rs * ss * (1.0f / D) + ep.eps);
#pragma unroll
      for (int hc = 0; hc < D / 64; ++hc) {
        uint32_t lo[32], hi[32];
        tmem_ld32(tb + hc * 32, lo);
        tmem_ld32(tb + D / 2 + hc * 32, hi);
        tmem_ld_wait(lo);
        tmem_ld_wait(hi);
#pragma unroll
        for (int j8 = 0; j8 < 32; j8 += 8) {
          uint32_t py[4], pz[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int j = j8 + 2 * t;
            const float2 c0 = cs[hc * 32 + j], c1 = cs[hc * 32 + j + 1];
            const float a0 = __uint_as_float(lo[j]), b0 = __uint_as_float(hi[j]);
            const float a1 = __uint_as_float(lo[j + 1]), b1 = __uint_as_float(hi[j + 1]);
            py[t] = pack_bf16((a0 * c0.x + b0 * c0.y) * sc, (a1 * c1.x + b1 * c1.y) * sc);
            pz[t] = pack_bf16((b0 * c0.x - a0 * c0.y) * sc, (b1 * c1.x - a1 * c1.y) * sc);
          }
          const int cy = hc * 32 + j8, cz = D / 2 + hc * 32 + j8;   // head columns
          *slab_chunk(sl.buf_ahead(cy / 64), lane, (cy % 64) / 8) = make_uint4(py[0], py[1], py[2], py[3]);
          *slab_chunk(sl.buf_ahead(cz / 64), lane, (cz % 64) / 8) = make_uint4(pz[0], pz[1], pz[2], pz[3]);
        }
      }
    } else {
      xcol = c - qcols - kcols;
      map = &om.o2;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tb + cc * 64, r0);
        tmem_ld32(tb + cc * 64 + 32, r1);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t pv[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int idx = c8 * 8 + 2 * t;
            const float v0 = __uint_as_float(idx < 32 ? r0[idx] : r1[idx - 32]);
            const float v1 = __uint_as_float(idx + 1 < 32 ? r0[idx + 1] : r1[idx + 1 - 32]);
            pv[t] = pack_bf16(v0 * rs, v1 * rs);
          }
          *slab_chunk(sl.buf_ahead(cc), lane, c8) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
        }
      }
    }
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) sl.store(map, xcol + cc * 64, m0w, lane);
  }
  release_acc(lane, tempty);
}

// A value-embedding head's tile of the packed q|k|v projection: accumulator columns [0, D) are the
// head's v, column D the gate's pre-activation x . w_gate (columns D+1.. are zero rows).
//   v = rs * acc + gate * ve[token, head],  gate = gate_scale * sigmoid(rs * acc[D])
// With D = 128 the two warpgroups take 64 columns each; with D = 64 the first takes the head.
template <int D>
__device__ __forceinline__ void epi_vgate(uint32_t taddr, uint32_t tempty, int lane, int m0w, int M, int group,
                                          int vhead, const GemmEpi& ep, const OutMaps& om, Slab& sl,
                                          const EpiPre& pre) {
  const int c0 = D == 128 ? group * 64 : 0;
  if (D == 64 && group == 1) {
    release_acc(lane, tempty);
    return;
  }
  const float rs = pre.rs_v;
  uint32_t gz[1];
  tmem_ld1(taddr + D, gz);
  // the 8-bit path: the gate's pre-activation (already row-scaled) from its own bf16 product
  const int m = m0w + lane;
  const float gpre = (ep.gpre != nullptr && m < M) ? ep.gpre[static_cast<size_t>(m) * ep.gpre_ld + vhead] : 0.f;
  uint32_t r0[32], r1[32];
  tmem_ld32(taddr + c0, r0);
  tmem_ld32(taddr + c0 + 32, r1);
  uint4 e[8];
  const uint4* vr = pre.tok >= 0 ? reinterpret_cast<const uint4*>(ep.ve + static_cast<size_t>(pre.tok) * ep.Hkv * D +
                                                                  static_cast<size_t>(vhead) * D + c0)
                                 : nullptr;
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) e[c8] = vr ? __ldg(vr + c8) : make_uint4(0u, 0u, 0u, 0u);
  tmem_ld_wait(gz);
  tmem_ld_wait(r0);
  tmem_ld_wait(r1);
  release_acc(lane, tempty);
  const float g = ep.gate_scale * sigmoid_fast(ep.gpre != nullptr ? gpre : rs * __uint_as_float(gz[0]));
  sl.acquire(lane);
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&e[c8]);
    uint32_t pv[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int idx = c8 * 8 + 2 * t;
      const float2 f = __bfloat1622float2(h2[t]);
      const float v0 = __uint_as_float(idx < 32 ? r0[idx] : r1[idx - 32]);
      const float v1 = __uint_as_float(idx + 1 < 32 ? r0[idx + 1] : r1[idx + 1 - 32]);
      pv[t] = pack_bf16(fmaf(g, f.x, v0 * rs), fmaf(g, f.y, v1 * rs));
    }
    *slab_chunk(sl.buf(), lane, c8) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
  }
  sl.store(&om.o2, vhead * D + c0, m0w, lane);
}

template <int KIND, int D, bool F8>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBv, const __grid_constant__ OutMaps om, int M, int N, int K,
                   int grp, const __grid_constant__ GemmEpi ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using L = Cfg<KIND, D>;
  constexpr int STAGES = L::STAGES;
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;
  typename L::Ctrl* ctl = reinterpret_cast<typename L::Ctrl*>(smem + L::OFF_CTRL);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();            // 0: pair leader (issues the MMAs)
  const int pair = static_cast<int>(blockIdx.x) >> 1, npairs = static_cast<int>(gridDim.x) >> 1;
  const int num_m = (M + PAIR_M - 1) / PAIR_M, num_n = num_col_tiles(KIND, N, ep.H, ep.Hkv, ep.D, ep.vgate);
  // a stage holds 128 bytes of K per row: 64 bf16 or 128 e4m3 elements; a ragged last k-block is zero-filled
  constexpr int kstep = F8 ? 2 * BK : BK;   // F8: e4m3 operands (the bf16 instantiations are unchanged)
  const int kblocks = (K + kstep - 1) / kstep;
  // split over K (EPI_F32): tile = s * out_tiles + output tile, k-blocks [s * kps, (s + 1) * kps)
  const int out_tiles = num_m * num_n, ksplit = ep.ksplit > 1 ? ep.ksplit : 1;
  const int num_tiles = out_tiles * ksplit, kps = (kblocks + ksplit - 1) / ksplit;
  const bool a_mn = ep.a_mn != 0, b_mn = ep.b_mn != 0;
  int* status = ep.status;
  const uint64_t wlim = ep.wait_ns;

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
    if (KIND == EPI_QKV && ep.vgate) tma_prefetch_desc(&tmBv);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  griddep_wait();     // the previous kernel's outputs are complete and visible
  griddep_launch();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp < EPI_WARP0) {
    regs_dec<REGS_CTRL>();
    if (warp == 0 && lane == 0) {
      // The operand shared by the pairs running at the same time is read once per wave; the
      // other one is re-read for every tile of the walk and should stay in L2.
      const bool share_a = grp == 1 || grp == -1;
      const uint64_t pol_a = share_a ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_b = share_a ? policy_evict_last() : policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        int mb, nb;
        tile_coords(tile % out_tiles, num_m, num_n, grp, mb, nb);
        const int kb0 = (tile / out_tiles) * kps, kb1 = min(kblocks, kb0 + kps);
        const ColTile ct = col_tile<KIND>(nb, N, ep);
        // a value-embedding head's tile loads its D + VGATE_ROWS rows of B through the map whose box
        // is half of that; every other tile loads BN / 2 rows per CTA (the MMA uses width / 2)
        const bool vt = ct.vhead >= 0;
        const uint32_t b_bytes = vt ? static_cast<uint32_t>(ct.width / 2) * BK * 2 : static_cast<uint32_t>(B_BYTES);
        for (int kb = kb0; kb < kb1; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&ctl->empty[s]), ph ^ 1, abort, status, wlim)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(smem_u32(&ctl->full[s]), 0);   // the leader's barrier
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), 2 * (A_BYTES + b_bytes));
          const int a_row = mb * PAIR_M + static_cast<int>(rank) * BM;
          const int b_row = ct.col0 + static_cast<int>(rank) * (ct.width / 2);
          // K-contiguous: one box [rows][64 k].  MN-contiguous: two boxes [64 k][64 rows], the
          // second (rows 64..127) MN_BLOCK bytes after the first.
          if (!a_mn) {
            tma_load_2d_pair_hint(sA + s * A_BYTES, &tmA, fb, kb * kstep, a_row, pol_a);
          } else {
            tma_load_2d_pair_hint(sA + s * A_BYTES, &tmA, fb, a_row, kb * BK, pol_a);
            tma_load_2d_pair_hint(sA + s * A_BYTES + MN_BLOCK, &tmA, fb, a_row + 64, kb * BK, pol_a);
          }
          if (!b_mn) {
            tma_load_2d_pair_hint(sB + s * B_BYTES, vt ? &tmBv : &tmB, fb, kb * kstep, b_row, pol_b);
          } else {
            tma_load_2d_pair_hint(sB + s * B_BYTES, &tmB, fb, b_row, kb * BK, pol_b);
            tma_load_2d_pair_hint(sB + s * B_BYTES + MN_BLOCK, &tmB, fb, b_row + 64, kb * BK, pol_b);
          }
          ++it;
        }
      }
      // The leader's full barriers count both CTAs' copies: once its last phases completed,
      // every copy issued by the pair has landed (the peer exits only after the final sync).
      if (rank == 0) {
        for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_cluster(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1, nullptr, status, wlim);
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs, ++tc) {
        int mb, nb;
        tile_coords(tile % out_tiles, num_m, num_n, grp, mb, nb);
        const int kb0 = (tile / out_tiles) * kps, kb1 = min(kblocks, kb0 + kps);
        const int width = col_tile<KIND>(nb, N, ep).width;
        const uint32_t idesc = F8 ? idesc_e4m3_f32(PAIR_M, width)
                                  : idesc_bf16_f32(PAIR_M, width) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
        const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
        if (!mbar_wait_cluster(smem_u32(&ctl->tempty[a]), aph ^ 1, abort, status, wlim)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&ctl->full[s]), ph, abort, status, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // a k-step of 16: 32 B along a K-contiguous row, or 16 rows of 128 B of an MN-contiguous box
            const uint64_t ad = a_mn ? sdesc_mnmajor_sw128(sA + s * A_BYTES + kk * 16 * 128, MN_BLOCK)
                                     : sdesc_kmajor_sw128(sA + s * A_BYTES + kk * 32);
            const uint64_t bd = b_mn ? sdesc_mnmajor_sw128(sB + s * B_BYTES + kk * 16 * 128, MN_BLOCK)
                                     : sdesc_kmajor_sw128(sB + s * B_BYTES + kk * 32);
            if constexpr (F8) umma_f8_pair(d_tmem, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
            else umma_bf16_pair(d_tmem, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&ctl->empty[s]), 0x3);
          ++it;
        }
        if (!ok) break;
        if (tile != ep.test_skip_tile) umma_commit_pair(smem_u32(&ctl->tfull[a]), 0x3);
      }
      umma_commit_pair(smem_u32(&ctl->drain), 0x1);
      mbar_wait(smem_u32(&ctl->drain), 0, nullptr, status, wlim);
    }
    __syncwarp();
  } else {
    regs_inc<REGS_EPI>();
    const int ew = warp - EPI_WARP0;
    const int quarter = warp & 3;   // TMEM lanes 32*(warp % 4) .. +31 are this warp's
    const int group = ew >> 2;
    Slab sl{smem + L::OFF_SLAB + ew * L::SLAB_WARP, smem_u32(smem + L::OFF_SLAB + ew * L::SLAB_WARP), 0u};
    auto coords = [&](int tile, int& m0w, ColTile& ct) {
      int mb, nb;
      tile_coords(tile % out_tiles, num_m, num_n, grp, mb, nb);
      m0w = mb * PAIR_M + static_cast<int>(rank) * BM + quarter * 32;
      ct = col_tile<KIND>(nb, N, ep);
    };
    PreRaw raw;
    raw.tok = -1;
    if (pair < num_tiles) {
      int m0w;
      ColTile ct;
      coords(pair, m0w, ct);
      pre_issue<KIND>(raw, lane, m0w, M, ep, ct);
    }
    uint32_t tc = 0;
    for (int tile = pair; tile < num_tiles; tile += npairs, ++tc) {
      const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
      int m0w;
      ColTile ct;
      coords(tile, m0w, ct);
      const int n0 = ct.col0 + group * 128;
      const EpiPre pre = pre_finish<KIND>(raw, lane, m0w, M, ep, ct);
      const bool ok = mbar_wait_cluster(smem_u32(&ctl->tfull[a]), aph, abort, status, wlim);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      if (tile + npairs < num_tiles) {   // the next tile's row data is in flight during this epilogue
        int m1;
        ColTile c1;
        coords(tile + npairs, m1, c1);
        pre_issue<KIND>(raw, lane, m1, M, ep, c1);
      }
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * BN;
      const uint32_t taddr = tbase + group * 128;
      const uint32_t tempty = mapa_shared(smem_u32(&ctl->tempty[a]), 0);
      if constexpr (KIND == EPI_SOFTCAP_F32) epi_f32out<true>(taddr, tempty, lane, m0w, n0, M, N, ep, pre, ep.out);
      else if constexpr (KIND == EPI_F32)   // a split tile writes its K range's slab
        epi_f32out<false>(taddr, tempty, lane, m0w, n0, M, N, ep, pre,
                          ksplit > 1 ? ep.split_ws + static_cast<size_t>(tile / out_tiles) * M * ep.ldo : ep.out);
      else if constexpr (KIND == EPI_CE_GRAD) epi_bf16<BF16_CEGRAD>(taddr, tempty, lane, m0w, n0, M, N, ep, om, sl, pre);
      else if constexpr (KIND == EPI_DRELU2) epi_bf16<BF16_DRELU2>(taddr, tempty, lane, m0w, n0, M, N, ep, om, sl, pre);
      else if constexpr (KIND == EPI_CE) epi_ce(taddr, tempty, lane, m0w, n0, M, N, ep, pre);
      else if constexpr (KIND == EPI_QKV) {
        if (ct.vhead >= 0) epi_vgate<D>(tbase, tempty, lane, m0w, M, group, ct.vhead, ep, om, sl, pre);
        else epi_qkv<D>(taddr, tempty, lane, m0w, n0, ct.end, M, ep, om, sl, pre);
      } else if constexpr (KIND == EPI_SOFTCAP_BF16) {
        epi_bf16<BF16_SOFTCAP>(taddr, tempty, lane, m0w, n0, M, N, ep, om, sl, pre);
      } else {
        epi_bf16<KIND == EPI_RELU2_BF16 ? BF16_RELU2 : BF16_PLAIN, F8 && KIND == EPI_RELU2_BF16>(
            taddr, tempty, lane, m0w, n0, M, N, ep, om, sl, pre);
      }
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

template <int KIND, int D, bool F8 = false>
cudaError_t launch_kind(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbv, const OutMaps& om,
                        int M, int N, int K, const GemmEpi& epi, int num_sms, cudaStream_t stream) {
  struct State {
    int max_pairs = 0;
  };
  static State states[MAX_DEVICES];
  static bool ready[MAX_DEVICES];
  static std::mutex mu;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg<KIND, D>::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // occupancy query without the PDL attribute
  State* st = nullptr;
  const cudaError_t init_err = per_device(states, ready, mu, [&](State& s) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<KIND, D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<KIND, D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * (num_sms / 2));
    if (cudaOccupancyMaxActiveClusters(&s.max_pairs, gemm_tc_kernel<KIND, D, F8>, &q) != cudaSuccess || s.max_pairs < 1) {
      cudaGetLastError();
      s.max_pairs = num_sms / 2;
    }
    return cudaSuccess;
  }, &st);
  if (init_err != cudaSuccess) return init_err;
  const int max_pairs = st->max_pairs;
  const int num_m = (M + PAIR_M - 1) / PAIR_M;
  const int tiles = num_m * num_col_tiles(KIND, N, epi.H, epi.Hkv, epi.D, epi.vgate) * (epi.ksplit > 1 ? epi.ksplit : 1);
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  cfg.gridDim = dim3(2 * pairs);
  // When A is the larger operand the pairs of a wave share its row block (grp = 1); otherwise
  // (the lm_head) they share a block of B (grp = every row block: on the d12 lm_head this beats
  // groups of 8 row blocks, whose B tiles are re-read 8 times as often).
  const int grp = M >= N ? 1 : num_m;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<KIND, D, F8>, ta, tb, tbv, om, M, N, K, grp, epi);
  if (e != cudaSuccess) cudaGetLastError();   // a failed launch must not resurface in a later call
  return e;
}

// out[m, c] = sum over s = 0, 1, ... of ws[s][m, c]: the K ranges of a split product, added in a
// fixed order (4 columns per thread, 128-bit loads and stores).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ ws, int S, size_t slab, int M,
                                                            int N, int ldo, float* __restrict__ out) {
  griddep_wait();   // the partial slabs are complete and visible
  griddep_launch();
  const int q = N / 4;
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(M) * q) return;
  const size_t off = (i / q) * static_cast<size_t>(ldo) + (i % q) * 4;
  float4 acc = *reinterpret_cast<const float4*>(ws + off);
  for (int s = 1; s < S; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(ws + static_cast<size_t>(s) * slab + off);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  *reinterpret_cast<float4*>(out + off) = acc;
}

cudaError_t launch_splitk_reduce(const GemmEpi& e, int M, int N, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  const size_t n = static_cast<size_t>(M) * (N / 4);
  cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, static_cast<const float*>(e.split_ws), e.ksplit,
                                             static_cast<size_t>(M) * e.ldo, M, N, e.ldo, static_cast<float*>(e.out));
  if (err != cudaSuccess) cudaGetLastError();
  return err;
}

}  // namespace

int gemm_ksplit(int M, int N, int K, int num_sms) {
  if (M < 1 || N < 1 || K < 1) return 1;
  const int tiles = ((M + PAIR_M - 1) / PAIR_M) * ((N + BN - 1) / BN);
  const int pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
  const int kblocks = (K + BK - 1) / BK;
  if (2 * tiles >= pairs) return 1;
  int s = pairs / tiles;
  s = s < kblocks ? s : kblocks;
  s = s < 16 ? s : 16;
  if (s < 2) return 1;
  const int kps = (kblocks + s - 1) / s;   // every range non-empty
  return (kblocks + kps - 1) / kps;
}

size_t gemm_split_ws_bytes(int M, int N, int K, int ldo, int num_sms) {
  const int s = gemm_ksplit(M, N, K, num_sms);
  return s > 1 ? static_cast<size_t>(s) * M * ldo * sizeof(float) : 0;
}

cudaError_t launch_gemm(const bf16* A, const bf16* B, int M, int N, int K, const GemmEpi& epi_in,
                        int num_sms, cudaStream_t stream) {
  GemmEpi epi = epi_in;
  epi.ksplit = 1;
  if (epi.kind == EPI_F32 && epi.split_ws != nullptr) {
    epi.ksplit = gemm_ksplit(M, N, K, num_sms);
    if (epi.ksplit > 1 && reinterpret_cast<uintptr_t>(epi.split_ws) % 16 != 0) return cudaErrorInvalidValue;
  }
  const bool vgate = epi.kind == EPI_QKV && epi.vgate;
  const bool a_mn = epi.a_mn != 0, b_mn = epi.b_mn != 0;
  if (M <= 0 || N <= 0 || K <= 0 || N % (vgate ? 16 : 32) != 0) return cudaErrorInvalidValue;
  if ((epi.a_mn != 0 && epi.a_mn != 1) || (epi.b_mn != 0 && epi.b_mn != 1)) return cudaErrorInvalidValue;
  // rows of a stored operand are 16-byte multiples (TMA strides); the q|k|v layout is K-contiguous
  if ((!a_mn || !b_mn) && K % 8 != 0) return cudaErrorInvalidValue;
  if ((a_mn && M % 8 != 0) || (b_mn && N % 8 != 0) || (epi.kind == EPI_QKV && (a_mn || b_mn)))
    return cudaErrorInvalidValue;
  const uint64_t Ku = static_cast<uint64_t>(K);
  const bool f8 = epi.fp8 != 0;
  // 8-bit operands: K-contiguous only, rows of K bytes (16-byte multiples), the dequantisation
  // scales given, and no epilogue of the backward
  if (f8 && (a_mn || b_mn || K % 16 != 0 || epi.fp8_sa == nullptr || epi.fp8_sw == nullptr ||
             epi.kind == EPI_CE_GRAD || epi.kind == EPI_DRELU2))
    return cudaErrorInvalidValue;
  CUtensorMap ta, tb, tbv;
  bool ok_a, ok_b;
  if (f8) {   // one 128-byte row of a stage = 128 e4m3 elements of K
    ok_a = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, Ku, M, Ku, 2 * BK, BM);
    ok_b = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, Ku, N, Ku, 2 * BK, B_ROWS);
  } else {
    ok_a = a_mn ? make_tmap_bf16_2d(&ta, A, M, Ku, static_cast<uint64_t>(M) * 2, 64, BK)
                : make_tmap_bf16_2d(&ta, A, Ku, M, Ku * 2, BK, BM);
    ok_b = b_mn ? make_tmap_bf16_2d(&tb, B, N, Ku, static_cast<uint64_t>(N) * 2, 64, BK)
                : make_tmap_bf16_2d(&tb, B, Ku, N, Ku * 2, BK, B_ROWS);
  }
  if (!ok_a || !ok_b) return cudaErrorInvalidValue;
  tbv = tb;
  OutMaps om;
  const uint64_t Mu = static_cast<uint64_t>(M);
  bool ok = true;
  switch (epi.kind) {
    case EPI_CE:
      ok = epi.targets != nullptr && epi.ce_part != nullptr && epi.ce_zt != nullptr && epi.cap > 0.f;
      break;
    case EPI_SOFTCAP_F32:   // written with plain 8-byte stores from the registers (16-byte aligned rows)
    case EPI_F32:
      ok = (reinterpret_cast<uintptr_t>(epi.out) % 16 == 0) && epi.ldo % 4 == 0 && epi.ldo >= N;
      break;
    case EPI_CE_GRAD:
      ok = epi.targets != nullptr && epi.ce_lse != nullptr && epi.inv_count != nullptr && epi.cap > 0.f &&
           (reinterpret_cast<uintptr_t>(epi.out) % 16 == 0) && epi.ldo % 8 == 0 && epi.ldo >= N;
      break;
    case EPI_DRELU2:
      ok = epi.h_in != nullptr && (reinterpret_cast<uintptr_t>(epi.h_in) % 16 == 0) &&
           (reinterpret_cast<uintptr_t>(epi.out) % 16 == 0) && epi.ldo % 8 == 0 && epi.ldo >= N;
      break;
    case EPI_BF16:
      ok = make_tmap_bf16_2d(&om.o0, epi.out, N, Mu, static_cast<uint64_t>(epi.ldo) * 2, 64, 32);
      break;
    case EPI_RELU2_BF16:   // row-coalesced plain stores (16-byte aligned rows)
    case EPI_SOFTCAP_BF16:
      ok = (reinterpret_cast<uintptr_t>(epi.out) % 16 == 0) && epi.ldo % 8 == 0 &&
           (epi.kind != EPI_SOFTCAP_BF16 || epi.cap > 0.f);
      break;
    case EPI_QKV: {
      const uint64_t qc = static_cast<uint64_t>(epi.H) * epi.D, kc = static_cast<uint64_t>(epi.Hkv) * epi.D;
      if (epi.rope == nullptr || epi.rope_ld < 1 || (epi.D != 64 && epi.D != 128)) return cudaErrorInvalidValue;
      if (vgate && (epi.ve == nullptr || epi.tokens == nullptr ||
                    N != static_cast<int>(qc + kc) + epi.Hkv * (epi.D + VGATE_ROWS)))
        return cudaErrorInvalidValue;
      if (!vgate && N != static_cast<int>(qc + 2 * kc)) return cudaErrorInvalidValue;
      ok = make_tmap_bf16_2d(&om.o0, epi.q, qc, Mu, qc * 2, 64, 32) &&
           make_tmap_bf16_2d(&om.o1, epi.k, kc, Mu, kc * 2, 64, 32) &&
           make_tmap_bf16_2d(&om.o2, epi.v, kc, Mu, kc * 2, 64, 32);
      // a value-embedding head's tile: D + VGATE_ROWS rows of B, half per CTA
      if (ok && vgate)
        ok = f8 ? make_tmap_2d(&tbv, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, Ku, N, Ku, 2 * BK, (epi.D + VGATE_ROWS) / 2)
                : make_tmap_bf16_2d(&tbv, B, K, N, static_cast<uint64_t>(K) * 2, BK, (epi.D + VGATE_ROWS) / 2);
      break;
    }
    default: return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  switch (epi.kind) {
#define NC_KIND(K_, D_)                                                                      \
  (f8 ? launch_kind<K_, D_, true>(ta, tb, tbv, om, M, N, K, epi, num_sms, stream)            \
      : launch_kind<K_, D_, false>(ta, tb, tbv, om, M, N, K, epi, num_sms, stream))
    case EPI_BF16: return NC_KIND(EPI_BF16, 0);
    case EPI_RELU2_BF16: return NC_KIND(EPI_RELU2_BF16, 0);
    case EPI_SOFTCAP_F32: return NC_KIND(EPI_SOFTCAP_F32, 0);
    case EPI_SOFTCAP_BF16: return NC_KIND(EPI_SOFTCAP_BF16, 0);
    case EPI_CE: return NC_KIND(EPI_CE, 0);
    case EPI_F32: {
      const cudaError_t e = NC_KIND(EPI_F32, 0);
      if (e != cudaSuccess || epi.ksplit < 2) return e;
      return launch_splitk_reduce(epi, M, N, stream);
    }
    case EPI_CE_GRAD: return launch_kind<EPI_CE_GRAD, 0>(ta, tb, tbv, om, M, N, K, epi, num_sms, stream);
    case EPI_DRELU2: return launch_kind<EPI_DRELU2, 0>(ta, tb, tbv, om, M, N, K, epi, num_sms, stream);
    case EPI_QKV:
      if (epi.D == 128) return NC_KIND(EPI_QKV, 128);
      return NC_KIND(EPI_QKV, 64);
#undef NC_KIND
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nc
