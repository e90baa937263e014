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
// Persistent CTAs, one per SM, walk work items: a pair of 128-query tiles of one (head, batch
// row), heaviest pairs first, in serpentine order across the grid.
// Key tiles are 128 keys wide, so every tensor-core step is a full-rate 128 x 128 (x 16) or
// 128 x D (x 16) MMA.  The two query tiles (Q0: rows q0..q0+127, Q1: the next 128 rows) walk
// the same key tiles; a query tile skips the key tiles it does not see.
//   tensor memory (512 columns): S_k for query tile k at columns 128k (fp32 scores); softmax k
//               overwrites the first 64 of them with P_k (bf16, two per column), which the
//               P V step reads as its A operand straight from tensor memory; O_k at 256 + k*D.
//   warp 0      TMA: Q0 and Q1 once per item (and an L2 prefetch of the next item's, so that its
//               load at the item transition hits L2), then the key tiles (128 keys) into a ring
//               (2 stages at D = 128, 3 at D = 64).
//   warp 2      TMA: the value tiles into a 3-stage ring of their own.
//   warp 1      TMEM allocation; one lane issues, for each key tile j:
//                 O_0 += P_0(j) V(j), S_0(j+1) = Q_0 K(j+1)^T, O_1 += P_1(j) V(j), S_1(j+1) ...
//               so that while softmax 0 works on its scores the tensor core runs query tile 1's
//               steps and the other way round.  Tensor-core operations issued by one thread run
//               in issue order, so S_k(j+1) overwrites P_k(j) only after O_k += P_k(j) V(j) has
//               read it, and the completion of S_k(j+1) also tells softmax k that O_k is stable.
//   warps 4..7  softmax of Q0, warps 8..11 softmax of Q1, one thread per query row: load the
//               128 scores of its row, mask only on key tiles that cross the diagonal, the
//               window edge or the sequence end, online softmax in base 2 (scale folded into one
//               FMA, hardware exp2; maxima, scaling and sums on packed two-lane fp32
//               instructions), P to tensor memory in two halves of 64 keys (the P V step
//               of the first half starts while the second is computed).  The running max moves
//               only when a row's max grows by more than 2^8; only then is that row of O
//               rescaled.
//               Final: O / l -> bf16 -> y.
//   warp 3      idle.
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace nc {
namespace {

constexpr int BQ = 128, BKV = 128;
constexpr int SM_WARP0 = 4;                    // softmax warps 4..11
constexpr int THREADS = 32 * (SM_WARP0 + 8);
constexpr uint32_t TMEM_COLS = 512;
constexpr int REGS_CTRL = 88, REGS_SOFTMAX = 200;   // 128*88 + 256*200 <= 384*168
static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= THREADS * 168, "register split exceeds the launch");

constexpr int MAX_KS = 3, MAX_VS = 3;

struct __align__(8) AttnCtrl {
  uint64_t q_full;
  uint64_t q_empty;     // the last S MMA of an item has run: its Q tiles may be replaced
  uint64_t k_full[MAX_KS];
  uint64_t k_empty[MAX_KS];   // both query tiles' S steps on this key tile have run
  uint64_t v_full[MAX_VS];
  uint64_t v_empty[MAX_VS];   // both query tiles' P V steps on this key tile have run
  uint64_t s_full[2];   // S_k(j) (and every earlier tensor-core step) complete
  uint64_t p_full[2][2];   // softmax k wrote keys [64 h, 64 h + 64) of P_k(j)  ([k][h])
  uint64_t o_done[2];   // O_k final (its last P V step complete)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Keys and values have rings of their own: a key tile is free once both query tiles' S steps on
// it have run, a value tile only after their P V steps.  A commit fires when every tensor-core
// step issued before it is done, so a V slot is handed back only at the end of a key tile's
// work; with two V slots the P V step of the next key tile waited for its value tile to arrive
// and held back the S steps queued behind it.  At D = 128 shared memory holds two query tiles
// (64 KB), two K stages and three V stages (32 KB each).
template <int D>
struct Lay {
  static constexpr int Q_BOX = BQ * 64 * 2;      // [128 rows][64 d] bf16, 16 KB
  static constexpr int KV_BOX = BKV * 64 * 2;    // [128 keys][64 d] bf16, 16 KB
  static constexpr int NB = D / 64;              // boxes along d
  static constexpr int Q_BYTES = NB * Q_BOX;     // one query tile
  static constexpr int K_BYTES = NB * KV_BOX;    // one key (or value) tile
  static constexpr int KS = D == 128 ? 2 : 3, VS = 3;
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KS * K_BYTES;
  static constexpr int OFF_CTRL = OFF_V + VS * K_BYTES;
  static constexpr int TOTAL = OFF_CTRL + 256;
  static_assert(KS <= MAX_KS && VS <= MAX_VS, "ring depth");
  static_assert(TOTAL <= 232448, "shared memory");
  static_assert(sizeof(AttnCtrl) <= 256, "control block");
};

// Key-tile range [lo, hi] (128-key tiles) of query tile rows [q0, q0 + 127] (rows < T).
__device__ __forceinline__ void key_tiles(int q0, int T, int window, int& lo, int& hi) {
  lo = window < 0 ? 0 : max(0, q0 - window) / BKV;
  hi = min(q0 + BQ - 1, T - 1) / BKV;
}

// 32 lanes x 32 consecutive 32-bit columns from registers (tcgen05.st.32x32b.x32).
__device__ __forceinline__ void tmem_st32_u(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}

// One work item: a pair of query tiles of one (batch row, head).  Items are numbered heaviest
// first (the pair index descends).  CTA c of G takes, in round r, item r*G + c when r is even and
// r*G + G-1-c when r is odd: the heaviest items of one round meet the lightest of the next, which
// evens out causal work (whose items shrink with the pair index).
__device__ __forceinline__ int item_index(int c, int r, int G) { return r * G + ((r & 1) ? G - 1 - c : c); }

struct Item {
  int b, h, g, qbase;
  bool has_q1;
  int lo0, hi0, lo1, hi1, jlo, jhi;
};

__device__ __forceinline__ Item decode_item(int it, int T, int H, int Hkv, int B, int window) {
  Item w;
  const int HB = H * B;
  const int npair = (T + 2 * BQ - 1) / (2 * BQ);
  const int pr = npair - 1 - it / HB;
  const int hb = it % HB;
  w.h = hb % H;
  w.b = hb / H;
  w.g = w.h / (H / Hkv);
  w.qbase = pr * 2 * BQ;
  w.has_q1 = w.qbase + BQ < T;
  w.lo1 = 1;
  w.hi1 = 0;   // Q1's range is empty unless it exists
  key_tiles(w.qbase, T, window, w.lo0, w.hi0);
  if (w.has_q1) key_tiles(w.qbase + BQ, T, window, w.lo1, w.hi1);
  w.jlo = w.lo0;
  w.jhi = w.has_q1 ? w.hi1 : w.hi0;   // lo0 <= lo1 and hi0 <= hi1
  return w;
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, int T, int H, int Hkv, int B, int window,
                   int num_items, float scale_log2, bf16* __restrict__ y, int* status) {
  using L = Lay<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {   // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_error(status, NC_ERR_UNSUPPORTED);
    return;
  }
  AttnCtrl* ctl = reinterpret_cast<AttnCtrl*>(smem + L::OFF_CTRL);
  const uint32_t sQ = smem_u32(smem), sK0 = sQ + L::OFF_K, sV0 = sQ + L::OFF_V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first = static_cast<int>(blockIdx.x), stride = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_full), 1);
    mbar_init(smem_u32(&ctl->q_empty), 1);
    for (int s = 0; s < L::KS; ++s) {
      mbar_init(smem_u32(&ctl->k_full[s]), 1);
      mbar_init(smem_u32(&ctl->k_empty[s]), 1);
    }
    for (int s = 0; s < L::VS; ++s) {
      mbar_init(smem_u32(&ctl->v_full[s]), 1);
      mbar_init(smem_u32(&ctl->v_empty[s]), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&ctl->s_full[k]), 1);
      mbar_init(smem_u32(&ctl->p_full[k][0]), 4);
      mbar_init(smem_u32(&ctl->p_full[k][1]), 4);
      mbar_init(smem_u32(&ctl->o_done[k]), 1);
    }
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
  griddep_wait();     // the previous kernel's outputs are complete and visible
  griddep_launch();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp < SM_WARP0) {
    regs_dec<REGS_CTRL>();
    if (warp == 0 && lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint32_t qb = smem_u32(&ctl->q_full);
      uint32_t gkv = 0;   // key tiles loaded so far (ring position)
      int ic = 0;
      bool ok = true;
      for (int r = 0; ok; ++r, ++ic) {
        const int it = item_index(first, r, stride);
        if (it >= num_items) break;
        const Item w = decode_item(it, T, H, Hkv, B, window);
        {   // the next item's query tiles into L2 while this item runs
          const int nx = item_index(first, r + 1, stride);
          if (nx < num_items) {
            const Item wn = decode_item(nx, T, H, Hkv, B, window);
#pragma unroll
            for (int c = 0; c < L::NB; ++c) {
              tma_prefetch_l2_2d(&tmQ, wn.h * D + c * 64, wn.b * T + wn.qbase);
              if (wn.has_q1) tma_prefetch_l2_2d(&tmQ, wn.h * D + c * 64, wn.b * T + wn.qbase + BQ);
            }
          }
        }
        if (ic > 0 && !mbar_wait(smem_u32(&ctl->q_empty), (ic - 1) & 1, abort, status)) break;
        mbar_arrive_expect_tx(qb, (w.has_q1 ? 2 : 1) * L::Q_BYTES);
#pragma unroll
        for (int c = 0; c < L::NB; ++c) {
          tma_load_2d(sQ + c * L::Q_BOX, &tmQ, qb, w.h * D + c * 64, w.b * T + w.qbase);
          if (w.has_q1)
            tma_load_2d(sQ + L::Q_BYTES + c * L::Q_BOX, &tmQ, qb, w.h * D + c * 64, w.b * T + w.qbase + BQ);
        }
        for (int j = w.jlo; j <= w.jhi; ++j, ++gkv) {
          const uint32_t s = gkv % L::KS;
          if (!mbar_wait(smem_u32(&ctl->k_empty[s]), ((gkv / L::KS) & 1) ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->k_full[s]);
          mbar_arrive_expect_tx(fb, L::K_BYTES);
#pragma unroll
          for (int c = 0; c < L::NB; ++c)
            tma_load_2d(sK0 + s * L::K_BYTES + c * L::KV_BOX, &tmK, fb, w.g * D + c * 64, w.b * T + j * BKV);
        }
      }
      // every issued copy must land before the CTA may exit
      if (ic > 0) mbar_wait(qb, (ic - 1) & 1, nullptr, status);
      for (uint32_t q = (gkv > L::KS ? gkv - L::KS : 0); q < gkv; ++q)
        mbar_wait(smem_u32(&ctl->k_full[q % L::KS]), (q / L::KS) & 1, nullptr, status);
    } else if (warp == 2 && lane == 0) {   // value tiles, in the same item and key-tile order
      uint32_t gkv = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int it = item_index(first, r, stride);
        if (it >= num_items) break;
        const Item w = decode_item(it, T, H, Hkv, B, window);
        for (int j = w.jlo; j <= w.jhi; ++j, ++gkv) {
          const uint32_t s = gkv % L::VS;
          if (!mbar_wait(smem_u32(&ctl->v_empty[s]), ((gkv / L::VS) & 1) ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->v_full[s]);
          mbar_arrive_expect_tx(fb, L::K_BYTES);
#pragma unroll
          for (int c = 0; c < L::NB; ++c)
            tma_load_2d(sV0 + s * L::K_BYTES + c * L::KV_BOX, &tmV, fb, w.g * D + c * 64, w.b * T + j * BKV);
        }
      }
      for (uint32_t q = (gkv > L::VS ? gkv - L::VS : 0); q < gkv; ++q)
        mbar_wait(smem_u32(&ctl->v_full[q % L::VS]), (q / L::VS) & 1, nullptr, status);
    } else if (warp == 1 && lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BQ, BKV);
      constexpr uint32_t idO = idesc_bf16_f32_bmn(BQ, D);
      uint32_t gkv = 0;                 // ring position of the current item's first key tile
      uint32_t pv_cnt[2] = {0u, 0u};    // P V steps issued per query tile (p_full phases)
      int ic = 0;
      bool ok = true;
      for (int r = 0; ok; ++r, ++ic) {
        const int it = item_index(first, r, stride);
        if (it >= num_items) break;
        const Item w = decode_item(it, T, H, Hkv, B, window);
        const int lo[2] = {w.lo0, w.lo1}, hi[2] = {w.hi0, w.hi1};
        const int jlo = w.jlo, jhi = w.jhi;
        if (!mbar_wait(smem_u32(&ctl->q_full), ic & 1, abort, status)) break;
        auto pos_of = [&](int j) { return gkv + static_cast<uint32_t>(j - jlo); };   // ring position of key tile j
        auto k_ready = [&](int j) -> bool {
          const uint32_t q = pos_of(j);
          if (!mbar_wait(smem_u32(&ctl->k_full[q % L::KS]), (q / L::KS) & 1, abort, status)) return false;
          tc_fence_after();
          return true;
        };
        auto v_ready = [&](int j) -> bool {
          const uint32_t q = pos_of(j);
          if (!mbar_wait(smem_u32(&ctl->v_full[q % L::VS]), (q / L::VS) & 1, abort, status)) return false;
          tc_fence_after();
          return true;
        };
        auto issue_s = [&](int k, int j) {
          const uint32_t sK = sK0 + (pos_of(j) % L::KS) * L::K_BYTES;
          const uint32_t qk = sQ + k * L::Q_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = sdesc_kmajor_sw128(qk + (kk / 4) * L::Q_BOX + (kk % 4) * 32);
            const uint64_t bd = sdesc_kmajor_sw128(sK + (kk / 4) * L::KV_BOX + (kk % 4) * 32);
            umma_bf16(tmem + 128 * k, a, bd, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&ctl->s_full[k]));
        };
        if (!k_ready(jlo)) break;
        for (int k = 0; k < 2; ++k)
          if (jlo >= lo[k] && jlo <= hi[k]) issue_s(k, jlo);
        umma_commit(smem_u32(&ctl->k_empty[pos_of(jlo) % L::KS]));   // both S steps on key tile jlo issued
        if (jlo == jhi) umma_commit(smem_u32(&ctl->q_empty));   // no S step of this item is left
        for (int j = jlo; j <= jhi && ok; ++j) {
          if (!v_ready(j)) {
            ok = false;
            break;
          }
          const uint32_t sV = sV0 + (pos_of(j) % L::VS) * L::K_BYTES;
          bool next_ready = false;
#pragma unroll
          for (int k = 0; k < 2 && ok; ++k) {
            if (j >= lo[k] && j <= hi[k]) {
              // P V in two halves of 64 keys: the first half runs while softmax k still
              // computes the second
#pragma unroll
              for (int ph = 0; ph < 2; ++ph) {
                if (!mbar_wait(smem_u32(&ctl->p_full[k][ph]), pv_cnt[k] & 1, abort, status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 4 * ph; kk < 4 * ph + 4; ++kk) {
                  const uint64_t bd = sdesc_mnmajor_sw128(sV + kk * 16 * 128, L::KV_BOX);
                  umma_bf16_ts(tmem + 256 + k * D, tmem + 128 * k + kk * 8, bd, idO,
                               (j > lo[k] || kk > 0) ? 1u : 0u);
                }
              }
              if (!ok) break;
              ++pv_cnt[k];
              if (j == hi[k]) umma_commit(smem_u32(&ctl->o_done[k]));   // O_k of this item final
            }
            if (j + 1 <= jhi && j + 1 >= lo[k] && j + 1 <= hi[k]) {
              if (!next_ready) {
                if (!k_ready(j + 1)) {
                  ok = false;
                  break;
                }
                next_ready = true;
              }
              issue_s(k, j + 1);
            }
          }
          if (!ok) break;
          if (j + 1 <= jhi) umma_commit(smem_u32(&ctl->k_empty[pos_of(j + 1) % L::KS]));   // its S steps issued
          if (j + 1 == jhi) umma_commit(smem_u32(&ctl->q_empty));   // no S step of this item is left
          umma_commit(smem_u32(&ctl->v_empty[pos_of(j) % L::VS]));
        }
        gkv += static_cast<uint32_t>(jhi - jlo + 1);
      }
      umma_commit(smem_u32(&ctl->drain));
      mbar_wait(smem_u32(&ctl->drain), 0, nullptr, status);
    }
    __syncwarp();
  } else {
    regs_inc<REGS_SOFTMAX>();
    const int k = (warp - SM_WARP0) >> 2;   // query tile of this warpgroup
    const int quarter = warp & 3;          // TMEM lanes 32*(warp % 4) .. +31
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + 128 * k + lane_off, tO = tmem + 256 + k * D + lane_off;
    const float thr = 8.0f / scale_log2;   // raw-score growth that triggers a rescale (2^8)
    uint32_t tcnt = 0, icnt = 0;           // S tiles and items handled by this query tile slot
    bool ok = true;
    for (int r = 0; ok; ++r) {
    const int it = item_index(first, r, stride);
    if (it >= num_items) break;
    const Item w = decode_item(it, T, H, Hkv, B, window);
    const int q0 = w.qbase + k * BQ;
    const int i = q0 + row;
    const int lo = k == 0 ? w.lo0 : w.lo1, hi = k == 0 ? w.hi0 : w.hi1;
    const int nk = hi - lo + 1;   // 0 when the item has no second query tile
    if (nk <= 0) continue;
    const int kmin = window < 0 ? 0 : i - window;
    const int kmax = min(i, T - 1);
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = 0; t < nk; ++t, ++tcnt) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full[k]), tcnt & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      float sv[BKV];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
        tmem_ld_wait(r2);
        tmem_ld_wait(r3);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sv[c] = __uint_as_float(r0[c]);
          sv[32 + c] = __uint_as_float(r1[c]);
          sv[64 + c] = __uint_as_float(r2[c]);
          sv[96 + c] = __uint_as_float(r3[c]);
        }
      }
      const int key0 = (lo + t) * BKV;
      // Tiles inside every row's visible range need no per-element mask: the last key is at
      // most the first query, the tile lies inside the sequence, and (with a window) its first
      // key is within the window of the last query.  The test is the same for the warpgroup.
      const bool interior = key0 + BKV - 1 <= q0 && key0 + BKV <= T &&
                            (window < 0 || key0 >= q0 + BQ - 1 - window);
      if (!interior) {
        // visible columns [kmin - key0, kmax - key0] as four 32-bit masks: a select per column
        // on a mask bit, with no branch (a per-column compare chain costs about three times as much)
        const int clo = kmin - key0, chi = kmax - key0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int a = max(clo - 32 * q, 0), b = min(chi - 32 * q, 31);
          const uint32_t m = a > b ? 0u : ((0xffffffffu >> (31 - (b - a))) << a);
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[32 * q + c] = ((m >> c) & 1u) ? sv[32 * q + c] : -INFINITY;
        }
      }
      // row max: 8 independent chains of three-input maxima, then a tree
      float mx[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx[q] = fmaxf(sv[2 * q], sv[2 * q + 1]);
#pragma unroll
      for (int c = 16; c < BKV; c += 2) mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], sv[c], sv[c + 1]);
      const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_run + thr) {
        alpha = ex2_approx((m_run - mt) * scale_log2);   // 0 when m_run = -inf
        resc = m_run != -INFINITY;
        m_run = mt;
      }
      const float negm = (m_run == -INFINITY) ? 0.f : -m_run * scale_log2;
      // S_k(j) complete implies O_k += P_k(j-1) V(j-1) complete: O_k may be rescaled now.
      if (__any_sync(0xffffffffu, resc)) {
        const float a = resc ? alpha : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + ch * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
          tmem_st32(tO + ch * 32, o);
        }
        tmem_st_wait();
      }
      // exponents two keys at a time with packed fp32 arithmetic; 4 independent partial sums
      const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(negm, negm);
      float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float2 e = ffma2(make_float2(sv[half * 64 + c], sv[half * 64 + c + 1]), sc2, nm2);
          e.x = ex2_approx(e.x);
          e.y = ex2_approx(e.y);
          ps[(c >> 1) & 3] = fadd2(ps[(c >> 1) & 3], e);
          pk[c / 2] = pack_bf16(e.x, e.y);
        }
        tmem_st32_u(tS + half * 32, pk);   // keys 64 half .. 64 half + 63 -> columns 32 half ..
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[k][half]));
      }
      const float2 pt = fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3]));
      l_run = l_run * alpha + (pt.x + pt.y);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_done[k]), icnt & 1, abort, status));
    ++icnt;
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      bf16* dst = y + (static_cast<size_t>(w.b) * T + i) * (static_cast<size_t>(H) * D) + w.h * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(tO + ch * 32, o);
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
  struct State {
    int num_sms = 0;
  };
  static State states[MAX_DEVICES];
  static bool ready[MAX_DEVICES];
  static std::mutex mu;
  State* st = nullptr;
  const cudaError_t init_err = per_device(states, ready, mu, [](State& s) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lt::TOTAL);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || s.num_sms < 1) {
      cudaGetLastError();
      s.num_sms = 148;
    }
    return cudaSuccess;
  }, &st);
  if (init_err != cudaSuccess) return init_err;
  const int num_sms = st->num_sms;
  const uint64_t M = static_cast<uint64_t>(B) * T;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_2d(&tq, q, static_cast<uint64_t>(H) * D, M, static_cast<uint64_t>(H) * D * 2, 64, BQ) ||
      !make_tmap_bf16_2d(&tk, k, static_cast<uint64_t>(Hkv) * D, M, static_cast<uint64_t>(Hkv) * D * 2, 64, BKV) ||
      !make_tmap_bf16_2d(&tv, v, static_cast<uint64_t>(Hkv) * D, M, static_cast<uint64_t>(Hkv) * D * 2, 64, BKV))
    return cudaErrorInvalidValue;
  const int npair = (T + 2 * BQ - 1) / (2 * BQ);
  const int num_items = npair * H * B;
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute lattr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(num_items < num_sms ? num_items : num_sms);   // persistent: one CTA per SM
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Lt::TOTAL;
  cfg.stream = stream;
  cfg.attrs = lattr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, attn_tc_kernel<D>, tq, tk, tv, T, H, Hkv, B, window, num_items, scale_log2, y, status);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace

cudaError_t launch_attention(const bf16* q, const bf16* k, const bf16* v, int B, int T, int H,
                             int Hkv, int D, int window, bf16* y, int* status, cudaStream_t stream) {
  if (D == 128) return launch_d<128>(q, k, v, B, T, H, Hkv, window, y, status, stream);
  if (D == 64) return launch_d<64>(q, k, v, B, T, H, Hkv, window, y, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nc
