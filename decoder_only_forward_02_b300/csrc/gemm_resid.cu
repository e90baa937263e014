// gemm_resid.cu -- residual-stream update of the output projections (attention c_proj and MLP
// c_proj) as a transposed, persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   xr = resid + A[M, K] . W[N, K]^T          (A: the projection's input, W: its nn.Linear weight)
//   then the fused updates listed at GemmEpi (EPI_RESID): backout cache, the next block's
//   resid_lambdas / x0_lambdas mix or the final backout, the bf16 copy of the new stream and its
//   partial sums of squares per 128-column group (the next RMSNorm's row scale).
//
// ("Nanochat在nanoGPT之上的新增功能", section 1 feature table and notes: pre-norm blocks with
// separate output projections, RMSNorm without weights, per-layer resid/x0 scaling, backout.)
//
// Why transposed: the tensor core computes D^T[n, m] = W[n, :] . A[m, :] -- the weight is the
// MMA's M side (256 output columns per CTA pair, 128 per CTA) and the tokens are its N side -- so
// a TMEM lane is an output column and a TMEM column is a token.  An epilogue warp then holds 32
// consecutive output columns of each token it processes, the layout of a [tokens][32 columns]
// box of the row-major stream: the residual and x0 arrive by TMA into such boxes in shared
// memory, each thread reads and writes its column there (bank-conflict free), and the new stream
// and its bf16 copy leave by TMA stores.  The epilogue's data movement is thus asynchronous bulk
// traffic with deep lookahead, and its instructions are a few per element.  The per-row sums of
// squares become sums across lanes (a reduce-scatter with shuffles) kept in shared memory for the
// whole tile, then across the four warps of a warpgroup after one named barrier per tile.
//
// Tokens per pair tile (NT, a multiple of 32 up to 256) are chosen per launch so that the tiles
// fill whole waves of the resident pairs: at M = 16384, N = 768 on 74 pairs, NT = 224 gives
// 222 tiles = 3 full waves, where 256 gives 192 tiles (the third wave 59% full).
//
// Roles (384 threads = 12 warps; warpgroup 0 at 56 registers per thread, the two epilogue
// warpgroups at 224, within the launch's 384 x 168):
//   warp 0       operand TMA producer (both CTAs): W box [128 rows][64 k] and A box
//                [NT/2 tokens][64 k] per stage, 128-byte swizzle, 4-stage ring, completing on the
//                leader's barrier.
//   warp 1       TMEM (512 columns: two accumulators of up to 256 tokens); in the leader one lane
//                issues tcgen05.mma (M = 256, N = NT, K = 16) for the pair.
//   warps 2, 3   epilogue input producers, one per epilogue warpgroup: for each slot of 8 tokens,
//                the residual (and x0 / backout cache) boxes of the warpgroup's four warps, into a
//                5-slot ring.
//   warps 4..11  epilogue: warp w owns TMEM lanes 32 (w % 4) .. +31 (output columns) and
//                warpgroup (w - 4) / 4 owns tokens [g NT/2, (g + 1) NT/2) of the tile, 16 at a time
//                (two slots), so that two slots' latency chains overlap.
#include "internal.h"
#include "ptx.cuh"

namespace nc {
namespace {

constexpr int BM = 128;                         // output columns (weight rows) per CTA
constexpr int PAIR_N = 2 * BM;                  // output columns of one pair tile
constexpr int BK = 64;
constexpr int MAX_NT = 256;                     // tokens of one pair tile (runtime NT <= MAX_NT)
constexpr int W_BYTES = BM * BK * 2;            // 16 KB
constexpr int A_SLOT = (MAX_NT / 2) * BK * 2;   // 16 KB: up to 128 tokens per CTA
constexpr int STAGES = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;
constexpr int THREADS = 32 * (EPI_WARP0 + NUM_EPI_WARPS);
constexpr int REGS_CTRL = 56, REGS_EPI = 224;
static_assert(128 * REGS_CTRL + 256 * REGS_EPI <= THREADS * 168, "register split exceeds the launch allocation");
constexpr int CH = 8;                            // tokens per epilogue slot (two slots per step)
constexpr int RING = 5;                          // epilogue input slots per warpgroup
// One warp's part of a slot: the residual box [CH][32] fp32 (becomes the new stream in place) and
// the second input box [CH][32] fp32 (x0 or the backout cache; once read, its first half becomes
// the [CH][32] bf16 copy of the new stream).
constexpr int BOX_F32 = CH * 32 * 4;             // 1 KB
constexpr int WSLOT = 2 * BOX_F32;               // 2 KB (a multiple of 128: TMA box alignment)
constexpr int SLOT = 4 * WSLOT;                  // one warpgroup's slot
constexpr int RED_FLOATS = 4 * (MAX_NT / 2);     // one warpgroup's per-warp row sums of one tile: [quarter][token]
constexpr int OFF_RING = STAGES * (W_BYTES + A_SLOT);
constexpr int OFF_RED = OFF_RING + 2 * RING * SLOT;
constexpr int OFF_CTRL = OFF_RED + 2 * 2 * RED_FLOATS * 4;   // [tile parity][warpgroup]
constexpr uint32_t TMEM_COLS = 512;
constexpr int ACC_STRIDE = 256;                  // TMEM columns between the two accumulators
static_assert(WSLOT % 128 == 0 && OFF_RING % 1024 == 0, "TMA box alignment");

struct __align__(8) Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t efull[2][RING];    // epilogue inputs of a slot landed         [warpgroup][slot]
  uint64_t eempty[2][RING];   // the slot's four warps are done with it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr int SMEM_BYTES = 1024 + OFF_CTRL + static_cast<int>(sizeof(Ctrl));
static_assert(SMEM_BYTES <= 232448, "shared memory");

// The tensor maps of the epilogue's streams: [M rows][N columns], boxes of [CH rows][32 columns],
// no swizzle (a box is a dense row-major array in shared memory).
struct ResidMaps {
  CUtensorMap resid, y, x_out, xb;
};

// Pair tile t -> (token block, column block); the column block is the fastest index, so the pairs
// running at the same time share a token block of A (read from DRAM once).  `reverse` walks the
// same order from the last tile.
__device__ __forceinline__ void tile_coords(int t, int num_n, int num_tiles, bool reverse, int& tb, int& nb) {
  if (reverse) t = num_tiles - 1 - t;
  tb = t / num_n;
  nb = t % num_n;
}

// v[0..15] summed over the 32 lanes of the warp, one sum per index: on return lane l holds the
// total of index l >> 1 (lanes l and l ^ 1 hold the same value).  Halving exchange: at each step a
// lane keeps one half of its values, adds the partner's copy of that half and sends the other.
template <bool MAX>
__device__ __forceinline__ float op(float a, float b) { return MAX ? fmaxf(a, b) : a + b; }

template <bool MAX = false>
__device__ __forceinline__ float lane_reduce16(const float (&v)[16], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  float w8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = b4 ? v[i] : v[i + 8];
    w8[i] = op<MAX>(b4 ? v[i + 8] : v[i], __shfl_xor_sync(0xffffffffu, send, 16));
  }
  float w4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b3 ? w8[i] : w8[i + 4];
    w4[i] = op<MAX>(b3 ? w8[i + 4] : w8[i], __shfl_xor_sync(0xffffffffu, send, 8));
  }
  float w2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b2 ? w4[i] : w4[i + 2];
    w2[i] = op<MAX>(b2 ? w4[i + 2] : w4[i], __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float send = b1 ? w2[0] : w2[1];
  const float w = op<MAX>(b1 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, send, 2));
  return op<MAX>(w, __shfl_xor_sync(0xffffffffu, w, 1));
}

template <bool F8>   // F8: e4m3 operands (the bf16 instantiation is unchanged)
__global__ void __launch_bounds__(THREADS, 1)
    gemm_resid_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ ResidMaps rm, int M, int N, int K, int NT, int reverse,
                      const __grid_constant__ GemmEpi ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sW = smem_u32(smem);
  const uint32_t sA = sW + STAGES * W_BYTES;
  float* red = reinterpret_cast<float*>(smem + OFF_RED);
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + OFF_CTRL);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();            // 0: pair leader (issues the MMAs)
  const int pair = static_cast<int>(blockIdx.x) >> 1, npairs = static_cast<int>(gridDim.x) >> 1;
  const int half = NT / 2;
  const int nsteps = half / CH;                       // epilogue slots per tile and warpgroup (even)
  const int num_n = (N + PAIR_N - 1) / PAIR_N, num_t = (M + NT - 1) / NT;
  // a stage holds 128 bytes of K per row: 64 bf16 or 128 e4m3 elements
  constexpr int kstep = F8 ? 2 * BK : BK;
  const int num_tiles = num_n * num_t, kblocks = K / kstep;
  const bool has_y = ep.Y != nullptr;
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
    for (int g = 0; g < 2; ++g)
      for (int s = 0; s < RING; ++s) {
        mbar_init(smem_u32(&ctl->efull[g][s]), 1);
        mbar_init(smem_u32(&ctl->eempty[g][s]), 4);
      }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  griddep_wait();   // the previous kernel's outputs are complete and visible
  griddep_launch();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp < EPI_WARP0) {
    regs_dec<REGS_CTRL>();
    if (warp == 0 && lane == 0) {
      // W is re-read for every token block and stays in L2; a token block of A is read by the
      // num_n pairs of one wave and then never again.
      const uint64_t pol_w = policy_evict_last(), pol_a = policy_evict_first();
      const uint32_t stage_tx = 2u * (W_BYTES + static_cast<uint32_t>(half) * BK * 2);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        int tb, nb;
        tile_coords(tile, num_n, num_tiles, reverse != 0, tb, nb);
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&ctl->empty[s]), ph ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(smem_u32(&ctl->full[s]), 0);   // the leader's barrier
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), stage_tx);
          tma_load_2d_pair_hint(sW + s * W_BYTES, &tmW, fb, kb * kstep, nb * PAIR_N + static_cast<int>(rank) * BM,
                                pol_w);
          tma_load_2d_pair_hint(sA + s * A_SLOT, &tmA, fb, kb * kstep, tb * NT + static_cast<int>(rank) * half, pol_a);
          ++it;
        }
      }
      // The leader's full barriers count both CTAs' copies: once its last phases completed, every
      // copy issued by the pair has landed (the peer exits only after the final sync).
      if (rank == 0) {
        for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_cluster(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1, nullptr, status);
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      const uint32_t idesc = F8 ? idesc_e4m3_f32(2 * BM, NT) : idesc_bf16_f32(2 * BM, NT);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs, ++tc) {
        const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
        if (!mbar_wait_cluster(smem_u32(&ctl->tempty[a]), aph ^ 1, abort, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * ACC_STRIDE;
        for (int kb = 0; kb < kblocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait_cluster(smem_u32(&ctl->full[s]), ph, abort, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t wd = sdesc_kmajor_sw128(sW + s * W_BYTES + kk * 32);
            const uint64_t ad = sdesc_kmajor_sw128(sA + s * A_SLOT + kk * 32);
            if constexpr (F8) umma_f8_pair(d_tmem, wd, ad, idesc, (kb | kk) != 0 ? 1u : 0u);
            else umma_bf16_pair(d_tmem, wd, ad, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&ctl->empty[s]), 0x3);
          ++it;
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&ctl->tfull[a]), 0x3);
      }
      umma_commit_pair(smem_u32(&ctl->drain), 0x1);
      mbar_wait(smem_u32(&ctl->drain), 0, nullptr, status);
    } else if ((warp == 2 || warp == 3) && lane == 0) {
      // epilogue inputs of warpgroup g: per step, the four warps' [CH][32] boxes of the residual
      // (and of Y), into slot k % RING
      const int g = warp - 2;
      const uint32_t ring = smem_u32(smem + OFF_RING + g * RING * SLOT);
      const uint32_t step_tx = 4u * BOX_F32 * (has_y ? 2u : 1u);
      uint32_t k = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        int tb, nb;
        tile_coords(tile, num_n, num_tiles, reverse != 0, tb, nb);
        const int n0 = nb * PAIR_N + static_cast<int>(rank) * BM;
        const bool col_ok = n0 < N;
        const int m0 = tb * NT + g * half;
        for (int c = 0; c < nsteps; ++c, ++k) {
          const uint32_t s = k % RING, ph = (k / RING) & 1;
          if (!mbar_wait(smem_u32(&ctl->eempty[g][s]), ph ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->efull[g][s]);
          if (!col_ok) {   // nothing to load: the warps skip this CTA's (absent) columns
            mbar_arrive(fb);
            continue;
          }
          mbar_arrive_expect_tx(fb, step_tx);
          for (int q = 0; q < 4; ++q) {
            const uint32_t dst = ring + s * SLOT + q * WSLOT;
            tma_load_2d(dst, &rm.resid, fb, n0 + 32 * q, m0 + c * CH);
            if (has_y) tma_load_2d(dst + BOX_F32, &rm.y, fb, n0 + 32 * q, m0 + c * CH);
          }
        }
      }
      // every issued copy must land before the CTA may exit
      for (uint32_t j = (k > RING ? k - RING : 0); j < k; ++j)
        mbar_wait(smem_u32(&ctl->efull[g][j % RING]), (j / RING) & 1, nullptr, status);
    }
    __syncwarp();
  } else {
    regs_inc<REGS_EPI>();
    const int q = warp & 3;                     // TMEM lanes 32 q .. +31: this warp's output columns
    const int wg = (warp - EPI_WARP0) >> 2;     // tokens [wg * half, (wg + 1) * half) of each tile
    const int tq = q * 32 + lane;               // thread index within the warpgroup
    const int bar_id = 1 + wg;
    const float ea = ep.a, eb = ep.b;
    // 8-bit operands: the accumulator times the input's and the weight's 1 / scale (exactly xv + acc
    // for bf16, where dq = 1)
    const float dq = F8 ? __ldg(ep.fp8_sa) * __ldg(ep.fp8_sw) : 1.f;
    const bool has_xm = ep.xm_out != nullptr, has_x = ep.x_out != nullptr;
    uint8_t* ring = smem + OFF_RING + wg * RING * SLOT;
    uint32_t k = 0;    // steps handled (ring position)
    uint32_t tc = 0;   // tiles handled
    for (int tile = pair; tile < num_tiles; tile += npairs, ++tc) {
      const uint32_t a = tc & 1, aph = (tc >> 1) & 1;
      int tb, nb;
      tile_coords(tile, num_n, num_tiles, reverse != 0, tb, nb);
      const int n0 = nb * PAIR_N + static_cast<int>(rank) * BM;   // this CTA's 128 output columns
      const int m0 = tb * NT + wg * half;
      const bool col_ok = n0 < N;   // N % 128 == 0: all of the CTA's columns or none
      const bool ok = mbar_wait_cluster(smem_u32(&ctl->tfull[a]), aph, abort, status);
      if (named_bar_any(bar_id, 128, !ok)) break;   // the warpgroup leaves together
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * ACC_STRIDE + wg * half;
      const uint32_t tempty = mapa_shared(smem_u32(&ctl->tempty[a]), 0);
      float* red_t = red + (a * 2 + wg) * RED_FLOATS;   // this tile's per-warp row sums [quarter][token]
      bool fail = false;
      // two slots (2 CH tokens) per step: the two halves' latency chains overlap
#pragma unroll 1
      for (int c = 0; c < nsteps; c += 2, k += 2) {
        const uint32_t s0 = k % RING, s1 = (k + 1) % RING;
        uint32_t r[16];
        tmem_ld16(taddr + c * CH, r);
        bool in_ok = mbar_wait(smem_u32(&ctl->efull[wg][s0]), (k / RING) & 1, abort, status);
        in_ok = in_ok && mbar_wait(smem_u32(&ctl->efull[wg][s1]), ((k + 1) / RING) & 1, abort, status);
        tmem_ld_wait(r);
        if (c + 2 >= nsteps) {   // the accumulator's last reads are done: it may take the tile after next
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(tempty);
        }
        if (!__all_sync(0xffffffffu, in_ok)) {
          fail = true;
          break;
        }
        uint8_t* w0 = ring + s0 * SLOT + q * WSLOT;
        uint8_t* w1 = ring + s1 * SLOT + q * WSLOT;
        float* xs[2] = {reinterpret_cast<float*>(w0) + lane, reinterpret_cast<float*>(w1) + lane};
        const float* ys[2] = {reinterpret_cast<const float*>(w0 + BOX_F32) + lane,
                              reinterpret_cast<const float*>(w1 + BOX_F32) + lane};
        bf16* bs[2] = {reinterpret_cast<bf16*>(w0 + BOX_F32) + lane, reinterpret_cast<bf16*>(w1 + BOX_F32) + lane};
        float xv[16], yv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          xv[j] = xs[j / CH][(j % CH) * 32];
          yv[j] = has_y ? ys[j / CH][(j % CH) * 32] : 0.f;
        }
        float sq[16], xrv[16], ax[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float xr = fmaf(dq, __uint_as_float(r[j]), xv[j]);
          const float x = has_y ? fmaf(ea, xr, eb * yv[j]) : ea * xr;
          xrv[j] = xr;
          sq[j] = x * x;
          ax[j] = fabsf(x);
          xs[j / CH][(j % CH) * 32] = x;
          bs[j / CH][(j % CH) * 32] = __float2bfloat16_rn(x);   // over the second input, already read
        }
        // the warp's boxes to global memory (a box that runs past row M is clipped by the tensor
        // maps; one that starts there is not stored)
        fence_proxy_async_smem();
        __syncwarp();
        const int col = n0 + 32 * q, row = m0 + c * CH;
        if (lane == 0 && col_ok) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (row + h * CH >= M) break;
            const uint32_t w = smem_u32(h == 0 ? w0 : w1);
            if (has_x) tma_store_2d(&rm.x_out, w, col, row + h * CH);
            tma_store_2d(&rm.xb, w + BOX_F32, col, row + h * CH);
          }
          bulk_commit();
        }
        if (has_xm && col_ok) {   // the backout cache (one layer per forward): plain stores
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (row + j < M) ep.xm_out[static_cast<size_t>(row + j) * N + col + lane] = xrv[j];
        }
        // 8-bit path: each token's largest |x'| over this warp's 32 columns, for the maximum
        // the next quantisation of the stream needs
        if constexpr (F8) {
          if (ep.rowmax_out != nullptr) {
            const float amx = lane_reduce16<true>(ax, lane);
            const int tok = row + (lane >> 1);
            if ((lane & 1) == 0 && col_ok && tok < M)
              ep.rowmax_out[static_cast<size_t>(tok) * (N / 32) + col / 32] = amx;
          }
        }
        // this warp's 32 columns of each token's sum of squares (across lanes)
        const float ssum = lane_reduce16(sq, lane);
        if ((lane & 1) == 0) red_t[q * (MAX_NT / 2) + c * CH + (lane >> 1)] = ssum;
        if (lane == 0) {   // the slots may be refilled once the stores have read them
          bulk_wait_read<0>();
          mbar_arrive(smem_u32(&ctl->eempty[wg][s0]));
          mbar_arrive(smem_u32(&ctl->eempty[wg][s1]));
        }
        __syncwarp();
      }
      if (named_bar_any(bar_id, 128, fail)) break;
      // the tile's row sums over the CTA's 128 columns: the four warps' parts, in a fixed order
      if (col_ok) {
        const int gcol = n0 / SS_GROUP;
        for (int t = tq; t < half; t += 128) {
          const int m = m0 + t;
          if (m < M) {
            const float* p = red_t + t;
            ep.ssp_out[static_cast<size_t>(m) * ep.ncg + gcol] =
                ((p[0] + p[MAX_NT / 2]) + p[2 * (MAX_NT / 2)]) + p[3 * (MAX_NT / 2)];
          }
        }
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

// Tokens per pair tile: the NT (a multiple of 32, at most 256) whose tile count fills the resident
// pairs' waves best, counting a fixed overhead of 32 token-columns per tile.
int choose_nt(int M, int N, int max_pairs) {
  const int num_n = (N + PAIR_N - 1) / PAIR_N;
  int best = MAX_NT;
  long best_cost = -1;
  for (int nt = MAX_NT; nt >= 32; nt -= 32) {
    const long tiles = static_cast<long>((M + nt - 1) / nt) * num_n;
    const long waves = (tiles + max_pairs - 1) / max_pairs;
    const long cost = waves * (nt + 32);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = nt;
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_gemm_resid(const bf16* A, const bf16* W, int M, int N, int K, const GemmEpi& ep, int num_sms,
                              cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || K % (ep.fp8 ? 2 * BK : BK) != 0 || N % SS_GROUP != 0) return cudaErrorInvalidValue;
  if (ep.fp8 && (ep.fp8_sa == nullptr || ep.fp8_sw == nullptr)) return cudaErrorInvalidValue;
  if (ep.resid == nullptr || ep.xb == nullptr || ep.ssp_out == nullptr || ep.ncg != N / SS_GROUP)
    return cudaErrorInvalidValue;
  // the TMA boxes of the stream start on 16-byte boundaries
  const auto a16 = [](const void* p) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  if (!a16(ep.resid) || !a16(ep.Y) || !a16(ep.x_out) || !a16(ep.xm_out) || !a16(ep.xb)) return cudaErrorInvalidValue;
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
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // occupancy query without the PDL attribute
  State* st = nullptr;
  const cudaError_t init_err = per_device(states, ready, mu, [&](State& s) {
    cudaError_t e = cudaFuncSetAttribute(gemm_resid_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_resid_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * (num_sms / 2));
    if (cudaOccupancyMaxActiveClusters(&s.max_pairs, gemm_resid_kernel<false>, &q) != cudaSuccess || s.max_pairs < 1) {
      cudaGetLastError();
      s.max_pairs = num_sms / 2;
    }
    return cudaSuccess;
  }, &st);
  if (init_err != cudaSuccess) return init_err;
  const int NT = choose_nt(M, N, st->max_pairs);
  CUtensorMap tw, ta;
  ResidMaps rm;
  const uint64_t Mu = static_cast<uint64_t>(M), Nu = static_cast<uint64_t>(N);
  if (ep.fp8) {   // e4m3 operands: rows of K bytes, one 128-byte stage row = 128 elements of K
    const uint64_t Ku = static_cast<uint64_t>(K);
    if (!make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, Ku, N, Ku, 2 * BK, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, Ku, M, Ku, 2 * BK, NT / 2)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_bf16_2d(&tw, W, K, N, static_cast<uint64_t>(K) * 2, BK, BM)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_2d(&ta, A, K, M, static_cast<uint64_t>(K) * 2, BK, NT / 2)) return cudaErrorInvalidValue;
  }
  auto f32map = [&](CUtensorMap* m, const float* p) {
    return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p, Nu, Mu, Nu * 4, 32, CH, false);
  };
  // maps of absent streams alias the residual's (never used: the kernel checks the pointers)
  if (!f32map(&rm.resid, ep.resid) || !f32map(&rm.y, ep.Y ? ep.Y : ep.resid) ||
      !f32map(&rm.x_out, ep.x_out ? ep.x_out : ep.resid) ||
      !make_tmap_2d(&rm.xb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ep.xb, Nu, Mu, Nu * 2, 32, CH, false))
    return cudaErrorInvalidValue;
  const int tiles = ((M + NT - 1) / NT) * ((N + PAIR_N - 1) / PAIR_N);
  const int pairs = tiles < st->max_pairs ? tiles : st->max_pairs;
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = 2;
  // The MLP down projection reads h, which the up projection has just written in ascending token
  // order: walking its tiles from the last one starts on the rows most likely still in L2.
  const int reverse = K > 1024 ? 1 : 0;
  const cudaError_t e = ep.fp8 ? cudaLaunchKernelEx(&cfg, gemm_resid_kernel<true>, tw, ta, rm, M, N, K, NT, reverse, ep)
                              : cudaLaunchKernelEx(&cfg, gemm_resid_kernel<false>, tw, ta, rm, M, N, K, NT, reverse, ep);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace nc
