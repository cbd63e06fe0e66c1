// Grouped W8A8 GEMM, int32-accumulator engine for fp16-stored activation
// codes: weights widened into tensor memory, token tiles shared by CTA pairs
// (tcgen05, sm_103a).
//
// The channel-wise INT8 GEMM of "[Feature] DeepSeek V3/R1 INT8 Quantization
// (channel-wise)" with the int32 accumulator: C = A_e W_e^T exactly, then
// v = (float(C) * sa[r]) * sw[e][n].  Activation codes arrive stored as fp16
// values with each row's squared norm (written by the permute and
// SiLU-mul-quant kernels); TMA puts them straight into the 128-byte swizzled
// K-major layout the MMA reads, each CTA of a cluster pair loading half of a
// token tile and multicasting it to both.  The int8 weights are widened to
// fp16 by converter warps that own one weight row each and write it into
// tensor memory (tcgen05.st), which the MMA then reads as its A operand: no
// fp16 copy of the weights ever goes through shared memory.  tcgen05.mma
// kind::f16 accumulates in float32 over the whole K range in one pass, exact
// when max||a||^2 * max||w||^2 < 2^48 (Cauchy-Schwarz bounds every partial
// sum below 2^24); the epilogue checks that with the producers' token norms
// and the converters' weight norms, and a failing tile raises a device flag
// for the exact recompute.
//
// Operand roles are swapped relative to the row-major problem: MMA M = 128
// output channels, N = the item's tokens.  An item holds up to TN = 320 (or,
// for experts averaging more than 320 rows, 384) tokens of one expert (two
// MMAs per K step beyond 256), so an expert is one item per weight block and
// its weight tile is widened once.  Tensor memory: columns [0, TN) the
// accumulator, then four 32-column weight stages.
//   warp 0      TMA producer of the int8 weights
//   warp 22     TMA producer of the tokens (half of each stage, multicast);
//               separate from the weight producer so neither ring's wait
//               holds back the other's copies
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-9   converters, two groups of four taking alternate K stages:
//               one weight row per thread, int8 -> fp16 -> TMEM; a stage is
//               signalled ready once its token slot has landed as well, so
//               the MMA issuer waits on one barrier per stage
//   warps 10-21 epilogue: dequant, bf16; three triples of four warps (one
//               per lane quarter) take every third 32-token group, so the
//               single accumulator is drained three times faster.  In the
//               TN = 320 plan a full group goes through an 8 KB shared-memory
//               box (32 tokens x 128 channels) and leaves in one TMA store of
//               whole 256-byte rows; the ragged last group of an item, and
//               every group of the TN = 384 plan, is stored directly (a box
//               would run into the next expert's rows).
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int WM = 128, BK = 64;
constexpr int NCG = 2;                 // converter groups (four warps each), alternate K stages
constexpr int NEPI = 12;               // epilogue warps (three per tensor-memory lane quarter)
constexpr int NTRIP = NEPI / 4;        // epilogue triples
constexpr int WARP_EPI = 2 + 4 * NCG;  // first epilogue warp
constexpr int WARP_TOK = WARP_EPI + NEPI;  // token producer
constexpr int NTHREADS = (WARP_TOK + 1) * 32;

// Shared- and tensor-memory plan of one instantiation.  TN = most tokens of
// one item (accumulator columns); BOX = full output groups leave through a
// shared-memory box and one TMA store (the 24 KB of boxes fit beside four
// token slots only for TN = 320; the TN = 384 plan stores directly and
// serves experts, or a dense linear, of more than 320 rows on average).
template <int TN, bool BOX>
struct Tc5Plan {
  static constexpr int TNMAX = TN;          // most tokens of one item
  static constexpr int ACC_COLS = TNMAX;    // accumulator columns
  static constexpr int WT_COL = ACC_COLS;   // first tensor-memory column of the weight stages
  static constexpr int NWT = 4;             // weight stages in tensor memory (32 columns each)
  static constexpr int SW8 = 4;             // int8 weight staging ring (shared memory)
  static constexpr int ST = 4;              // token slots (shared memory)
  // a K stage's weight columns and token slot are released together: one
  // commit per stage, multicast to both CTAs' token-empty barriers, which
  // the converters wait on as well
  static_assert(NWT == ST, "a weight stage is released with its token slot");
  static constexpr int W8B = WM * BK;        // int8 weight stage bytes
  static constexpr int TB = TNMAX * BK * 2;  // token slot bytes (fp16)
  static constexpr int TBOX = TNMAX / 2;     // token rows each CTA loads for the widest items
  static_assert(TBOX % 8 == 0 && TBOX <= 256, "token box heights");
  static constexpr int OUTB = 32 * WM * 2;   // one bf16 output box: 32 tokens x 128 channels
  static constexpr int OFF_T = 0;
  static constexpr int OFF_W8 = OFF_T + ST * TB;
  static constexpr int OFF_OUT = OFF_W8 + SW8 * W8B;  // [NTRIP] output boxes when BOX
  static constexpr int OFF_BAR = OFF_OUT + (BOX ? NTRIP * OUTB : 0);
  static constexpr int B_W8_FULL = 0, B_W8_EMPTY = SW8, B_WT_FULL = 2 * SW8,
                       B_T_FULL = 2 * SW8 + NWT, B_T_EMPTY = B_T_FULL + ST,
                       B_ACC_FULL = B_T_EMPTY + ST, B_ACC_EMPTY = B_ACC_FULL + 1,
                       B_NORM_READY = B_ACC_FULL + 2,  // [2]
      B_NORM_FREE = B_ACC_FULL + 4,                    // [2]
      B_NORM_READ = B_ACC_FULL + 6,                    // [2]
      B_MMA_DONE = B_ACC_FULL + 8, NBAR = B_ACC_FULL + 9;
  static constexpr int OFF_NORM = OFF_BAR + NBAR * 8;  // int32 [2 buffers][NCG converter groups]
  static constexpr int OFF_TMEM = OFF_NORM + 8 * NCG;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int NGRP = TNMAX / 32;  // 32-token groups of the largest item
  static constexpr int GPT = (NGRP + NTRIP - 1) / NTRIP;  // groups per triple
  // each thread of a triple stages one token scale of one of its groups
  static_assert(!BOX || GPT <= 4, "a triple's token scales fit its four warps");
  // BOX plan: each triple's token scales of its groups, [triple][item parity][GPT * 32]
  static constexpr int OFF_TSC = (OFF_ABORT + 4 + 15) & ~15;
  static constexpr int TSC_BYTES = BOX ? NTRIP * 2 * GPT * 32 * 4 : 0;
  static constexpr int SMEM_BYTES = OFF_TSC + TSC_BYTES + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
  static_assert((TB % 1024) == 0 && (W8B % 1024) == 0 && (OUTB % 1024) == 0 &&
                    (TBOX * BK * 2) % 1024 == 0,
                "stage alignment");
  static_assert(ACC_COLS + NWT * 32 <= 512, "tensor memory plan");
};

__device__ __forceinline__ int sq4(uint32_t w, int acc) { return __dp4a(int(w), int(w), acc); }

// Token tensor maps, one per box height 8, 16, ..., TN / 2: each CTA of a
// pair loads exactly half of an item's rows rounded up to the MMA's
// 16-token granularity, so no L2 bandwidth goes to rows the MMA skips.
template <int TN>
struct TokenMaps {
  static constexpr int N = TN / 16;  // box heights 8 * (i + 1)
  CUtensorMap m[N];
};

template <int TN, bool BOX>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    gemm_tc5_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ TokenMaps<TN> tmT,
                    const __grid_constant__ CUtensorMap tmO, const GemmArgs a,
                    const Tile *__restrict__ tiles, const int32_t *__restrict__ ntiles,
                    int32_t *__restrict__ redo) {
  using P = Tc5Plan<TN, BOX>;
  extern __shared__ uint8_t smem_raw[];
  const int NBP = int(a.N / (2 * WM));  // pairs of 128-row weight blocks
  const int items = ntiles[0] * NBP;
  const int pair = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  if (pair >= items) return;  // uniform over the pair, before any setup
  const uint32_t rank = cluster_ctarank();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + P::OFF_ABORT);
  volatile int *norm = reinterpret_cast<volatile int *>(sm + P::OFF_NORM);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + P::OFF_TMEM);
  auto bar = [&](int i) { return base + P::OFF_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = int(a.K / BK);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2 * NCG; ++i) norm[i] = 0;
    for (int s = 0; s < P::SW8; ++s) {
      mbar_init(bar(P::B_W8_FULL + s), 1);
      mbar_init(bar(P::B_W8_EMPTY + s), 4);
    }
    for (int s = 0; s < P::NWT; ++s) {
      mbar_init(bar(P::B_WT_FULL + s), 4);
    }
    for (int s = 0; s < P::ST; ++s) {
      mbar_init(bar(P::B_T_FULL + s), 1);   // local expect_tx; bytes from both CTAs' copies
      mbar_init(bar(P::B_T_EMPTY + s), 2);  // MMA completions of both CTAs
    }
    mbar_init(bar(P::B_ACC_FULL), 1);
    mbar_init(bar(P::B_ACC_EMPTY), NEPI);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(P::B_NORM_READY + b), 4 * NCG);  // every converter warp
      mbar_init(bar(P::B_NORM_FREE + b), 1);
      mbar_init(bar(P::B_NORM_READ + b), NEPI);
    }
    mbar_init(bar(P::B_MMA_DONE), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any multicast lands
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(a.status, WQ_ERR_TIMEOUT);
  };
  auto nmma_of = [](int rows) { return (rows + 15) & ~15; };
  // The pair's r-th item: rounds of npairs items, alternate rounds walked in
  // reverse, over the longest-first tile list, so the shortest items fill
  // the last round (every role walks the same sequence).
  auto item_at = [&](int r) { return r * npairs + ((r & 1) ? npairs - 1 - pair : pair); };

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int g = 0, gw = 0;
      bool ok = true;
      for (int r = 0, ip = pair; ip < items && ok; ip = item_at(++r)) {
        const Tile tl = tiles[ip / NBP];
        const int wb = (ip % NBP) * 2 + int(rank);
        const int wrow = int(int64_t(tl.expert) * a.N + int64_t(wb) * WM);
        for (int i = 0; i < KT; ++i, ++g) {
          const int sw = g % P::SW8;
          if (!mbar_wait<200>(bar(P::B_W8_EMPTY + sw), ((g / P::SW8) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(bar(P::B_W8_FULL + sw), P::W8B);
          tma_load_2d(base + P::OFF_W8 + uint32_t(sw) * P::W8B, &tmW, i * BK, wrow, bar(P::B_W8_FULL + sw));
          gw = g + 1;
        }
      }
      if (!ok) {
        for (int j = gw > P::SW8 ? gw - P::SW8 : 0; j < gw; ++j)
          mbar_wait_bounded(bar(P::B_W8_FULL + j % P::SW8), (j / P::SW8) & 1);
      }
    }
  } else if (warp == WARP_TOK) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      int g = 0, gt = 0;
      bool ok = true;
      for (int r = 0, ip = pair; ip < items && ok; ip = item_at(++r)) {
        const Tile tl = tiles[ip / NBP];
        const int box = nmma_of(tl.rows) / 2;  // this CTA's half: a multiple of 8 rows
        const CUtensorMap *tmap = &tmT.m[box / 8 - 1];
        const uint32_t ttx = uint32_t(2 * box * BK * 2);
        const int trow = tl.row0 + int(rank) * box;
        for (int i = 0; i < KT; ++i, ++g) {
          const int stt = g % P::ST;
          if (!mbar_wait<200>(bar(P::B_T_EMPTY + stt), ((g / P::ST) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(bar(P::B_T_FULL + stt), ttx);
          tma_load_2d_mc(base + P::OFF_T + uint32_t(stt) * P::TB + rank * uint32_t(box * BK * 2), tmap,
                         i * BK, trow, bar(P::B_T_FULL + stt), 3);
          gt = g + 1;
        }
      }
      if (!ok) {
        for (int j = gt > P::ST ? gt - P::ST : 0; j < gt; ++j)
          mbar_wait_bounded(bar(P::B_T_FULL + j % P::ST), (j / P::ST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int g = 0, ii = 0;
      bool ok = true;
      Tile next = tiles[pair / NBP];  // the next item's tile, loaded an item ahead
      for (int ip = pair; ip < items && ok; ip = item_at(++ii)) {
        const Tile tl = next;
        if (item_at(ii + 1) < items) next = tiles[item_at(ii + 1) / NBP];
        const int nm = nmma_of(tl.rows);
        // above 256 tokens: two MMAs of balanced widths (multiples of 16, so
        // the second token block starts on an 8-row swizzle group)
        const int n0 = nm <= 256 ? nm : ((nm / 2 + 15) & ~15), n1 = nm - n0;
        const uint32_t idesc0 = idesc_f16(WM, n0), idesc1 = idesc_f16(WM, n1 > 0 ? n1 : 16);
        if (!mbar_wait(bar(P::B_ACC_EMPTY), (ii & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        for (int i = 0; i < KT; ++i, ++g) {
          const int swt = g % P::NWT, stt = g % P::ST;
          // weights widened and tokens landed (the converters wait for both)
          if (!mbar_wait(bar(P::B_WT_FULL + swt), (g / P::NWT) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t wt = tmem + uint32_t(P::WT_COL + swt * 32);
          const uint32_t t0 = base + P::OFF_T + uint32_t(stt) * P::TB;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16_ts(tmem, wt + 8u * kk, sdesc(t0 + 32u * kk), idesc0, (i | kk) ? 1u : 0u);
          if (n1 > 0) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16_ts(tmem + uint32_t(n0), wt + 8u * kk, sdesc(t0 + uint32_t(n0) * 128u + 32u * kk), idesc1,
                         (i | kk) ? 1u : 0u);
          }
          mma_commit_mc(bar(P::B_T_EMPTY + stt), 3);
        }
        if (ok) mma_commit(bar(P::B_ACC_FULL));
      }
      mma_commit(bar(P::B_MMA_DONE));
      mbar_wait_bounded(bar(P::B_MMA_DONE), 0);
    }
  } else if (warp < WARP_EPI) {
    // ------------------------------------------------------------ converters
    // thread = weight row (its tensor-memory lane); group `grp` takes the K
    // stages of parity grp
    const int grp = (warp - 2) >> 2;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t tlane = uint32_t(q * 32) << 16;
    int gbase = 0, ii = 0;
    bool ok = true;
    for (int ip = pair; ip < items && ok; ip = item_at(++ii), gbase += KT) {
      int nrm = 0;
      for (int i = grp; i < KT; i += NCG) {
        const int g = gbase + i;
        const int sw = g % P::SW8, swt = g % P::NWT;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(P::B_W8_FULL + sw), (g / P::SW8) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        // the slot is 64-byte swizzled: piece m of a row sits at piece
        // m ^ ((row / 2) % 4), so the eight rows a quarter-warp reads at once
        // hit eight different 16-byte bank groups
        const uint8_t *src = sm + P::OFF_W8 + sw * P::W8B + row * 64;
        const int swz = (row >> 1) & 3;
        uint4 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = *reinterpret_cast<const uint4 *>(src + ((m ^ swz) << 4));
        fence_async_smem();  // these reads before the next copy into the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P::B_W8_EMPTY + sw));
        uint32_t f[32];
        int part[4];  // the stage's squared norm in four independent partial sums
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          s8x4_to_f16x4(v[m].x, f[8 * m + 0], f[8 * m + 1]);
          s8x4_to_f16x4(v[m].y, f[8 * m + 2], f[8 * m + 3]);
          s8x4_to_f16x4(v[m].z, f[8 * m + 4], f[8 * m + 5]);
          s8x4_to_f16x4(v[m].w, f[8 * m + 6], f[8 * m + 7]);
          part[m] = sq4(v[m].w, sq4(v[m].z, 0)) + sq4(v[m].y, sq4(v[m].x, 0));
        }
        // one add per stage joins the running norm (a serial chain of dot
        // products through it was the converters' critical path)
        nrm += (part[0] + part[1]) + (part[2] + part[3]);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(P::B_T_EMPTY + swt), ((g / P::NWT) & 1) ^ 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        tmem_st32(tmem + tlane + uint32_t(P::WT_COL + swt * 32), f);
        tmem_wait_st();
        tc_fence_before();
        // the stage's token slot has landed too: the MMA issuer then checks
        // a single barrier per stage (it is the pipeline's critical thread;
        // the converters run stages ahead of it)
        if (!__all_sync(0xffffffffu, mbar_wait(bar(P::B_T_FULL + swt), (g / P::ST) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P::B_WT_FULL + swt));
      }
      if (!ok) break;
      int wmax = nrm;  // this row's squared norm over this group's K stages
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      const int b = ii & 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar(P::B_NORM_FREE + b), ((ii >> 1) & 1) ^ 1, abort_flag))) {
        fail();
        break;
      }
      if (lane == 0) atomicMax(const_cast<int *>(norm + NCG * b + grp), wmax);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P::B_NORM_READY + b));
    }
  } else if (warp < WARP_TOK) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // tensor-memory lane quarter of this warp
    const int trip = (warp - WARP_EPI) >> 2;  // triple: 32-token groups trip, trip + NTRIP, ...
    const bool leader = q == 0 && lane == 0;  // issues the triple's box stores
    uint16_t *box = reinterpret_cast<uint16_t *>(sm + P::OFF_OUT + trip * P::OUTB);
    const uint32_t box_s = base + P::OFF_OUT + uint32_t(trip) * P::OUTB;
    int ii = 0;
    for (int ip = pair; ip < items; ip = item_at(++ii)) {
      const Tile tl = tiles[ip / NBP];
      const int wb = (ip % NBP) * 2 + int(rank);
      const int b = ii & 1, par = (ii >> 1) & 1;
      int tmax = 0;  // largest squared token-row norm of the item
      for (int j = lane; j < tl.rows; j += 32) tmax = max(tmax, a.a_norm2[int64_t(tl.row0) + j]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      // the item's token scales and this thread's weight scale, loaded while
      // the item's MMAs still run.  BOX plan: each thread of the triple puts
      // one token scale of the triple's groups into shared memory (published
      // by the triple's barrier below) and the drain reads them as
      // broadcasts; otherwise lane j of register sal[p] holds token 32p + j.
      const int64_t n = int64_t(wb) * WM + q * 32 + lane;  // this thread's output channel
      const float swn = a.sw[int64_t(tl.expert) * a.N + n];
      float sal[BOX ? 1 : P::NGRP];
      float *tsc = reinterpret_cast<float *>(sm + P::OFF_TSC) + (trip * 2 + (ii & 1)) * P::GPT * 32;
      if constexpr (BOX) {
        const int tok = (trip + NTRIP * q) * 32 + lane;  // group trip + NTRIP*q, token lane
        if (q < P::GPT) tsc[q * 32 + lane] = tok < tl.rows ? a.sa[int64_t(tl.row0) + tok] : 0.0f;
      } else {
#pragma unroll
        for (int p = 0; p < P::NGRP; ++p)
          sal[p] = p * 32 + lane < tl.rows ? a.sa[int64_t(tl.row0) + p * 32 + lane] : 0.0f;
      }
      bool okw = __all_sync(0xffffffffu, mbar_wait<500>(bar(P::B_ACC_FULL), ii & 1, abort_flag));
      if (okw) okw = __all_sync(0xffffffffu, mbar_wait(bar(P::B_NORM_READY + b), par, abort_flag));
      // the four warps of a triple take one decision (every one of them
      // reaches this barrier), so none is left at the triple's barriers below
      if (!(BOX ? named_sync_and(1 + trip, 128, okw) : okw)) {
        fail();
        break;
      }
      tc_fence_after();
      // a row's norm is at most the sum of the groups' largest partial norms
      long long nw = 0;
#pragma unroll
      for (int c = 0; c < NCG; ++c) nw += norm[NCG * b + c];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P::B_NORM_READ + b));
      if (warp == WARP_EPI && lane == 0) {
        // once every epilogue warp has read the norm, clear it for the
        // item after next and hand the slot back to the converters
        if (mbar_wait(bar(P::B_NORM_READ + b), par, abort_flag)) {
          for (int c = 0; c < NCG; ++c) norm[NCG * b + c] = 0;
          mbar_arrive(bar(P::B_NORM_FREE + b));
        } else {
          fail();
        }
      }
      if (nw * (long long)tmax >= (1ll << 48) && q == 0 && lane == 0) atomicExch(redo, 1);
      const int nm = nmma_of(tl.rows);
      const uint32_t taddr = tmem + (uint32_t(q * 32) << 16);
#pragma unroll 1
      for (int p = trip; p < P::NGRP; p += NTRIP) {
        if (p * 32 >= nm) break;
        uint32_t v[32];
        tmem_ld32(taddr + 32u * p, v);
        const int tok0 = p * 32;
        float sp = sal[0];  // sal[p] without a dynamic register index
        if constexpr (!BOX) {
#pragma unroll
          for (int m = 1; m < P::NGRP; ++m) sp = p == m ? sal[m] : sp;
        }
        tmem_wait_ld();
        const int lim = min(32, tl.rows - tok0);
        if constexpr (BOX) {
          if (a.out_type != WQ_OUT_I32) {
            // (v * sa) * sw for token pairs in packed products, rounded to
            // bf16 pairs; the group's token scales are shared-memory broadcasts
            const float *ts = tsc + ((p - trip) / NTRIP) * 32;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 s2 = *reinterpret_cast<const float2 *>(ts + 2 * i);
              float x0 = __uint_as_float(v[2 * i]), x1 = __uint_as_float(v[2 * i + 1]);
              fmul2(x0, x1, s2.x, s2.y);
              fmul2(x0, x1, swn, swn);
              pk[i] = bf16x2_rn(x0, x1);
            }
            if (lim < 32) {
              uint16_t *o = static_cast<uint16_t *>(a.out) + (int64_t(tl.row0) + tok0) * a.N + n;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < lim) o[int64_t(j) * a.N] = uint16_t(pk[j >> 1] >> ((j & 1) * 16));
            } else {
              // a full group: the triple writes its 32 x 128 box, the leader
              // stores it once every warp has written and fenced its part
              if (leader) bulk_wait_read_all();  // the previous box has been read out
              named_sync(1 + trip, 128);
              uint16_t *col = box + q * 32 + lane;
#pragma unroll
              for (int j = 0; j < 32; ++j) col[j * WM] = uint16_t(pk[j >> 1] >> ((j & 1) * 16));
              fence_async_smem();
              named_sync(1 + trip, 128);
              if (leader) {
                tma_store_2d(&tmO, box_s, wb * WM, tl.row0 + tok0);
                bulk_commit();
              }
            }
            continue;
          }
        }
        if (a.out_type == WQ_OUT_I32) {
          int32_t *o = static_cast<int32_t *>(a.out) + (int64_t(tl.row0) + tok0) * a.N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < lim) o[int64_t(j) * a.N] = __float2int_rn(__uint_as_float(v[j]));
        } else if (!BOX || lim < 32) {
          uint16_t *o = static_cast<uint16_t *>(a.out) + (int64_t(tl.row0) + tok0) * a.N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float s = __shfl_sync(0xffffffffu, sp, j);
            if (j < lim)
              o[int64_t(j) * a.N] = f_to_bf16(__fmul_rn(__fmul_rn(__uint_as_float(v[j]), s), swn));
          }
        } else {
          // a full group: the triple writes its 32 x 128 box, the leader
          // stores it once every warp has written and fenced its part
          if (leader) bulk_wait_read_all();  // the previous box has been read out
          named_sync(1 + trip, 128);
          uint16_t *col = box + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float s = __shfl_sync(0xffffffffu, sp, j);
            col[j * WM] = f_to_bf16(__fmul_rn(__fmul_rn(__uint_as_float(v[j]), s), swn));
          }
          fence_async_smem();
          named_sync(1 + trip, 128);
          if (leader) {
            tma_store_2d(&tmO, box_s, wb * WM, tl.row0 + tok0);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P::B_ACC_EMPTY));
    }
    if (BOX && leader) bulk_wait_all();  // every box store has landed before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no multicast copy or completion targets either CTA after this
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool gemm_tc5_supported(const GemmArgs &a) {
  return a.A16 != nullptr && a.a_norm2 != nullptr && a.scheme == WQ_SCHEME_CHANNEL &&
         acc_modes_agree(a) && a.N % (2 * WM) == 0 && a.K % BK == 0 && a.K <= 65536 &&
         a.E * a.N < (int64_t(1) << 31) && a.R < (int64_t(1) << 31) && tma_available() &&
         num_sms() >= 2;
}

// 384-token items when the experts average more than 320 rows (fewer items,
// each expert's weights streamed fewer times), else 320-token items with
// the shared-memory output boxes
static bool tc5_wide(const GemmArgs &a) {
  // (the masked layout's row count includes its invalid rows: the box plan)
  return a.masked_m == nullptr && int64_t(a.R) > 320 * int64_t(a.E);
}

int gemm_tc5_tile_rows(const GemmArgs &a) { return tc5_wide(a) ? 384 : 320; }

template <int TN, bool BOX>
static int launch_tc5(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                      int32_t *redo, cudaStream_t st) {
  using P = Tc5Plan<TN, BOX>;
  CUtensorMap mW, mO;
  TokenMaps<TN> mT;
  // the output box map: bf16 [R][N]; the direct-store plan and int32 output
  // never use it (the same rows read as 16-bit values stay inside the buffer)
  static_assert(BK == 64, "one 64-byte-swizzled row of weight codes per K stage");
  if (!make_tma_2d_u8_sw64(&mW, a.W, int64_t(a.E) * a.N, a.K, WM) ||
      !make_tma_2d_b16(&mO, a.out, a.R, a.N, WM, 32))
    return WQ_ERR_LAUNCH;
  for (int i = 0; i < TokenMaps<TN>::N; ++i)
    if (!make_tma_2d_b16_sw128(&mT.m[i], a.A16, a.R, a.K, 8 * (i + 1))) return WQ_ERR_LAUNCH;
  static bool attr = false;
  static int pairs_resident = 0;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc5_kernel<TN, BOX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             P::SMEM_BYTES) != cudaSuccess)
      return WQ_ERR_LAUNCH;
    // a persistent grid must be fully co-resident: ask how many 2-CTA
    // clusters of this kernel fit at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * (num_sms() / 2)));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = P::SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc5_kernel<TN, BOX>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    pairs_resident = n;
    attr = true;
  }
  const int64_t max_items = int64_t(max_tiles) * (a.N / (2 * WM));
  const int pairs = int(max_items < pairs_resident ? max_items : pairs_resident);
  gemm_tc5_kernel<TN, BOX><<<2 * pairs, NTHREADS, P::SMEM_BYTES, st>>>(mW, mT, mO, a, tiles,
                                                                      ntiles, redo);
  return launched(1);
}

// `tiles` holds token tiles of at most gemm_tc5_tile_rows(a) rows.
int launch_gemm_tc5(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    int32_t *redo, cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  return tc5_wide(a) ? launch_tc5<384, false>(a, tiles, ntiles, max_tiles, redo, st)
                     : launch_tc5<320, true>(a, tiles, ntiles, max_tiles, redo, st);
}

}  // namespace wq
