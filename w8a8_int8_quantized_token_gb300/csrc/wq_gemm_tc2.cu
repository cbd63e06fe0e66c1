// Grouped W8A8 GEMM, int32-accumulator fast engine (tcgen05, sm_103a).
//
// The channel-wise INT8 GEMM of "[Feature] DeepSeek V3/R1 INT8 Quantization
// (channel-wise)" with the int32 accumulator: C = A_e W_e^T exactly, then
// v = (float(C) * sa[r]) * sw[e][n].  Codes are widened to fp16 (exact) and
// multiplied by tcgen05.mma kind::f16 with float32 accumulation in tensor
// memory over the whole K range in one pass.  That single pass is exact when
// every partial sum stays an integer of magnitude below 2^24; by the
// Cauchy-Schwarz inequality every partial sum of a row a and a channel w is
// at most ||a||_2 ||w||_2 in magnitude, so the converter warps accumulate the
// squared norms of all rows and channels of a tile (dp4a) while they widen
// the codes, and the epilogue checks  max||a||^2 * max||w||^2 < 2^48.
// A tile that fails the check raises a device flag; the chunked exact engine
// (wq_gemm_tc.cu) then recomputes the whole launch.  Realistic activations
// and weights pass with a wide margin (||a|| ||w|| ~ 1e6).
//
// Operand roles are swapped relative to the row-major problem: the MMA's
// M = 128 rows are output channels (weights, A operand) and its N = 16..256
// columns are tokens (B operand), so a ragged expert wastes at most 15 token
// columns.  Persistent CTAs; work item = (token tile <= 256 rows of one expert)
// x (128 output channels), handed out dynamically: a CTA starts with item
// blockIdx.x and claims each further item from a global counter
// (gridDim.x + atomicAdd), so CTAs that drew short items take more of them;
// the producer posts the claimed indices into a small ring in shared memory,
// from which every role reads the same sequence.  Two tensor-memory
// accumulators (columns [0,256) and [256,512)) let the epilogue of one item
// overlap the MMAs of the next.
//   warp 0      item claims and TMA producer (weights 128 x 64, tokens box x 64 int8)
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-9   converters (two groups taking alternate K stages): int8 ->
//               fp16 (128-byte swizzled K-major) + squared row norms
//   warps 10-13 epilogue: dequant, bf16, coalesced stores (32 channels/warp)
//   warp 14     (fp16 token form only) token TMA producer
// In the fp16 token form (GemmArgs::tok16, 256-token plan) the token tiles
// arrive as fp16 codes by TMA, 128-byte swizzled, in a ring of their own, and
// the converters widen only the weights: a token tile is no longer widened
// again for each of the N / 128 weight blocks.  The token rows' squared
// norms then come with them (a_norm2), or are not needed (int4 weights).
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int WM = 128, BK = 64;
constexpr int NTHREADS = 448;   // 480 in the fp16 token form (the token producer warp)
constexpr int WARP_TOKP = 14;   // token producer warp of the fp16 token form
constexpr int NCONV = 256;  // converter threads: two groups of 128
constexpr int GCONV = 128;  // threads of one converter group (its stages alternate with the other's)
constexpr int NR = 8;       // item ring depth
// readers of each posted item: the MMA thread, the eight converter warps and
// the four epilogue warps (one arrival each)
constexpr int ITEM_READERS = 1 + NCONV / 32 + 4;

// Shared-memory plan of one instantiation: TN = most tokens per item (MMA N),
// S8 / S16 = depths of the int8 staging ring and of the fp16 ring.  Large
// TN suits many rows per expert (prefill); a small TN with a deep int8 ring
// keeps enough weight bytes in flight when experts hold a few tokens each
// (decode), where the GEMM streams weights from HBM.
template <int TN, int S8, int S16, bool W4, bool FT = false, int STK = 0>
struct Plan {
  // bytes per stage: W8 the staged weight codes (int8, or int4 two per byte),
  // T8 the int8 token codes; W16 / T16 the widened fp16 tiles.  FT: the fp16
  // token form, whose STK-deep token ring holds TK16-byte fp16 tiles loaded
  // by TMA (no int8 token staging, no widened token tile in the fp16 ring)
  static_assert(FT == (STK > 0), "a token ring exactly in the fp16 token form");
  static constexpr int W8 = WM * BK / (W4 ? 2 : 1), T8 = FT ? 0 : TN * BK;
  static constexpr int W16 = 2 * WM * BK, T16 = 2 * T8, TK16 = FT ? 2 * TN * BK : 0;
  static constexpr int ST8 = W8 + T8, ST16 = W16 + T16;
  static constexpr int OFF_F16 = 0;
  // every stage size is a multiple of 1024 bytes, so each token stage starts
  // 1024-aligned, as the 128-byte swizzle of its TMA copy requires
  static constexpr int OFF_TOK = OFF_F16 + S16 * ST16;
  static constexpr int OFF_I8 = OFF_TOK + STK * TK16;
  static constexpr int OFF_BAR = OFF_I8 + S8 * ST8;
  static constexpr int B_S8_FULL = 0, B_S8_EMPTY = S8, B_F16_FULL = 2 * S8,
                       B_F16_EMPTY = 2 * S8 + S16, B_ACC_FULL = 2 * S8 + 2 * S16,  // [2]
      B_ACC_EMPTY = B_ACC_FULL + 2,                                                // [2]
      B_NORM_READY = B_ACC_FULL + 4,                                               // [2]
      B_NORM_FREE = B_ACC_FULL + 6,                                                // [2]
      B_NORM_READ = B_ACC_FULL + 8,                                                // [2]
      B_MMA_DONE = B_ACC_FULL + 10,
                       B_ITEM_FULL = B_ACC_FULL + 11,   // [NR] a claimed item index posted
      B_ITEM_EMPTY = B_ITEM_FULL + NR,                 // [NR] every role has read it
      B_TOK_FULL = B_ITEM_EMPTY + NR,                  // [STK] fp16 token tile landed
      B_TOK_EMPTY = B_TOK_FULL + STK,                  // [STK] its MMAs are done
      NBAR = B_TOK_EMPTY + STK;
  // int32 [2 buffers][2 converter groups][weights, tokens]
  static constexpr int OFF_NORM = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ITEMS = OFF_NORM + 32;  // int32 [NR] item ring
  static constexpr int OFF_TMEM = OFF_ITEMS + NR * 4;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
  static constexpr int NJW = WM * 4 / GCONV;  // weight 16-byte pieces per converter thread
  // token 16-byte pieces per converter thread (none in the fp16 token form)
  static constexpr int NJT = FT ? 0 : TN * 4 / GCONV;
  static_assert(FT || (NJT >= 1 && TN * 4 == NJT * GCONV), "token tile must fill a converter group");
  static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
};

__device__ __forceinline__ int sq4(uint32_t w, int acc) { return __dp4a(int(w), int(w), acc); }

// TG: the token rows' squared norms come in a.a_norm2 (int8 weights only),
// so the converters sum only the weight rows'.  FT: the fp16 token form, its
// token maps (tmT16/64/256) describing a.tok16; STK its token ring depth.
template <int TN, int S8, int S16, bool W4, bool TG, bool FT = false, int STK = 0>
__global__ void __launch_bounds__(FT ? NTHREADS + 32 : NTHREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT16,
                    const __grid_constant__ CUtensorMap tmT64,
                    const __grid_constant__ CUtensorMap tmT256, const GemmArgs a,
                    const Tile *__restrict__ tiles, const int32_t *__restrict__ ntiles,
                    int32_t *__restrict__ redo, int32_t *__restrict__ claim) {
  static_assert(!FT || TG || W4, "the fp16 token form sums no token norms");
  using P = Plan<TN, S8, S16, W4, FT, STK>;
  constexpr int W8 = P::W8, W16 = P::W16, ST8 = P::ST8, ST16 = P::ST16, TK16 = P::TK16;
  constexpr int OFF_TOK = P::OFF_TOK, B_TOK_FULL = P::B_TOK_FULL, B_TOK_EMPTY = P::B_TOK_EMPTY;
  constexpr int READERS = ITEM_READERS + (FT ? 1 : 0);
  constexpr int OFF_F16 = P::OFF_F16, OFF_I8 = P::OFF_I8, OFF_BAR = P::OFF_BAR;
  constexpr int B_S8_FULL = P::B_S8_FULL, B_S8_EMPTY = P::B_S8_EMPTY, B_F16_FULL = P::B_F16_FULL,
                B_F16_EMPTY = P::B_F16_EMPTY, B_ACC_FULL = P::B_ACC_FULL,
                B_ACC_EMPTY = P::B_ACC_EMPTY, B_NORM_READY = P::B_NORM_READY,
                B_NORM_FREE = P::B_NORM_FREE, B_NORM_READ = P::B_NORM_READ,
                B_MMA_DONE = P::B_MMA_DONE, B_ITEM_FULL = P::B_ITEM_FULL,
                B_ITEM_EMPTY = P::B_ITEM_EMPTY;
  constexpr int OFF_NORM = P::OFF_NORM, OFF_TMEM = P::OFF_TMEM, OFF_ABORT = P::OFF_ABORT;
  constexpr int NJW = P::NJW, NJT = P::NJT;
  extern __shared__ uint8_t smem_raw[];
  const int NB = int(a.N / WM);
  const int items = ntiles[0] * NB;
  if (int(blockIdx.x) >= items) return;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_ABORT);
  volatile int *norm = reinterpret_cast<volatile int *>(sm + OFF_NORM);
  volatile int *item_ring = reinterpret_cast<volatile int *>(sm + P::OFF_ITEMS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = int(a.K / BK);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 8; ++i) norm[i] = 0;
    for (int s = 0; s < S8; ++s) {
      mbar_init(bar(B_S8_FULL + s), 1);
      mbar_init(bar(B_S8_EMPTY + s), GCONV / 32);
    }
    for (int s = 0; s < S16; ++s) {
      mbar_init(bar(B_F16_FULL + s), GCONV / 32);
      mbar_init(bar(B_F16_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_ACC_FULL + b), 1);
      mbar_init(bar(B_ACC_EMPTY + b), 4);
      mbar_init(bar(B_NORM_READY + b), NCONV / 32);
      mbar_init(bar(B_NORM_FREE + b), 1);
      mbar_init(bar(B_NORM_READ + b), 4);
    }
    mbar_init(bar(B_MMA_DONE), 1);
    for (int r = 0; r < NR; ++r) {
      mbar_init(bar(B_ITEM_FULL + r), 1);
      mbar_init(bar(B_ITEM_EMPTY + r), READERS);
    }
    for (int s = 0; s < STK; ++s) {
      mbar_init(bar(B_TOK_FULL + s), 1);
      mbar_init(bar(B_TOK_EMPTY + s), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(a.status, WQ_ERR_TIMEOUT);
  };
  // token box height for a tile of `rows` tokens, and the MMA's N
  auto nmma_of = [](int rows) { return (rows + 15) & ~15; };
  auto box_of = [](int nmma) { return nmma <= 16 ? 16 : (nmma <= 64 || TN <= 64 ? 64 : 256); };
  // the r-th item of this CTA (-1: none left), read from the ring by every
  // thread of a role; the caller then arrives once per warp on ITEM_EMPTY
  auto read_item = [&](int r, int &it) {
    if (!mbar_wait(bar(B_ITEM_FULL + r % NR), (r / NR) & 1, abort_flag)) return false;
    it = item_ring[r % NR];
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      int it = blockIdx.x;  // the first item is the CTA's own; later ones are claimed
      for (int r = 0; ok; ++r) {
        const int s = r % NR;
        if (!mbar_wait<200>(bar(B_ITEM_EMPTY + s), ((r / NR) & 1) ^ 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        item_ring[s] = it < items ? it : -1;
        mbar_arrive(bar(B_ITEM_FULL + s));
        if (it >= items) break;
        const int next = int(gridDim.x) + atomicAdd(claim, 1);  // claimed while this item streams
        const Tile tl = tiles[it / NB];
        const int wb = it % NB;
        const int box = box_of(nmma_of(tl.rows));
        const CUtensorMap *tmT = box == 16 ? &tmT16 : (box == 64 ? &tmT64 : &tmT256);
        const uint32_t tx = W8 + (FT ? 0 : box * BK);
        const int wrow = int(int64_t(tl.expert) * a.N + int64_t(wb) * WM);
        for (int i = 0; i < KT; ++i, ++g) {
          const int s8 = g % S8;
          if (!mbar_wait<200>(bar(B_S8_EMPTY + s8), ((g / S8) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t dst = base + OFF_I8 + uint32_t(s8) * ST8;
          mbar_expect_tx(bar(B_S8_FULL + s8), tx);
          tma_load_2d(dst, &tmW, i * (W4 ? BK / 2 : BK), wrow, bar(B_S8_FULL + s8));  // bytes
          if constexpr (!FT) tma_load_2d(dst + W8, tmT, i * BK, tl.row0, bar(B_S8_FULL + s8));
        }
        it = next;
      }
      if (!ok) {
        for (int j = g > S8 ? g - S8 : 0; j < g; ++j)
          mbar_wait_bounded(bar(B_S8_FULL + j % S8), (j / S8) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int ii = 0; ok; ++ii) {
        int it;
        if (!read_item(ii, it)) {
          fail();
          break;
        }
        mbar_arrive(bar(B_ITEM_EMPTY + ii % NR));
        if (it < 0) break;
        const Tile tl = tiles[it / NB];
        const uint32_t idesc = idesc_f16(WM, nmma_of(tl.rows));
        const int b = ii & 1;
        if (!mbar_wait(bar(B_ACC_EMPTY + b), ((ii >> 1) & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        const uint32_t d = tmem + uint32_t(b) * 256u;
        for (int i = 0; i < KT; ++i, ++g) {
          const int s = g % S16;
          constexpr int SKD = FT ? STK : 1;  // token ring depth (no ring: unused)
          const int sk = g % SKD;
          if (!mbar_wait(bar(B_F16_FULL + s), (g / S16) & 1, abort_flag) ||
              (FT && !mbar_wait(bar(B_TOK_FULL + sk), (g / SKD) & 1, abort_flag))) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w0 = base + OFF_F16 + uint32_t(s) * ST16;
          const uint32_t t0 = FT ? base + OFF_TOK + uint32_t(sk) * TK16 : w0 + W16;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16(d, sdesc(w0 + 32u * kk), sdesc(t0 + 32u * kk), idesc, (i | kk) ? 1u : 0u);
          mma_commit(bar(B_F16_EMPTY + s));
          if constexpr (FT) mma_commit(bar(B_TOK_EMPTY + sk));
        }
        if (ok) mma_commit(bar(B_ACC_FULL + b));
      }
      mma_commit(bar(B_MMA_DONE));
      mbar_wait_bounded(bar(B_MMA_DONE), 0);
    }
  } else if (warp < 2 + NCONV / 32) {
    // ------------------------------------------------------------ converters
    // Two groups of four warps; group `grp` widens the stages of parity grp
    // (K / 64 is even), so two stages are in flight through the converters.
    const int grp = (warp - 2) >> 2;
    const int t = threadIdx.x - 64 - grp * GCONV;  // 0..127 within the group
    int gbase = 0;
    bool ok = true;
    for (int ii = 0; ok; ++ii, gbase += KT) {
      int it;
      if (!__all_sync(0xffffffffu, read_item(ii, it))) {
        fail();
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ITEM_EMPTY + ii % NR));
      if (it < 0) break;
      const Tile tl = tiles[it / NB];
      const int box = box_of(nmma_of(tl.rows));
      const int tchunks = box * 4;  // 16-byte pieces of the token tile
      int nrm[NJW + NJT];
#pragma unroll
      for (int j = 0; j < NJW + NJT; ++j) nrm[j] = 0;
      for (int i = grp; i < KT; i += 2) {
        const int g = gbase + i;
        const int s8 = g % S8, s16 = g % S16;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S8_FULL + s8), (g / S8) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        const uint8_t *src = sm + OFF_I8 + s8 * ST8;
        uint4 v[NJW + NJT];
        if constexpr (W4) {
          // packed piece c4 = 32 codes: row c4 >> 1, codes 32 * (c4 & 1) onwards
#pragma unroll
          for (int j = 0; j < NJW / 2; ++j) {
            const uint4 p = *reinterpret_cast<const uint4 *>(src + (j * GCONV + t) * 16);
            s4x8_to_s8x8(p.x, v[2 * j].x, v[2 * j].y);
            s4x8_to_s8x8(p.y, v[2 * j].z, v[2 * j].w);
            s4x8_to_s8x8(p.z, v[2 * j + 1].x, v[2 * j + 1].y);
            s4x8_to_s8x8(p.w, v[2 * j + 1].z, v[2 * j + 1].w);
          }
        } else {
#pragma unroll
          for (int j = 0; j < NJW; ++j)
            v[j] = *reinterpret_cast<const uint4 *>(src + (j * GCONV + t) * 16);
        }
#pragma unroll
        for (int j = NJW; j < NJW + NJT; ++j) {
          const int c = (j - NJW) * GCONV + t;
          v[j] = c < tchunks ? *reinterpret_cast<const uint4 *>(src + W8 + c * 16)
                             : make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();  // these reads before the next copy into the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_S8_EMPTY + s8));
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(B_F16_EMPTY + s16), ((g / S16) & 1) ^ 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        uint8_t *dst = sm + OFF_F16 + s16 * ST16;
#pragma unroll
        for (int j = 0; j < NJW + NJT; ++j) {
          const int c = (j < NJW ? j : j - NJW) * GCONV + t;
          if (j < NJW || c < tchunks) {
            // 16 int8 codes: row and 16-code part within the 64-code stage row
            int row = c >> 2, part = c & 3;
            if (W4 && j < NJW) {
              const int c4 = (j >> 1) * GCONV + t;
              row = c4 >> 1;
              part = 2 * (c4 & 1) + (j & 1);
            }
            store_f16_row_piece(dst + (j < NJW ? 0 : W16) + row * 128, row, part, v[j]);
            // squared norms of the weight rows, and of the token rows unless
            // the caller gave them (then the epilogue reads those).  The int4
            // form needs none: with |w| <= 7 and K <= 16384 every partial
            // sum stays below 127 * 7 * 16384 < 2^24, exact in float32.
            if (!W4 && (j < NJW || !TG))
              nrm[j] += sq4(v[j].w, sq4(v[j].z, 0)) + sq4(v[j].y, sq4(v[j].x, 0));
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_F16_FULL + s16));
      }
      if (!ok) break;
      // squared norms over this group's stages: the 4 lanes 4m..4m+3 hold the
      // 4 pieces of one row; a row's full norm is at most the sum of the two
      // groups' largest partial norms, which is what the epilogue checks
      int wmax = 0, tmax = 0;
#pragma unroll
      for (int j = 0; j < NJW + NJT; ++j) {
        if (W4 && j < NJW) {
          // int4: a row's 64 codes of a stage are the two pieces of one
          // thread and its neighbour t ^ 1
          if (j & 1) continue;
          int n2 = nrm[j] + nrm[j + 1];
          n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
          wmax = max(wmax, n2);
          continue;
        }
        int n2 = nrm[j];
        n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
        n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
        if (j < NJW) {
          wmax = max(wmax, n2);
        } else {
          const int row = ((j - NJW) * GCONV + t) >> 2;
          if (row < tl.rows) tmax = max(tmax, n2);
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
        tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      }
      const int b = ii & 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar(B_NORM_FREE + b), ((ii >> 1) & 1) ^ 1, abort_flag))) {
        fail();
        break;
      }
      if (lane == 0) {
        atomicMax(const_cast<int *>(norm + 4 * b + 2 * grp), wmax);
        atomicMax(const_cast<int *>(norm + 4 * b + 2 * grp + 1), tmax);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_NORM_READY + b));
    }
  } else if (warp == WARP_TOKP) {
    // ------------------------------------------------------------ token producer
    // (fp16 token form): each item's K stages of fp16 token tiles, as deep
    // ahead as the token ring allows, independent of the weight ring
    if constexpr (FT) {
      if (lane == 0) {
        int gt = 0;
        bool ok = true;
        for (int ii = 0; ok; ++ii) {
          int it;
          if (!read_item(ii, it)) {
            fail();
            break;
          }
          mbar_arrive(bar(B_ITEM_EMPTY + ii % NR));
          if (it < 0) break;
          const Tile tl = tiles[it / NB];
          const int box = box_of(nmma_of(tl.rows));
          const CUtensorMap *tmT = box == 16 ? &tmT16 : (box == 64 ? &tmT64 : &tmT256);
          const uint32_t tx = uint32_t(box) * BK * 2;
          for (int i = 0; i < KT; ++i, ++gt) {
            const int sk = gt % STK;
            if (!mbar_wait<200>(bar(B_TOK_EMPTY + sk), ((gt / STK) & 1) ^ 1, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            mbar_expect_tx(bar(B_TOK_FULL + sk), tx);
            tma_load_2d(base + OFF_TOK + uint32_t(sk) * TK16, tmT, i * BK, tl.row0,
                        bar(B_TOK_FULL + sk));
          }
        }
        if (!ok) {
          for (int j = gt > STK ? gt - STK : 0; j < gt; ++j)
            mbar_wait_bounded(bar(B_TOK_FULL + j % STK), (j / STK) & 1);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quarter of this warp
    for (int ii = 0;; ++ii) {
      int it;
      if (!__all_sync(0xffffffffu, read_item(ii, it))) {
        fail();
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ITEM_EMPTY + ii % NR));
      if (it < 0) break;
      const Tile tl = tiles[it / NB];
      const int wb = it % NB;
      const int b = ii & 1, par = (ii >> 1) & 1;
      // the item's token scales (lane j of group p holds token 32p + j) and
      // this thread's weight scale, loaded while the item's MMAs still run
      constexpr int NGRP = TN / 32;
      const int64_t n = int64_t(wb) * WM + q * 32 + lane;  // this thread's output channel
      const float swn = a.sw[int64_t(tl.expert) * a.N + n];
      float sal[NGRP];
#pragma unroll
      for (int p = 0; p < NGRP; ++p)
        sal[p] = p * 32 + lane < tl.rows ? a.sa[int64_t(tl.row0) + p * 32 + lane] : 0.0f;
      // given token-row norms: the item's largest, also read while the MMAs run
      int tgiven = 0;
      if constexpr (TG) {
        for (int r = lane; r < tl.rows; r += 32) tgiven = max(tgiven, a.a_norm2[int64_t(tl.row0) + r]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tgiven = max(tgiven, __shfl_xor_sync(0xffffffffu, tgiven, o));
      }
      if (!__all_sync(0xffffffffu, mbar_wait<500>(bar(B_ACC_FULL + b), par, abort_flag)) ||
          !__all_sync(0xffffffffu, mbar_wait(bar(B_NORM_READY + b), par, abort_flag))) {
        fail();
        break;
      }
      tc_fence_after();
      const long long nw = (long long)norm[4 * b] + norm[4 * b + 2];
      const long long nt =
          TG ? (long long)tgiven : (long long)norm[4 * b + 1] + norm[4 * b + 3];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_NORM_READ + b));
      if (warp == 10 && lane == 0) {
        // once all four epilogue warps have read the norms, clear them for the
        // item after next and hand the slots back to the converters
        if (mbar_wait(bar(B_NORM_READ + b), par, abort_flag)) {
          for (int i = 0; i < 4; ++i) norm[4 * b + i] = 0;
          mbar_arrive(bar(B_NORM_FREE + b));
        } else {
          fail();
        }
      }
      if (!W4 && nw * nt >= (1ll << 48) && q == 0 && lane == 0) atomicExch(redo, 1);
      const int nmma = nmma_of(tl.rows);
      const uint32_t taddr = tmem + (uint32_t(q * 32) << 16) + uint32_t(b) * 256u;
#pragma unroll 1
      for (int p = 0; p < NGRP; ++p) {
        if (p * 32 >= nmma) break;
        uint32_t v[32];
        tmem_ld32(taddr + 32u * p, v);
        const int tok0 = p * 32;
        float sp = sal[0];  // sal[p] without a dynamic register index
#pragma unroll
        for (int m = 1; m < NGRP; ++m) sp = p == m ? sal[m] : sp;
        tmem_wait_ld();
        const int lim = min(32, tl.rows - tok0);
        if (a.out_type == WQ_OUT_I32) {
          int32_t *o = static_cast<int32_t *>(a.out) + (int64_t(tl.row0) + tok0) * a.N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < lim) o[int64_t(j) * a.N] = __float2int_rn(__uint_as_float(v[j]));
        } else {
          uint16_t *o = static_cast<uint16_t *>(a.out) + (int64_t(tl.row0) + tok0) * a.N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float s = __shfl_sync(0xffffffffu, sp, j);
            if (j < lim)
              o[int64_t(j) * a.N] = f_to_bf16(__fmul_rn(__fmul_rn(__uint_as_float(v[j]), s), swn));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY + b));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool gemm_tc2_supported(const GemmArgs &a) {
  return a.scheme == WQ_SCHEME_CHANNEL && acc_modes_agree(a) && a.N % WM == 0 &&
         a.K % BK == 0 && a.K <= 65536 && a.E * a.N < (int64_t(1) << 31) &&
         a.R < (int64_t(1) << 31) && tma_available();
}

// Token-tile height the engine uses for this launch: 64 when experts hold few
// rows on average (decode-like), else 256.
int gemm_tc2_tile_rows(const GemmArgs &a) {
  const int64_t rows = a.masked_m ? int64_t(a.E) * a.Mmax : a.R;
  return rows <= int64_t(64) * a.E ? 64 : 256;
}

template <int TN, int S8, int S16, bool W4, bool TG = false, bool FT = false, int STK = 0>
int launch_tc2(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
               int32_t *redo, cudaStream_t st) {
  using P = Plan<TN, S8, S16, W4, FT, STK>;
  constexpr int NT = FT ? NTHREADS + 32 : NTHREADS;
  CUtensorMap mW, m16, m64, m256;
  // int4 weights: K / 2 bytes a row, a 32-byte box per 64-code stage
  if (!make_tma_2d_u8(&mW, a.W, int64_t(a.E) * a.N, W4 ? a.K / 2 : a.K, W4 ? BK / 2 : BK, WM))
    return WQ_ERR_LAUNCH;
  if (FT) {  // fp16 token tiles, 128-byte swizzled as the MMA reads them
    if (!make_tma_2d_b16_sw128(&m16, a.tok16, a.R, a.K, 16) ||
        !make_tma_2d_b16_sw128(&m64, a.tok16, a.R, a.K, 64) ||
        !make_tma_2d_b16_sw128(&m256, a.tok16, a.R, a.K, TN > 64 ? 256 : 64))
      return WQ_ERR_LAUNCH;
  } else if (!make_tma_2d_u8(&m16, a.A, a.R, a.K, BK, 16) ||
             !make_tma_2d_u8(&m64, a.A, a.R, a.K, BK, 64) ||
             !make_tma_2d_u8(&m256, a.A, a.R, a.K, BK, TN > 64 ? 256 : 64)) {
    return WQ_ERR_LAUNCH;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc2_kernel<TN, S8, S16, W4, TG, FT, STK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_BYTES) != cudaSuccess)
      return WQ_ERR_LAUNCH;
    attr = true;
  }
  const int64_t max_items = int64_t(max_tiles) * (a.N / WM);
  const int grid = int(max_items < num_sms() ? max_items : num_sms());
  // redo[1] is the item counter (zeroed with the flag by the tile builder)
  gemm_tc2_kernel<TN, S8, S16, W4, TG, FT, STK><<<grid, NT, P::SMEM_BYTES, st>>>(mW, m16, m64, m256, a,
                                                                          tiles, ntiles, redo,
                                                                          redo + 1);
  return launched(1);
}

// `tiles` must be built with gemm_tc2_tile_rows(a) rows per tile.
int launch_gemm_tc2(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    int32_t *redo, cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  const bool small = gemm_tc2_tile_rows(a) == 64;
  // fp16 token form: 256-token plan, token norms given (int8 weights) or not
  // needed (int4)
  if (a.tok16 != nullptr && !small) {
    if (a.w4) return launch_tc2<256, 4, 4, true, false, true, 4>(a, tiles, ntiles, max_tiles, redo, st);
    if (a.a_norm2 != nullptr)
      return launch_tc2<256, 4, 4, false, true, true, 4>(a, tiles, ntiles, max_tiles, redo, st);
  }
  if (a.w4) {
    return small ? launch_tc2<64, 8, 4, true>(a, tiles, ntiles, max_tiles, redo, st)
                 : launch_tc2<256, 3, 3, true>(a, tiles, ntiles, max_tiles, redo, st);
  }
  if (small) return launch_tc2<64, 8, 4, false>(a, tiles, ntiles, max_tiles, redo, st);
  // given token-row norms are used by the 256-token form only (the 64-token
  // form sums its own: correct either way, one instantiation fewer)
  return a.a_norm2 != nullptr ? launch_tc2<256, 3, 3, false, true>(a, tiles, ntiles, max_tiles, redo, st)
                              : launch_tc2<256, 3, 3, false>(a, tiles, ntiles, max_tiles, redo, st);
}

}  // namespace wq
