// Grouped W8A8 GEMM, block-wise scheme, for fp16-stored activation codes, on
// CTA pairs that share token tiles (tcgen05, sm_103a).
//
// The block-wise INT8 GEMM of the Meituan INT8 DeepSeek R1 article
// (量化技术的探索): weights quantized per [128,128] block, activations per
// token per 128-element group, float32 accumulation across the K blocks:
//   acc = 0;  for kb ascending:  acc = acc + float(C_kb) * (sa[r][kb] * sw[e][n/128][kb])
// with C_kb the integer product over K block kb.  C_kb is a sum of 128
// products of magnitude <= 127^2, an integer below 2^21, so the tensor core's
// float32 sum over one K block is exact in any order; the epilogue then takes
// the definition's float32 steps in order (every product and sum rounded to
// nearest, none fused).
//
// Same structure as the channel-wise pair engine: the two CTAs of a cluster
// share each token tile (each loads half of a token stage and multicasts it),
// each widens its own 128 weight channels, which are exactly one row of
// weight-scale blocks, to fp16 in shared memory.  MMA M = 128 channels, N = up
// to 160 tokens.  Each K block (two 64-wide stages) goes into one of two
// 160-column chunk accumulators in tensor memory while the epilogue drains
// the other: it scales the chunk column by column and adds it to a running
// sum held in tensor memory (columns [320, 480)), and after the last K block
// writes bf16.
//   warp 0      TMA producer of the int8 weights
//   warp 14     TMA producer of the tokens (half of each stage, multicast);
//               the two producers wait on separate rings, so weight copies
//               run up to SW8 stages ahead of the converters whatever the
//               token ring holds
// A K stage's widened weights and token slot are released together: one
// commit per stage, multicast to both CTAs' token-empty barriers, which the
// converters wait on as well (the two rings have the same depth).
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-5   converters: int8 weights -> fp16 (128-byte swizzled K-major)
//   warps 6-13  epilogue (two per tensor-memory lane quarter, alternate
//               32-column groups, so one warp's tensor-memory loads overlap
//               the other's arithmetic)
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int WM = 128, TN = 160, BK = 64;
constexpr int W8B = WM * BK, W16B = 2 * W8B;    // weight stage bytes
constexpr int TB = TN * BK * 2;                 // token stage bytes (fp16)
constexpr int NCH = 3;                          // chunk accumulators (tensor-memory columns [0, 3*TN))
constexpr int EPI_COLS = TN / 2;                // token columns each epilogue warp owns
constexpr int NEPI = 8;                         // epilogue warps
constexpr int KEEP = EPI_COLS / 2;              // fused: columns a thread finishes itself
constexpr int XW = KEEP / 2;                    // fused: bf16 pairs a thread sends to the peer

// Shared-memory plan.  The fused variant (SiLU-and-mul and re-quantization in
// the epilogue) adds an exchange area that the peer CTA writes, the group
// maxima of the four lane-quarter warps and their barriers, and gives up one
// int8 weight stage to make room.
template <bool FUSE>
struct Plan {
  static constexpr int ST = 4;                  // token ring depth (fp16 tokens)
  static constexpr int SW16 = ST;               // widened-weight ring depth
  static constexpr int SW8 = FUSE ? 7 : 8;      // int8 weight ring depth
  static constexpr int OFF_T = 0;
  static constexpr int OFF_W16 = OFF_T + ST * TB;
  static constexpr int OFF_W8 = OFF_W16 + SW16 * W16B;
  static constexpr int OFF_SC = OFF_W8 + SW8 * W8B;         // float [NEPI][EPI_COLS] column scales
  static constexpr int OFF_XCH = OFF_SC + NEPI * EPI_COLS * 4;  // uint32 [NEPI][32][XW]
  static constexpr int OFF_RED = OFF_XCH + (FUSE ? NEPI * 32 * XW * 4 : 0);  // float [2][2][4][KEEP]
  static constexpr int OFF_BAR = OFF_RED + (FUSE ? 2 * 2 * 4 * KEEP * 4 : 0);
  static constexpr int B_W8_FULL = 0, B_W8_EMPTY = SW8, B_W16_FULL = 2 * SW8,
                       B_T_FULL = 2 * SW8 + SW16, B_T_EMPTY = B_T_FULL + ST,
                       B_ACC_FULL = B_T_EMPTY + ST,  // [NCH]
      B_ACC_EMPTY = B_ACC_FULL + NCH,                // [NCH]
      B_MMA_DONE = B_ACC_FULL + 2 * NCH,
                       B_XF = B_MMA_DONE + 1,        // fused: [NEPI] peer's half arrived
      B_XE = B_XF + NEPI,                            // fused: [NEPI] peer has read our half
      B_RED = B_XE + NEPI,                           // fused: [2 item parities][2 halves]
      B_TEST = FUSE ? B_RED + 4 : B_MMA_DONE + 1,    // never completed (failure-path test)
      NBAR = B_TEST + 1;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
  static_assert(SW16 == ST, "a widened-weight slot is released with its token slot");
  static_assert(TB % 1024 == 0 && OFF_W16 % 1024 == 0 && OFF_W8 % 1024 == 0, "swizzle alignment");
  static_assert(OFF_XCH % 16 == 0 && OFF_BAR % 8 == 0, "exchange and barrier alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
};
static_assert(NCH * TN <= 512, "tensor memory plan");
static_assert(EPI_COLS % 16 == 0 && NEPI == 8, "each epilogue warp owns 16-column pieces");
static_assert(XW % 4 == 0, "the exchange goes in 16-byte pieces");
constexpr int NTHREADS = 480;
constexpr int WARP_TOK = 14;            // token producer
constexpr int GCONV = 128;              // threads of one converter group
constexpr int NJW = WM * 4 / GCONV;     // weight 16-byte pieces per converter thread

// (r0, r1) = (c0 + a0 * b0, c1 + a1 * b1), the product and the sum each
// rounded to nearest, never fused into one rounding: two scalar products and
// one packed float32 pair add.  (A packed product feeding a packed add was
// measured to come out fused on sm_103a; these mixed forms were measured
// bit-identical to separate scalar products and sums.)
__device__ __forceinline__ void mul_add2(float &r0, float &r1, float a0, float a1, float b0,
                                         float b1, float c0, float c1) {
  const float t0 = __fmul_rn(a0, b0), t1 = __fmul_rn(a1, b1);
  asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " add.rn.f32x2 z, x, y;\n mov.b64 {%0, %1}, z;\n}"
      : "=f"(r0), "=f"(r1)
      : "f"(c0), "f"(c1), "f"(t0), "f"(t1));
}

template <bool FUSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    gemm_tc6_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT8,
                    const __grid_constant__ CUtensorMap tmT32,
                    const __grid_constant__ CUtensorMap tmT80, const GemmArgs a,
                    const Tile *__restrict__ tiles, const int32_t *__restrict__ ntiles) {
  using P = Plan<FUSE>;
  constexpr int ST = P::ST, SW16 = P::SW16;
  constexpr int SW8 = P::SW8, OFF_T = P::OFF_T, OFF_W16 = P::OFF_W16, OFF_W8 = P::OFF_W8,
                OFF_SC = P::OFF_SC, OFF_BAR = P::OFF_BAR, OFF_TMEM = P::OFF_TMEM,
                OFF_ABORT = P::OFF_ABORT;
  constexpr int B_W8_FULL = P::B_W8_FULL, B_W8_EMPTY = P::B_W8_EMPTY, B_W16_FULL = P::B_W16_FULL,
                B_T_FULL = P::B_T_FULL, B_T_EMPTY = P::B_T_EMPTY, B_ACC_FULL = P::B_ACC_FULL,
                B_ACC_EMPTY = P::B_ACC_EMPTY, B_MMA_DONE = P::B_MMA_DONE;
  extern __shared__ uint8_t smem_raw[];
  const int NBP = int(a.N / (2 * WM));  // pairs of 128-row weight blocks
  const int items = ntiles[0] * NBP;
  const int pair = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  if (pair >= items) return;  // uniform over the pair, before any setup
  const uint32_t rank = cluster_ctarank();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_ABORT);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = int(a.K / BK);
  const int KB = KT / 2;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < SW8; ++s) {
      mbar_init(bar(B_W8_FULL + s), 1);
      mbar_init(bar(B_W8_EMPTY + s), GCONV / 32);
    }
    for (int s = 0; s < SW16; ++s) {
      mbar_init(bar(B_W16_FULL + s), GCONV / 32);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar(B_T_FULL + s), 1);   // local expect_tx; bytes from both CTAs' copies
      mbar_init(bar(B_T_EMPTY + s), 2);  // MMA completions of both CTAs
    }
    for (int b = 0; b < NCH; ++b) {
      mbar_init(bar(B_ACC_FULL + b), 1);
      mbar_init(bar(B_ACC_EMPTY + b), NEPI);
    }
    mbar_init(bar(B_MMA_DONE), 1);
    mbar_init(bar(P::B_TEST), 1);
    if constexpr (FUSE) {
      for (int w = 0; w < NEPI; ++w) {
        mbar_init(bar(P::B_XF + w), 1);  // one elected lane of the peer's warp
        mbar_init(bar(P::B_XE + w), 1);
      }
      for (int i = 0; i < 4; ++i) mbar_init(bar(P::B_RED + i), 4);  // the four lane quarters
    }
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
  // this CTA's 128-row weight block of item ip: adjacent blocks per pair, or
  // (fused) gate block p on rank 0 and the matching up block NBP + p on rank 1
  auto wblock = [&](int ip) {
    return FUSE ? ip % NBP + int(rank) * NBP : (ip % NBP) * 2 + int(rank);
  };
  // token rows each CTA of the pair loads for an MMA of width nmma
  auto box_of = [](int nmma) { return nmma <= 16 ? 8 : (nmma <= 64 ? 32 : 80); };

  if (a.wait_test) {
    // failure-path test: thread 0 waits on a barrier that nothing completes;
    // the bounded wait gives up, the kernel records WQ_ERR_TIMEOUT and every
    // role skips to the teardown before any copy or MMA is issued
    if (threadIdx.x == 0 && !mbar_wait(bar(P::B_TEST), 0, abort_flag)) fail();
  } else if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int g = 0, gw = 0;  // stage counter; weight stages issued
      bool ok = true;
      for (int ip = pair; ip < items && ok; ip += npairs) {
        const Tile tl = tiles[ip / NBP];
        const int wb = wblock(ip);
        const int wrow = int(int64_t(tl.expert) * a.N + int64_t(wb) * WM);
        for (int i = 0; i < KT; ++i, ++g) {
          const int sw = g % SW8;
          if (!mbar_wait<200>(bar(B_W8_EMPTY + sw), ((g / SW8) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(bar(B_W8_FULL + sw), W8B);
          tma_load_2d(base + OFF_W8 + uint32_t(sw) * W8B, &tmW, i * BK, wrow, bar(B_W8_FULL + sw));
          gw = g + 1;
        }
      }
      if (!ok) {  // let copies already in flight land before the CTA goes away
        for (int j = gw > SW8 ? gw - SW8 : 0; j < gw; ++j)
          mbar_wait_bounded(bar(B_W8_FULL + j % SW8), (j / SW8) & 1);
      }
    }
  } else if (warp == WARP_TOK) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      int g = 0, gt = 0;  // stage counter; token stages issued
      bool ok = true;
      for (int ip = pair; ip < items && ok; ip += npairs) {
        const Tile tl = tiles[ip / NBP];
        const int box = box_of(nmma_of(tl.rows));
        const CUtensorMap *tmT = box == 8 ? &tmT8 : (box == 32 ? &tmT32 : &tmT80);
        const uint32_t ttx = uint32_t(2 * box * BK * 2);
        const int trow = tl.row0 + int(rank) * box;
        for (int i = 0; i < KT; ++i, ++g) {
          const int stt = g % ST;
          if (!mbar_wait<200>(bar(B_T_EMPTY + stt), ((g / ST) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(bar(B_T_FULL + stt), ttx);
          tma_load_2d_mc(base + OFF_T + uint32_t(stt) * TB + rank * uint32_t(box * BK * 2), tmT,
                         i * BK, trow, bar(B_T_FULL + stt), 3);
          gt = g + 1;
        }
      }
      if (!ok) {
        for (int j = gt > ST ? gt - ST : 0; j < gt; ++j)
          mbar_wait_bounded(bar(B_T_FULL + j % ST), (j / ST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int g = 0, gk = 0;  // stage and K-block counters across items
      bool ok = true;
      for (int ip = pair; ip < items && ok; ip += npairs) {
        const Tile tl = tiles[ip / NBP];
        const uint32_t idesc = idesc_f16(WM, nmma_of(tl.rows));
        for (int kb = 0; kb < KB && ok; ++kb, ++gk) {
          const int b = gk % NCH;
          if (!mbar_wait<1000>(bar(B_ACC_EMPTY + b), ((gk / NCH) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t d = tmem + uint32_t(b * TN);
          for (int h = 0; h < 2; ++h, ++g) {
            const int s16 = g % SW16, stt = g % ST;
            if (!mbar_wait<1000>(bar(B_W16_FULL + s16), (g / SW16) & 1, abort_flag) ||
                !mbar_wait<1000>(bar(B_T_FULL + stt), (g / ST) & 1, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t w0 = base + OFF_W16 + uint32_t(s16) * W16B;
            const uint32_t t0 = base + OFF_T + uint32_t(stt) * TB;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16(d, sdesc(w0 + 32u * kk), sdesc(t0 + 32u * kk), idesc, (h | kk) ? 1u : 0u);
            mma_commit_mc(bar(B_T_EMPTY + stt), 3);
          }
          if (ok) mma_commit(bar(B_ACC_FULL + b));
        }
      }
      mma_commit(bar(B_MMA_DONE));
      mbar_wait_bounded(bar(B_MMA_DONE), 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ converters
    const int t = threadIdx.x - 64;  // 0..127
    int gbase = 0;
    bool ok = true;
    for (int ip = pair; ip < items && ok; ip += npairs, gbase += KT) {
      for (int i = 0; i < KT; ++i) {
        const int g = gbase + i;
        const int sw = g % SW8, s16 = g % SW16;
        if (!__all_sync(0xffffffffu, mbar_wait<1000>(bar(B_W8_FULL + sw), (g / SW8) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        const uint8_t *src = sm + OFF_W8 + sw * W8B;
        uint4 v[NJW];
#pragma unroll
        for (int j = 0; j < NJW; ++j)
          v[j] = *reinterpret_cast<const uint4 *>(src + (j * GCONV + t) * 16);
        fence_async_smem();  // these reads before the next copy into the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_W8_EMPTY + sw));
        if (!__all_sync(0xffffffffu,
                        mbar_wait<1000>(bar(B_T_EMPTY + s16), ((g / SW16) & 1) ^ 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        uint8_t *dst = sm + OFF_W16 + s16 * W16B;
#pragma unroll
        for (int j = 0; j < NJW; ++j) {
          const int c = j * GCONV + t;
          const int row = c >> 2;
          store_f16_row_piece(dst + row * 128, row, c & 3, v[j]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_W16_FULL + s16));
      }
    }
  } else if (warp < 6 + NEPI) {
    // ------------------------------------------------------------ epilogue
    // Warp (q, h) owns token columns [h * EPI_COLS, (h + 1) * EPI_COLS) of
    // tensor-memory lane quarter q (this thread: one output channel) for the
    // whole item and keeps their running sums in registers: per K block one
    // tensor-memory load, one product and one sum per element, no round trip
    // of the sum through tensor memory.  The block's column scales
    // sa[tok][kb] * sw[kb] are staged in this warp's shared-memory row and
    // read back as broadcasts.
    const int q = warp & 3;            // tensor-memory lane quarter of this warp
    const int h = (warp - 6) >> 2;     // which half of the chunk's columns it owns
    const int c0 = h * EPI_COLS;       // first owned column
    float *scal = reinterpret_cast<float *>(sm + OFF_SC) + (warp - 6) * EPI_COLS;
    const uint32_t tq = tmem + (uint32_t(q * 32) << 16);
    constexpr int NSC = (EPI_COLS + 31) / 32;  // owned columns per lane when staging scales
    int gk = 0, it = 0;  // K blocks and items so far
    bool ok = true;
    for (int ip = pair; ip < items && ok; ip += npairs, ++it) {
      const Tile tl = tiles[ip / NBP];
      const int wb = wblock(ip);  // this CTA's weight block = scale block row
      const int64_t n = int64_t(wb) * WM + q * 32 + lane;  // this thread's output channel
      const float *swp = a.sw + (int64_t(tl.expert) * (a.N / 128) + wb) * KB;
      // token scales of the owned columns, loaded one K block ahead
      float sap[NSC];
#pragma unroll
      for (int m = 0; m < NSC; ++m) {
        const int col = c0 + 32 * m + lane;
        sap[m] = (32 * m + lane < EPI_COLS && col < tl.rows) ? a.sa[(int64_t(tl.row0) + col) * KB] : 0.0f;
      }
      float swv = swp[0];
      float acc[EPI_COLS];
#pragma unroll
      for (int j = 0; j < EPI_COLS; ++j) acc[j] = 0.0f;  // acc starts at +0
      for (int kb = 0; kb < KB; ++kb, ++gk) {
        const int b = gk % NCH;
        // column scales sa[col][kb] * sw[kb] (0 past the tile's rows)
#pragma unroll
        for (int m = 0; m < NSC; ++m)
          if (32 * m + lane < EPI_COLS) scal[32 * m + lane] = __fmul_rn(sap[m], swv);
        if (kb + 1 < KB) {
          swv = swp[kb + 1];
#pragma unroll
          for (int m = 0; m < NSC; ++m) {
            const int col = c0 + 32 * m + lane;
            sap[m] = (32 * m + lane < EPI_COLS && col < tl.rows)
                         ? a.sa[(int64_t(tl.row0) + col) * KB + kb + 1] : 0.0f;
          }
        }
        __syncwarp();
        if (!__all_sync(0xffffffffu, mbar_wait<1000>(bar(B_ACC_FULL + b), (gk / NCH) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tch = tq + uint32_t(b * TN + c0);
        // 8-column pieces, the next one's load in flight while this one is
        // scaled and added (two register sets, alternating)
        auto add_piece = [&](int piece, const uint32_t (&v)[8]) {
          const float4 *s4 = reinterpret_cast<const float4 *>(scal + 8 * piece);
#pragma unroll
          for (int j = 0; j < 8; j += 4) {
            const float4 sc = s4[j / 4];
            float *r = acc + 8 * piece + j;
            mul_add2(r[0], r[1], __uint_as_float(v[j]), __uint_as_float(v[j + 1]), sc.x, sc.y, r[0], r[1]);
            mul_add2(r[2], r[3], __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]), sc.z, sc.w, r[2], r[3]);
          }
        };
        constexpr int NPC = EPI_COLS / 8;
        static_assert(NPC % 2 == 0, "pieces go in pairs");
        uint32_t va[8], vb[8];
        tmem_ld8(tch, va);
        tmem_wait_ld(va);
#pragma unroll
        for (int piece = 0; piece < NPC; piece += 2) {
          tmem_ld8(tch + 8u * uint32_t(piece + 1), vb);
          add_piece(piece, va);
          tmem_wait_ld(vb);
          if (piece + 2 < NPC) tmem_ld8(tch + 8u * uint32_t(piece + 2), va);
          add_piece(piece + 1, vb);
          if (piece + 2 < NPC) tmem_wait_ld(va);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY + b));
      }
      if (!ok) break;
      if constexpr (!FUSE) {
        // after the last K block: bf16 out for the owned columns inside the tile
        uint16_t *o = static_cast<uint16_t *>(a.out) + (int64_t(tl.row0) + c0) * a.N + n;
#pragma unroll
        for (int j = 0; j < EPI_COLS; ++j)
          if (c0 + j < tl.rows) o[int64_t(j) * a.N] = f_to_bf16(acc[j]);
      } else {
        // SiLU-and-mul and re-quantization of h column p*128 + q*32 + lane.
        // This thread holds the gate (rank 0) or up (rank 1) value of that
        // column for the owned tokens, rounded to bf16 exactly as the GEMM's
        // output; the peer thread at the same position holds the partner.
        // This CTA finishes tokens [rank*KEEP, rank*KEEP + KEEP) of the owned
        // columns and sends the other half to the peer.
        const int ew = warp - 6;
        const uint32_t peer = rank ^ 1u;
        const uint32_t xoff = uint32_t(P::OFF_XCH + (ew * 32 + lane) * XW * 4);
        const int col0 = c0 + int(rank) * KEEP;  // first kept token column of the tile
        // the peer has read what this warp sent for the previous item
        ok = mbar_wait_cluster(bar(P::B_XE + ew), (it & 1) ^ 1, abort_flag);
        if (ok) {
          const uint32_t dst = mapa(base + xoff, peer);
#pragma unroll
          for (int j = 0; j < XW; j += 4) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = 2 * (j + i);
              w4[i] = rank ? pack_bf16x2(acc[c], acc[c + 1]) : pack_bf16x2(acc[KEEP + c], acc[KEEP + c + 1]);
            }
            st_cluster_v4(dst + 4u * j, w4[0], w4[1], w4[2], w4[3]);
          }
          __syncwarp();  // every lane's copy before the one release below
          if (lane == 0) mbar_arrive_cluster(mapa(bar(P::B_XF + ew), peer));
        }
        uint32_t own[XW];
#pragma unroll
        for (int j = 0; j < XW; ++j)
          own[j] = rank ? pack_bf16x2(acc[KEEP + 2 * j], acc[KEEP + 2 * j + 1])
                        : pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
        uint32_t oth[XW];
        ok = ok && mbar_wait_cluster(bar(P::B_XF + ew), it & 1, abort_flag);
        if (ok) {
          const uint4 *src = reinterpret_cast<const uint4 *>(sm + xoff);
#pragma unroll
          for (int j = 0; j < XW / 4; ++j) {
            const uint4 v4 = src[j];
            oth[4 * j] = v4.x, oth[4 * j + 1] = v4.y, oth[4 * j + 2] = v4.z, oth[4 * j + 3] = v4.w;
          }
          __syncwarp();  // every lane's read before the release
          if (lane == 0) mbar_arrive_cluster(mapa(bar(P::B_XE + ew), peer));  // the peer may send again
        } else {
#pragma unroll
          for (int j = 0; j < XW; ++j) oth[j] = 0u;
        }
        // silu(g) of the kept tokens from the table (exact by construction);
        // misses (out-of-table gates of tokens inside the tile; the columns
        // past the tile's rows hold zeros) take the formula afterwards
        float hv[KEEP];
        uint64_t miss = 0;
#pragma unroll
        for (int jj = 0; jj < KEEP; ++jj) {
          const uint32_t g2 = rank ? oth[jj >> 1] : own[jj >> 1];
          const int idx = silu_index((jj & 1) ? g2 >> 16 : g2 & 0xffffu);
          miss |= uint64_t(idx < 0 && col0 + jj < tl.rows) << jj;
          hv[jj] = __ldg(a.fused_silu_tab + (idx < 0 ? 0 : idx));
        }
        if (__any_sync(0xffffffffu, miss != 0)) {
#pragma unroll
          for (int jj = 0; jj < KEEP; ++jj) {
            const uint32_t g2 = rank ? oth[jj >> 1] : own[jj >> 1];
            if (miss >> jj & 1u) hv[jj] = silu((jj & 1) ? bf16_hi(g2) : bf16_lo(g2));
          }
        }
        // h = silu(g) * u, each product rounded once
#pragma unroll
        for (int jj = 0; jj < KEEP; ++jj) {
          const uint32_t u2 = rank ? own[jj >> 1] : oth[jj >> 1];
          hv[jj] = __fmul_rn(hv[jj], (jj & 1) ? bf16_hi(u2) : bf16_lo(u2));
        }
        // each token's maximum |h| over the 128 columns of group p: this
        // warp's 32 lanes (tokens 0..31 by a reduce-scatter that leaves token
        // jj's maximum in lane jj, tokens 32.. by full reductions), then the
        // four lane quarters through shared memory
        const int par = it & 1;
        float *red = reinterpret_cast<float *>(sm + P::OFF_RED) + (par * 2 + h) * 4 * KEEP;
        if (ok) {
          float m[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) m[jj] = fabsf(hv[jj]);
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) {
            const bool up = (lane & w) != 0;  // this lane keeps the upper half
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = up ? m[i] : m[i + w];
              const float keep = up ? m[i + w] : m[i];
              m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
            }
          }
          red[q * KEEP + lane] = m[0];
#pragma unroll
          for (int jj = 32; jj < KEEP; ++jj) {
            const float mx = warp_max(fabsf(hv[jj]));
            if (lane == jj - 32) red[q * KEEP + jj] = mx;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(P::B_RED + par * 2 + h));
        }
        ok = ok && mbar_wait(bar(P::B_RED + par * 2 + h), (it >> 1) & 1, abort_flag);
        if (!ok) {
          fail();
          break;
        }
        float scl[2], rsl[2];  // scales of kept tokens lane and lane + 32
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int jj = lane + 32 * m;
          scl[m] = 1.0f, rsl[m] = 1.0f;
          if (jj < KEEP) {
            const float am = fmaxf(fmaxf(red[jj], red[KEEP + jj]),
                                   fmaxf(red[2 * KEEP + jj], red[3 * KEEP + jj]));
            scl[m] = quant_scale(am);
            rsl[m] = __frcp_rn(scl[m]);
          }
        }
        const int64_t I = a.N / 2;
        const int p = ip % NBP;
        uint16_t *o16 = a.fused_hq16 + (int64_t(tl.row0) + col0) * I + int64_t(p) * WM + q * 32 + lane;
#pragma unroll
        for (int jj = 0; jj < KEEP; jj += 2) {
          const float sc0 = __shfl_sync(0xffffffffu, scl[jj >> 5], jj & 31);
          const float rs0 = __shfl_sync(0xffffffffu, rsl[jj >> 5], jj & 31);
          const float sc1 = __shfl_sync(0xffffffffu, scl[(jj + 1) >> 5], (jj + 1) & 31);
          const float rs1 = __shfl_sync(0xffffffffu, rsl[(jj + 1) >> 5], (jj + 1) & 31);
          const uint32_t b = __byte_perm(quant_bits(hv[jj], sc0, rs0), quant_bits(hv[jj + 1], sc1, rs1), 0x0040);
          uint32_t f01, f23;  // the two codes as fp16 values (exact)
          s8x4_to_f16x4(b, f01, f23);
          if (col0 + jj < tl.rows) o16[int64_t(jj) * I] = uint16_t(f01);
          if (col0 + jj + 1 < tl.rows) o16[int64_t(jj + 1) * I] = uint16_t(f01 >> 16);
        }
        if (q == 0) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int jj = lane + 32 * m;
            if (jj < KEEP && col0 + jj < tl.rows)
              a.fused_sh[(int64_t(tl.row0) + col0 + jj) * (I / WM) + p] = scl[m];
          }
        }
      }
    }
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

bool gemm_tc6_supported(const GemmArgs &a) {
  return a.A16 != nullptr && a.scheme == WQ_SCHEME_BLOCK && a.out_type == WQ_OUT_BF16 &&
         a.N % (2 * WM) == 0 && a.K % 128 == 0 && a.K <= 65536 &&
         a.E * a.N < (int64_t(1) << 31) && a.R < (int64_t(1) << 31) && tma_available() &&
         num_sms() >= 2;
}

int gemm_tc6_tile_rows() { return TN; }

namespace {
template <bool FUSE>
int launch_tc6(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
               cudaStream_t st) {
  constexpr int SMEM_BYTES = Plan<FUSE>::SMEM_BYTES;
  CUtensorMap mW, m8, m32, m80;
  if (!make_tma_2d_u8(&mW, a.W, int64_t(a.E) * a.N, a.K, BK, WM) ||
      !make_tma_2d_b16_sw128(&m8, a.A16, a.R, a.K, 8) ||
      !make_tma_2d_b16_sw128(&m32, a.A16, a.R, a.K, 32) ||
      !make_tma_2d_b16_sw128(&m80, a.A16, a.R, a.K, 80))
    return WQ_ERR_LAUNCH;
  static bool attr = false;
  static int pairs_resident = 0;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc6_kernel<FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return WQ_ERR_LAUNCH;
    // a persistent grid must be fully co-resident: ask how many 2-CTA
    // clusters of this kernel fit at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * (num_sms() / 2)));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc6_kernel<FUSE>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    pairs_resident = n;
    attr = true;
  }
  const int64_t max_items = int64_t(max_tiles) * (a.N / (2 * WM));
  const int pairs = int(max_items < pairs_resident ? max_items : pairs_resident);
  gemm_tc6_kernel<FUSE><<<2 * pairs, NTHREADS, SMEM_BYTES, st>>>(mW, m8, m32, m80, a, tiles,
                                                                 ntiles);
  return launched(1);
}
}  // namespace

// `tiles` holds token tiles of at most TN rows.  With a.fused_hq16 set the
// kernel writes SiLU-and-mul re-quantized fp16 codes and group scales
// instead of a.out.
int launch_gemm_tc6(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  if (a.fused_hq16 != nullptr) {
    if (a.fused_sh == nullptr || a.N % (2 * WM) != 0) return WQ_ERR_INVALID_ARG;
    return launch_tc6<true>(a, tiles, ntiles, max_tiles, st);
  }
  return launch_tc6<false>(a, tiles, ntiles, max_tiles, st);
}

}  // namespace wq
