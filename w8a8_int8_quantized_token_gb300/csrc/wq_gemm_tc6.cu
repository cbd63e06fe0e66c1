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
constexpr int SW8 = 8, SW16 = 4, ST = 4;        // ring depths: int8 W, fp16 W, fp16 tokens
static_assert(SW16 == ST, "a widened-weight slot is released with its token slot");
constexpr int W8B = WM * BK, W16B = 2 * W8B;    // weight stage bytes
constexpr int TB = TN * BK * 2;                 // token stage bytes (fp16)
constexpr int NCH = 3;                          // chunk accumulators (tensor-memory columns [0, 3*TN))
constexpr int EPI_COLS = TN / 2;                // token columns each epilogue warp owns
constexpr int OFF_T = 0;
constexpr int OFF_W16 = OFF_T + ST * TB;
constexpr int OFF_W8 = OFF_W16 + SW16 * W16B;
constexpr int NEPI = 8;                         // epilogue warps
constexpr int OFF_SC = OFF_W8 + SW8 * W8B;      // float [NEPI][EPI_COLS] column scales
constexpr int OFF_BAR = OFF_SC + NEPI * EPI_COLS * 4;
constexpr int B_W8_FULL = 0, B_W8_EMPTY = SW8, B_W16_FULL = 2 * SW8,
              B_T_FULL = 2 * SW8 + SW16, B_T_EMPTY = B_T_FULL + ST,
              B_ACC_FULL = B_T_EMPTY + ST,  // [NCH]
    B_ACC_EMPTY = B_ACC_FULL + NCH,         // [NCH]
    B_MMA_DONE = B_ACC_FULL + 2 * NCH, NBAR = B_ACC_FULL + 2 * NCH + 1;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
static_assert(TB % 1024 == 0 && OFF_W16 % 1024 == 0 && OFF_W8 % 1024 == 0, "swizzle alignment");
static_assert(NCH * TN <= 512, "tensor memory plan");
static_assert(EPI_COLS % 16 == 0 && NEPI == 8, "each epilogue warp owns 16-column pieces");
static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    gemm_tc6_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT8,
                    const __grid_constant__ CUtensorMap tmT32,
                    const __grid_constant__ CUtensorMap tmT80, const GemmArgs a,
                    const Tile *__restrict__ tiles, const int32_t *__restrict__ ntiles) {
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
  // token rows each CTA of the pair loads for an MMA of width nmma
  auto box_of = [](int nmma) { return nmma <= 16 ? 8 : (nmma <= 64 ? 32 : 80); };

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int g = 0, gw = 0;  // stage counter; weight stages issued
      bool ok = true;
      for (int ip = pair; ip < items && ok; ip += npairs) {
        const Tile tl = tiles[ip / NBP];
        const int wb = (ip % NBP) * 2 + int(rank);
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
    int gk = 0;
    bool ok = true;
    for (int ip = pair; ip < items && ok; ip += npairs) {
      const Tile tl = tiles[ip / NBP];
      const int wb = (ip % NBP) * 2 + int(rank);  // this CTA's weight block = scale block row
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
#pragma unroll
        for (int piece = 0; piece < EPI_COLS / 16; ++piece) {
          uint32_t v[16];
          tmem_ld16(tch + 16u * piece, v);
          tmem_wait_ld();
          const float4 *s4 = reinterpret_cast<const float4 *>(scal + 16 * piece);
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 sc = s4[j / 4];
            float *r = acc + 16 * piece + j;
            mul_add2(r[0], r[1], __uint_as_float(v[j]), __uint_as_float(v[j + 1]), sc.x, sc.y, r[0], r[1]);
            mul_add2(r[2], r[3], __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]), sc.z, sc.w, r[2], r[3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY + b));
      }
      if (!ok) break;
      // after the last K block: bf16 out for the owned columns inside the tile
      uint16_t *o = static_cast<uint16_t *>(a.out) + (int64_t(tl.row0) + c0) * a.N + n;
#pragma unroll
      for (int j = 0; j < EPI_COLS; ++j)
        if (c0 + j < tl.rows) o[int64_t(j) * a.N] = f_to_bf16(acc[j]);
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

// `tiles` holds token tiles of at most TN rows.
int launch_gemm_tc6(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  CUtensorMap mW, m8, m32, m80;
  if (!make_tma_2d_u8(&mW, a.W, int64_t(a.E) * a.N, a.K, BK, WM) ||
      !make_tma_2d_b16_sw128(&m8, a.A16, a.R, a.K, 8) ||
      !make_tma_2d_b16_sw128(&m32, a.A16, a.R, a.K, 32) ||
      !make_tma_2d_b16_sw128(&m80, a.A16, a.R, a.K, 80))
    return WQ_ERR_LAUNCH;
  static bool attr = false;
  static int pairs_resident = 0;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc6_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return WQ_ERR_LAUNCH;
    // a persistent grid must be fully co-resident: ask how many 2-CTA
    // clusters of this kernel fit at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * (num_sms() / 2)));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc6_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    pairs_resident = n;
    attr = true;
  }
  const int64_t max_items = int64_t(max_tiles) * (a.N / (2 * WM));
  const int pairs = int(max_items < pairs_resident ? max_items : pairs_resident);
  gemm_tc6_kernel<<<2 * pairs, NTHREADS, SMEM_BYTES, st>>>(mW, m8, m32, m80, a, tiles, ntiles);
  return launched(1);
}

}  // namespace wq
