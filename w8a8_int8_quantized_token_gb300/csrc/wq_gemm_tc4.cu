// Grouped W8A8 GEMM, int32-accumulator engine for fp16-stored activation
// codes, on CTA pairs that share token tiles (tcgen05, sm_103a).
//
// The channel-wise INT8 GEMM of "[Feature] DeepSeek V3/R1 INT8 Quantization
// (channel-wise)" with the int32 accumulator: C = A_e W_e^T exactly, then
// v = (float(C) * sa[r]) * sw[e][n].  The activation codes arrive already
// stored as fp16 values (the same integers, written by the permute and
// SiLU-mul-quant kernels together with each row's squared norm), so TMA puts
// them straight into the 128-byte swizzled K-major layout the MMA reads; only
// the int8 weights are widened to fp16 in shared memory.  tcgen05.mma
// kind::f16 accumulates in float32 over the whole K range in one pass, exact
// when max||a||^2 * max||w||^2 < 2^48 (Cauchy-Schwarz bounds every partial
// sum below 2^24); the epilogue checks that with the producers' token norms
// and the converters' weight norms, and a failing tile raises a device flag
// for the exact recompute.
//
// The two CTAs of a cluster work on the same token tile and adjacent 128-row
// weight blocks: each loads half of every token stage and multicasts it to
// both, so a CTA reads 16 KB of tokens and 8 KB of weights from L2 per K
// stage.  A token stage is released when the MMAs of both CTAs are done with
// it (their completions are multicast to both CTAs' barriers); the
// widened-weight ring has the token ring's depth and waits on the same
// barriers, so one commit per K stage frees both slots.  Operand
// roles are swapped relative to the row-major problem: MMA M = 128 output
// channels, N = 16..256 tokens.  Two tensor-memory accumulators let the
// epilogue of one item overlap the MMAs of the next.
//   warp 0      TMA producer of the int8 weights
//   warp 14     TMA producer of the tokens (half of each stage, multicast);
//               separate from the weight producer so neither ring's wait
//               holds back the other's copies
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-9   converters (two groups taking alternate K stages): int8
//               weights -> fp16 (128-byte swizzled K-major) + row norms
//   warps 10-13 epilogue: dequant, bf16, coalesced stores (32 channels/warp)
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int WM = 128, TN = 256, BK = 64;
constexpr int SW8 = 4, SW16 = 4, ST = 4;        // ring depths: int8 W, fp16 W, fp16 tokens
static_assert(SW16 == ST, "a widened-weight slot is released with its token slot");
constexpr int W8B = WM * BK, W16B = 2 * W8B;    // weight stage bytes
constexpr int TB = TN * BK * 2;                 // token stage bytes (fp16)
constexpr int OFF_T = 0;
constexpr int OFF_W16 = OFF_T + ST * TB;
constexpr int OFF_W8 = OFF_W16 + SW16 * W16B;
constexpr int OFF_BAR = OFF_W8 + SW8 * W8B;
constexpr int B_W8_FULL = 0, B_W8_EMPTY = SW8, B_W16_FULL = 2 * SW8,
              B_T_FULL = 2 * SW8 + SW16, B_T_EMPTY = B_T_FULL + ST,
              B_ACC_FULL = B_T_EMPTY + ST,  // [2]
    B_ACC_EMPTY = B_ACC_FULL + 2,           // [2]
    B_NORM_READY = B_ACC_FULL + 4,          // [2]
    B_NORM_FREE = B_ACC_FULL + 6,           // [2]
    B_NORM_READ = B_ACC_FULL + 8,           // [2]
    B_MMA_DONE = B_ACC_FULL + 10, NBAR = B_ACC_FULL + 11;
constexpr int OFF_NORM = OFF_BAR + NBAR * 8;  // int32 [2 buffers][2 converter groups]
constexpr int OFF_TMEM = OFF_NORM + 16;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
constexpr int NTHREADS = 480;
constexpr int WARP_TOK = 14;  // token producer
constexpr int GCONV = 128;              // threads of one converter group
constexpr int NJW = WM * 4 / GCONV;     // weight 16-byte pieces per converter thread

__device__ __forceinline__ int sq4(uint32_t w, int acc) { return __dp4a(int(w), int(w), acc); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    gemm_tc4_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT8,
                    const __grid_constant__ CUtensorMap tmT32,
                    const __grid_constant__ CUtensorMap tmT128, const GemmArgs a,
                    const Tile *__restrict__ tiles, const int32_t *__restrict__ ntiles,
                    int32_t *__restrict__ redo) {
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
  volatile int *norm = reinterpret_cast<volatile int *>(sm + OFF_NORM);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = int(a.K / BK);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) norm[i] = 0;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_ACC_FULL + b), 1);
      mbar_init(bar(B_ACC_EMPTY + b), 4);
      mbar_init(bar(B_NORM_READY + b), 2 * GCONV / 32);
      mbar_init(bar(B_NORM_FREE + b), 1);
      mbar_init(bar(B_NORM_READ + b), 4);
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
  auto box_of = [](int nmma) { return nmma <= 16 ? 8 : (nmma <= 64 ? 32 : 128); };

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int g = 0, gw = 0;
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
      if (!ok) {
        for (int j = gw > SW8 ? gw - SW8 : 0; j < gw; ++j)
          mbar_wait_bounded(bar(B_W8_FULL + j % SW8), (j / SW8) & 1);
      }
    }
  } else if (warp == WARP_TOK) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      int g = 0, gt = 0;
      bool ok = true;
      for (int ip = pair; ip < items && ok; ip += npairs) {
        const Tile tl = tiles[ip / NBP];
        const int box = box_of(nmma_of(tl.rows));
        const CUtensorMap *tmT = box == 8 ? &tmT8 : (box == 32 ? &tmT32 : &tmT128);
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
      int g = 0, ii = 0;
      bool ok = true;
      for (int ip = pair; ip < items && ok; ip += npairs, ++ii) {
        const Tile tl = tiles[ip / NBP];
        const uint32_t idesc = idesc_f16(WM, nmma_of(tl.rows));
        const int b = ii & 1;
        if (!mbar_wait(bar(B_ACC_EMPTY + b), ((ii >> 1) & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        const uint32_t d = tmem + uint32_t(b) * 256u;
        for (int i = 0; i < KT; ++i, ++g) {
          const int s16 = g % SW16, stt = g % ST;
          // weights widened and tokens landed (the converters wait for both)
          if (!mbar_wait(bar(B_W16_FULL + s16), (g / SW16) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w0 = base + OFF_W16 + uint32_t(s16) * W16B;
          const uint32_t t0 = base + OFF_T + uint32_t(stt) * TB;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16(d, sdesc(w0 + 32u * kk), sdesc(t0 + 32u * kk), idesc, (i | kk) ? 1u : 0u);
          mma_commit_mc(bar(B_T_EMPTY + stt), 3);
        }
        if (ok) mma_commit(bar(B_ACC_FULL + b));
      }
      mma_commit(bar(B_MMA_DONE));
      mbar_wait_bounded(bar(B_MMA_DONE), 0);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ converters
    // two groups of four warps; group `grp` widens the stages of parity grp
    const int grp = (warp - 2) >> 2;
    const int t = threadIdx.x - 64 - grp * GCONV;  // 0..127 within the group
    int gbase = 0, ii = 0;
    bool ok = true;
    for (int ip = pair; ip < items && ok; ip += npairs, ++ii, gbase += KT) {
      int nrm[NJW];
#pragma unroll
      for (int j = 0; j < NJW; ++j) nrm[j] = 0;
      for (int i = grp; i < KT; i += 2) {
        const int g = gbase + i;
        const int sw = g % SW8, s16 = g % SW16;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_W8_FULL + sw), (g / SW8) & 1, abort_flag))) {
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
                        mbar_wait(bar(B_T_EMPTY + s16), ((g / SW16) & 1) ^ 1, abort_flag))) {
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
          nrm[j] += sq4(v[j].w, sq4(v[j].z, 0)) + sq4(v[j].y, sq4(v[j].x, 0));
        }
        fence_async_smem();
        // the stage's token slot has landed too: the MMA issuer then checks a
        // single barrier per stage
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_T_FULL + s16), (g / ST) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_W16_FULL + s16));
      }
      if (!ok) break;
      // squared weight-row norms over this group's stages (lanes 4m..4m+3
      // hold the 4 pieces of one row); a row's norm is at most the sum of the
      // two groups' largest partial norms, which the epilogue checks
      int wmax = 0;
#pragma unroll
      for (int j = 0; j < NJW; ++j) {
        int n2 = nrm[j];
        n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
        n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
        wmax = max(wmax, n2);
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      const int b = ii & 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar(B_NORM_FREE + b), ((ii >> 1) & 1) ^ 1, abort_flag))) {
        fail();
        break;
      }
      if (lane == 0) atomicMax(const_cast<int *>(norm + 2 * b + grp), wmax);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_NORM_READY + b));
    }
  } else if (warp < WARP_TOK) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quarter of this warp
    int ii = 0;
    for (int ip = pair; ip < items; ip += npairs, ++ii) {
      const Tile tl = tiles[ip / NBP];
      const int wb = (ip % NBP) * 2 + int(rank);
      const int b = ii & 1, par = (ii >> 1) & 1;
      int tmax = 0;  // largest squared token-row norm of the tile
      for (int j = lane; j < tl.rows; j += 32) tmax = max(tmax, a.a_norm2[int64_t(tl.row0) + j]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      // the item's token scales (lane j of group p holds token 32p + j) and
      // this thread's weight scale, loaded while the item's MMAs still run
      constexpr int NGRP = TN / 32;
      const int64_t n = int64_t(wb) * WM + q * 32 + lane;  // this thread's output channel
      const float swn = a.sw[int64_t(tl.expert) * a.N + n];
      float sal[NGRP];
#pragma unroll
      for (int p = 0; p < NGRP; ++p)
        sal[p] = p * 32 + lane < tl.rows ? a.sa[int64_t(tl.row0) + p * 32 + lane] : 0.0f;
      if (!__all_sync(0xffffffffu, mbar_wait<500>(bar(B_ACC_FULL + b), par, abort_flag)) ||
          !__all_sync(0xffffffffu, mbar_wait(bar(B_NORM_READY + b), par, abort_flag))) {
        fail();
        break;
      }
      tc_fence_after();
      const long long nw = (long long)norm[2 * b] + norm[2 * b + 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_NORM_READ + b));
      if (warp == 10 && lane == 0) {
        // once all four epilogue warps have read the norms, clear them for the
        // item after next and hand the slots back to the converters
        if (mbar_wait(bar(B_NORM_READ + b), par, abort_flag)) {
          norm[2 * b] = 0;
          norm[2 * b + 1] = 0;
          mbar_arrive(bar(B_NORM_FREE + b));
        } else {
          fail();
        }
      }
      if (nw * (long long)tmax >= (1ll << 48) && q == 0 && lane == 0) atomicExch(redo, 1);
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
  cluster_sync();  // no multicast copy or completion targets either CTA after this
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool gemm_tc4_supported(const GemmArgs &a) {
  return a.A16 != nullptr && a.a_norm2 != nullptr && a.scheme == WQ_SCHEME_CHANNEL &&
         acc_modes_agree(a) && a.N % (2 * WM) == 0 && a.K % BK == 0 && a.K <= 65536 &&
         a.E * a.N < (int64_t(1) << 31) && a.R < (int64_t(1) << 31) && tma_available() &&
         num_sms() >= 2;
}

// `tiles` holds token tiles of at most 256 rows.
int launch_gemm_tc4(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    int32_t *redo, cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  CUtensorMap mW, m8, m32, m128;
  if (!make_tma_2d_u8(&mW, a.W, int64_t(a.E) * a.N, a.K, BK, WM) ||
      !make_tma_2d_b16_sw128(&m8, a.A16, a.R, a.K, 8) ||
      !make_tma_2d_b16_sw128(&m32, a.A16, a.R, a.K, 32) ||
      !make_tma_2d_b16_sw128(&m128, a.A16, a.R, a.K, 128))
    return WQ_ERR_LAUNCH;
  static bool attr = false;
  static int pairs_resident = 0;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return WQ_ERR_LAUNCH;
    // a persistent grid must be fully co-resident: ask how many 2-CTA
    // clusters of this kernel fit at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * (num_sms() / 2)));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc4_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    pairs_resident = n;
    attr = true;
  }
  const int64_t max_items = int64_t(max_tiles) * (a.N / (2 * WM));
  const int pairs = int(max_items < pairs_resident ? max_items : pairs_resident);
  gemm_tc4_kernel<<<2 * pairs, NTHREADS, SMEM_BYTES, st>>>(mW, m8, m32, m128, a, tiles, ntiles,
                                                          redo);
  return launched(1);
}

}  // namespace wq
