// Grouped W8A8 GEMM for token tiles of at most 16 rows (CUDA cores, sm_103a).
//
// The channel-wise and block-wise INT8 GEMMs of "[Feature] DeepSeek V3/R1
// INT8 Quantization (channel-wise)" and of the Meituan INT8 article's
// quantization section, for experts that hold only a few routed tokens
// (decode batches, the ragged tail of an expert's rows).  There the GEMM
// streams the expert's weights from HBM and uses each weight byte for only a
// few tokens, so the tensor-core engines (which must widen every weight code
// to fp16 in shared memory before the MMA can read it) spend their time
// widening.  This engine reads the int8 codes as they are:
//   * one TMA producer thread streams weight tiles of 256 channels x 128 K
//     (128-byte swizzled) and the tile's token rows (4, 8 or 16 rows x
//     128 K) into a six-stage shared-memory ring;
//   * eight consumer warps own one output channel per thread; each reads its
//     channel's 16-byte pieces (the swizzle makes a warp's 32 rows
//     conflict-free) and the token pieces (the same address across the warp:
//     one broadcast), and accumulates with dp4a.
// Integer sums are exact, so every mode takes its own steps exactly and no
// recompute is ever needed:
//   channel, int32 acc: C over all K, v = (float(C) * sa[r]) * sw[e][n];
//   channel, fp32 acc:  acc = acc + float(C_t) per 128-wide K tile t, then
//                       v = (acc * sa[r]) * sw[e][n];
//   block:              acc = acc + float(C_kb) * (sa[r][kb] * sw[e][n/128][kb]).
// Persistent CTAs; work item = (token tile of one expert) x (256 channels).
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// lets its own copies land (bounded) and exits.
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int WN = 256;                  // output channels per item
constexpr int BK = 128;                  // K per stage (= one block of the block scheme)
// most token rows per tile: nine warps put three on one SM sub-partition,
// which caps a thread at 168 registers; 16 accumulators (and 16 float sums)
// fit with the unrolled loads
constexpr int TMAX = 16;
constexpr int NCW = WN / 32;             // consumer warps
constexpr int NTHREADS = 32 * (NCW + 1);  // + the producer warp
constexpr int STAGES = 6;
constexpr int W_BYTES = WN * BK;           // 32 KB of weight bytes per stage (256 rows x 128 B)
// Stage plan: int8 weights take BK = 128 codes of K a stage; int4 weights
// (two codes a byte) take 256, so a stage still carries 32 KB of weights and
// six stages keep the same bytes in flight.  Token rows are one byte a code.
template <bool W4>
struct SPlan {
  static constexpr int BKC = W4 ? 2 * BK : BK;         // K codes per stage
  static constexpr int ST_BYTES = W_BYTES + TMAX * BKC;  // + the token tile
  static constexpr int OFF_BAR = STAGES * ST_BYTES;      // full[STAGES], empty[STAGES]
  static constexpr int OFF_ABORT = OFF_BAR + 2 * STAGES * 8;
  static constexpr int SMEM_BYTES = OFF_ABORT + 16 + 1024;  // + alignment slack
  static_assert(ST_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
};

__device__ __forceinline__ int token_box(int rows) {
  return rows <= 4 ? 4 : (rows <= 8 ? 8 : 16);
}

// One item for a consumer thread: NT token rows are resident per stage (the
// tile's valid rows first); row r of the 256-channel weight tile is this
// thread's channel.  Returns false if a wait gave up.
template <int NT, bool W4>
__device__ __forceinline__ bool consume_item(const GemmArgs &a, const Tile &tl, int nb, int KT,
                                             const uint8_t *sm, uint32_t base, int &g, int r,
                                             volatile int *abort_flag) {
  const int lane = r & 31;
  const int64_t n = int64_t(nb) * WN + r;
  const bool blk = a.scheme == WQ_SCHEME_BLOCK;
  const bool f32c = !blk && a.acc == WQ_ACC_F32;
  const int nt = tl.rows < NT ? tl.rows : NT;
  const int64_t nc = n < a.N ? n : a.N - 1;  // channel for scale reads (idle lanes read a valid one)
  int acc[NT];
  float accf[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    acc[t] = 0;
    accf[t] = 0.0f;
  }
  constexpr int BKC = SPlan<W4>::BKC, ST_BYTES = SPlan<W4>::ST_BYTES, OFF_BAR = SPlan<W4>::OFF_BAR;
  const int sw8 = r & 7;
  for (int i = 0; i < KT; ++i, ++g) {
    const int s = g % STAGES;
    if (!mbar_wait(base + OFF_BAR + 8u * uint32_t(s), uint32_t(g / STAGES) & 1u, abort_flag))
      return false;
    const uint8_t *tk = sm + s * ST_BYTES + W_BYTES;
    if constexpr (W4) {
      // int4 weights: this channel's 128-byte row of the stage (256 codes),
      // 128-byte swizzled like the int8 rows; each 16-byte chunk is 32 codes
      // against 32 token bytes (read as broadcasts)
      const uint8_t *wrow = sm + s * ST_BYTES + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 p = *reinterpret_cast<const uint4 *>(wrow + ((c ^ sw8) << 4));
        uint32_t w8[8];
        s4x8_to_s8x8(p.x, w8[0], w8[1]);
        s4x8_to_s8x8(p.y, w8[2], w8[3]);
        s4x8_to_s8x8(p.z, w8[4], w8[5]);
        s4x8_to_s8x8(p.w, w8[6], w8[7]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 x0 = *reinterpret_cast<const uint4 *>(tk + t * BKC + c * 32);
          const uint4 x1 = *reinterpret_cast<const uint4 *>(tk + t * BKC + c * 32 + 16);
          acc[t] = __dp4a(int(w8[0]), int(x0.x), acc[t]);
          acc[t] = __dp4a(int(w8[1]), int(x0.y), acc[t]);
          acc[t] = __dp4a(int(w8[2]), int(x0.z), acc[t]);
          acc[t] = __dp4a(int(w8[3]), int(x0.w), acc[t]);
          acc[t] = __dp4a(int(w8[4]), int(x1.x), acc[t]);
          acc[t] = __dp4a(int(w8[5]), int(x1.y), acc[t]);
          acc[t] = __dp4a(int(w8[6]), int(x1.z), acc[t]);
          acc[t] = __dp4a(int(w8[7]), int(x1.w), acc[t]);
        }
      }
    } else {
      const uint8_t *wrow = sm + s * ST_BYTES + r * BK;
#pragma unroll
      for (int c = 0; c < BK / 16; ++c) {
        const uint4 w = *reinterpret_cast<const uint4 *>(wrow + ((c ^ sw8) << 4));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 x = *reinterpret_cast<const uint4 *>(tk + t * BK + c * 16);
          acc[t] = __dp4a(int(w.x), int(x.x), acc[t]);
          acc[t] = __dp4a(int(w.y), int(x.y), acc[t]);
          acc[t] = __dp4a(int(w.z), int(x.z), acc[t]);
          acc[t] = __dp4a(int(w.w), int(x.w), acc[t]);
        }
      }
    }
    fence_async_smem();  // these reads before the next copy into the slot
    __syncwarp();
    if (lane == 0) mbar_arrive(base + OFF_BAR + 8u * uint32_t(STAGES + s));
    if (blk) {
      const int KB = KT;
      const float swv =
          a.sw[(int64_t(tl.expert) * (a.N / 128) + nc / 128) * KB + i];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < nt) {
          const float sav = a.sa[int64_t(tl.row0 + t) * KB + i];
          accf[t] = __fadd_rn(accf[t], __fmul_rn(__int2float_rn(acc[t]), __fmul_rn(sav, swv)));
        }
        acc[t] = 0;
      }
    } else if (f32c) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        accf[t] = __fadd_rn(accf[t], __int2float_rn(acc[t]));
        acc[t] = 0;
      }
    }
  }
  if (n < a.N) {
    const float swn = blk ? 0.0f : a.sw[int64_t(tl.expert) * a.N + n];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const int64_t row = int64_t(tl.row0) + t;
        if (a.out_type == WQ_OUT_I32) {
          reinterpret_cast<int32_t *>(a.out)[row * a.N + n] = acc[t];
        } else {
          float v;
          if (blk) {
            v = accf[t];
          } else {
            const float c = f32c ? accf[t] : __int2float_rn(acc[t]);
            v = __fmul_rn(__fmul_rn(c, a.sa[row]), swn);
          }
          reinterpret_cast<uint16_t *>(a.out)[row * a.N + n] = f_to_bf16(v);
        }
      }
    }
  }
  return true;
}

template <bool W4>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_small_kernel(const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmT4,
                      const __grid_constant__ CUtensorMap tmT8,
                      const __grid_constant__ CUtensorMap tmT16, const GemmArgs a,
                      const Tile *__restrict__ tiles, const int32_t *__restrict__ ntiles) {
  extern __shared__ uint8_t smem_raw[];
  const int NB = int((a.N + WN - 1) / WN);
  const int items = ntiles[0] * NB;
  if (int(blockIdx.x) >= items) return;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  constexpr int BKC = SPlan<W4>::BKC, ST_BYTES = SPlan<W4>::ST_BYTES, OFF_BAR = SPlan<W4>::OFF_BAR,
                OFF_ABORT = SPlan<W4>::OFF_ABORT;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_ABORT);
  auto full = [&](int s) { return base + OFF_BAR + 8u * uint32_t(s); };
  auto empty = [&](int s) { return base + OFF_BAR + 8u * uint32_t(STAGES + s); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = int(a.K / BKC);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), NCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const Tile tl = tiles[it / NB];
        const int nb = it % NB;
        const int box = token_box(tl.rows);
        const CUtensorMap *tmT = box == 4 ? &tmT4 : (box == 8 ? &tmT8 : &tmT16);
        const uint32_t tx = uint32_t(W_BYTES + box * BKC);
        const int wrow = int(int64_t(tl.expert) * a.N + int64_t(nb) * WN);
        for (int i = 0; i < KT; ++i, ++g) {
          const int s = g % STAGES;
          if (!mbar_wait<200>(empty(s), (uint32_t(g / STAGES) & 1u) ^ 1u, abort_flag)) {
            *abort_flag = 1;
            set_status(a.status, WQ_ERR_TIMEOUT);
            ok = false;
            break;
          }
          const uint32_t dst = base + uint32_t(s) * ST_BYTES;
          mbar_expect_tx(full(s), tx);
          tma_load_2d(dst, &tmW, i * 128, wrow, full(s));  // 128 weight bytes a row per stage
          tma_load_2d(dst + W_BYTES, tmT, i * BKC, tl.row0, full(s));
        }
      }
      // the last copies issued into each slot must land before the CTA exits
      for (int j = g > STAGES ? g - STAGES : 0; j < g; ++j)
        mbar_wait_bounded(full(j % STAGES), uint32_t(j / STAGES) & 1u);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int r = warp * 32 + lane;
    int g = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
      const Tile tl = tiles[it / NB];
      const int nb = it % NB;
      const int box = token_box(tl.rows);
      bool ok;
      if (box == 4)
        ok = consume_item<4, W4>(a, tl, nb, KT, sm, base, g, r, abort_flag);
      else if (box == 8)
        ok = consume_item<8, W4>(a, tl, nb, KT, sm, base, g, r, abort_flag);
      else
        ok = consume_item<16, W4>(a, tl, nb, KT, sm, base, g, r, abort_flag);
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, WQ_ERR_TIMEOUT);
        break;
      }
    }
  }
}

}  // namespace

bool gemm_small_supported(const GemmArgs &a) {
  if (a.w4 && (a.scheme != WQ_SCHEME_CHANNEL || a.acc != WQ_ACC_I32 || a.K % (2 * BK))) return false;
  return a.A != nullptr && a.K % BK == 0 && a.K <= 65536 && a.N % 32 == 0 &&
         (a.scheme == WQ_SCHEME_CHANNEL || a.scheme == WQ_SCHEME_BLOCK) &&
         int64_t(a.E) * a.N < (int64_t(1) << 31) && a.R < (int64_t(1) << 31) && tma_available();
}

int gemm_small_max_rows() { return TMAX; }

// `tiles` holds at most max_tiles tiles of at most 16 rows each.
int launch_gemm_small(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                      cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  CUtensorMap mW, m4, m8, m16;
  // weights: a 128-byte row per stage (128 int8 codes, or 256 int4 codes),
  // 128-byte swizzled; tokens: one byte a code, BKC codes a stage
  const int bkc = a.w4 ? SPlan<true>::BKC : SPlan<false>::BKC;
  const int smem = a.w4 ? SPlan<true>::SMEM_BYTES : SPlan<false>::SMEM_BYTES;
  if (!make_tma_2d_u8_sw128(&mW, a.W, int64_t(a.E) * a.N, a.w4 ? a.K / 2 : a.K, WN) ||
      !make_tma_2d_u8(&m4, a.A, a.R, a.K, bkc, 4) || !make_tma_2d_u8(&m8, a.A, a.R, a.K, bkc, 8) ||
      !make_tma_2d_u8(&m16, a.A, a.R, a.K, bkc, 16))
    return WQ_ERR_LAUNCH;
  static bool attr[2] = {false, false};
  auto kern = a.w4 ? gemm_small_kernel<true> : gemm_small_kernel<false>;
  if (!attr[a.w4 ? 1 : 0]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return WQ_ERR_LAUNCH;
    attr[a.w4 ? 1 : 0] = true;
  }
  const int64_t max_items = int64_t(max_tiles) * ((a.N + WN - 1) / WN);
  const int grid = int(max_items < num_sms() ? max_items : num_sms());
  kern<<<grid, NTHREADS, smem, st>>>(mW, m4, m8, m16, a, tiles, ntiles);
  return launched(1);
}

}  // namespace wq
