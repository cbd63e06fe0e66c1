// Grouped W8A8 GEMM on the tcgen05 tensor cores, chunked exact engine.
//
// The INT8 products of "[Feature] DeepSeek V3/R1 INT8 Quantization
// (channel-wise)" and of the Meituan article's block-wise scheme, computed
// exactly.  sm_103a has no tcgen05 integer MMA, so every int8 code q (|q| <=
// 127; -128 also fits) is widened to an fp16 value equal to q (fp16 holds
// every integer below 2048) and multiplied by tcgen05.mma kind::f16 with
// float32 accumulation in tensor memory.  A product is at most 127^2 = 16129,
// so any sum of at most 1024 products is an integer of magnitude below 2^24:
// every partial sum the tensor core forms is exactly representable, and the
// float32 accumulator over a chunk of at most 1024 K elements holds the exact
// integer.  The epilogue drains each chunk into a running sum:
//   int32 accumulator:  chunks of 1024 K, run_i32 += int(chunk)   (exact C)
//   fp32 accumulator:   chunks of 128 K,  run_f32 = run_f32 + chunk
//   block scheme:       chunks of 128 K,  run_f32 = run_f32 + chunk * (sa * sw)
// which is the arithmetic, in the same order, of the definitions in
// include/wq.h.  This engine serves the fp32-accumulator and block-wise
// modes, and recomputes an int32 launch exactly when the fast engine
// (wq_gemm_tc2.cu) could not prove its single-pass sums exact (`gate`).
//
// Persistent CTAs; work item = (128-row tile of one expert) x (256 output
// channels); K in stages of 64.
//   warp 0     TMA producer: int8 A and W tiles -> int8 staging ring
//   warp 1     TMEM allocator and MMA issuer (one thread)
//   warps 2-5  converters: int8 staging -> fp16, 128-byte swizzled K-major
//   warps 6-9  epilogue: TMEM chunk -> running sum (TMEM) -> dequant -> out
// Tensor memory: columns [0,256) chunk accumulator, [256,512) running sum.
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "wq_tc.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int S8 = 3, S16 = 3;
constexpr int A8 = BM * BK, B8 = BN * BK;  // int8 tile bytes
constexpr int A16 = 2 * A8, B16 = 2 * B8;  // fp16 tile bytes
constexpr int ST8 = A8 + B8, ST16 = A16 + B16;
constexpr int OFF_F16 = 0;
constexpr int OFF_I8 = OFF_F16 + S16 * ST16;
constexpr int OFF_BAR = OFF_I8 + S8 * ST8;
constexpr int B_S8_FULL = 0, B_S8_EMPTY = S8, B_F16_FULL = 2 * S8, B_F16_EMPTY = 2 * S8 + S16,
              B_ACC_FULL = 2 * S8 + 2 * S16, B_ACC_EMPTY = B_ACC_FULL + 1,
              B_MMA_DONE = B_ACC_FULL + 2, NBAR = B_ACC_FULL + 3;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_USED = OFF_ABORT + 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
constexpr int NTHREADS = 320;
constexpr uint32_t kIdesc = idesc_f16(BM, BN);

__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const GemmArgs a, const Tile *__restrict__ tiles,
                   const int32_t *__restrict__ ntiles, const int32_t *__restrict__ gate,
                   int chunk_stages) {
  extern __shared__ uint8_t smem_raw[];
  if (gate != nullptr && *gate == 0) return;  // exact recompute not needed
  const int n_nt = int(a.N / BN);
  const int items = ntiles[0] * n_nt;
  if (int(blockIdx.x) >= items) return;  // uniform over the CTA, before any setup
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_ABORT);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = int(a.K / BK);
  const int NC = (KT + chunk_stages - 1) / chunk_stages;
  const bool block = a.scheme == WQ_SCHEME_BLOCK;
  const bool f32acc = block || a.acc == WQ_ACC_F32;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < S8; ++s) {
      mbar_init(bar(B_S8_FULL + s), 1);
      mbar_init(bar(B_S8_EMPTY + s), 4);
    }
    for (int s = 0; s < S16; ++s) {
      mbar_init(bar(B_F16_FULL + s), 4);
      mbar_init(bar(B_F16_EMPTY + s), 1);
    }
    mbar_init(bar(B_ACC_FULL), 1);
    mbar_init(bar(B_ACC_EMPTY), 4);
    mbar_init(bar(B_MMA_DONE), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int g = 0;  // global stage counter across items
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const Tile tl = tiles[it / n_nt];
        const int n0 = (it % n_nt) * BN;
        for (int i = 0; i < KT; ++i, ++g) {
          const int s = g % S8;
          if (!mbar_wait<200>(bar(B_S8_EMPTY + s), ((g / S8) & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t dst = base + OFF_I8 + uint32_t(s) * ST8;
          mbar_expect_tx(bar(B_S8_FULL + s), ST8);
          tma_load_2d(dst, &tmA, i * BK, tl.row0, bar(B_S8_FULL + s));
          tma_load_2d(dst + A8, &tmW, i * BK, int(int64_t(tl.expert) * a.N + n0),
                      bar(B_S8_FULL + s));
        }
      }
      if (!ok) {  // let the copies already in flight land before the CTA goes away
        for (int j = g > S8 ? g - S8 : 0; j < g; ++j) mbar_wait_bounded(bar(B_S8_FULL + j % S8), (j / S8) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int g = 0, gc = 0;  // global stage and chunk counters
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        for (int i = 0; i < KT; ++i, ++g) {
          const bool first = (i % chunk_stages) == 0;
          const bool last = (i % chunk_stages) == chunk_stages - 1 || i == KT - 1;
          if (first && !mbar_wait(bar(B_ACC_EMPTY), (gc & 1) ^ 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          const int s = g % S16;
          if (!mbar_wait(bar(B_F16_FULL + s), (g / S16) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = base + OFF_F16 + uint32_t(s) * ST16;
          const uint32_t b0 = a0 + A16;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16(tmem, sdesc(a0 + 32u * kk), sdesc(b0 + 32u * kk), kIdesc,
                    (first && kk == 0) ? 0u : 1u);
          mma_commit(bar(B_F16_EMPTY + s));
          if (last) {
            mma_commit(bar(B_ACC_FULL));
            ++gc;
          }
        }
      }
      // every MMA issued by this thread completes before tensor memory is freed
      mma_commit(bar(B_MMA_DONE));
      mbar_wait_bounded(bar(B_MMA_DONE), 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ converters
    const int t = threadIdx.x - 64;  // 0..127
    int g = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      for (int i = 0; i < KT; ++i, ++g) {
        const int s8 = g % S8, s16 = g % S16;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S8_FULL + s8), (g / S8) & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        const uint8_t *src = sm + OFF_I8 + s8 * ST8;
        uint4 v[12];
#pragma unroll
        for (int j = 0; j < 12; ++j)
          v[j] = *reinterpret_cast<const uint4 *>(src + (j * 128 + t) * 16);
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
        for (int j = 0; j < 12; ++j) {
          const int c = j * 128 + t;  // 16-byte piece: 0..511 of A, 512..1535 of W
          const int cc = c < 512 ? c : c - 512;
          const int row = cc >> 2;
          store_f16_row_piece(dst + (c < 512 ? 0 : A16) + row * 128, row, cc & 3, v[j]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_F16_FULL + s16));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    const int r = q * 32 + lane;
    const uint32_t t_c = tmem + (uint32_t(q * 32) << 16);
    const uint32_t t_r = t_c + 256;
    const int64_t KB = a.K / 128;
    int gc = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const Tile tl = tiles[it / n_nt];
      const int e = tl.expert;
      const int n0 = (it % n_nt) * BN;
      const bool valid = r < tl.rows;
      const int64_t row = int64_t(tl.row0) + r;
      const float sa_row = (valid && !block) ? a.sa[row] : 0.0f;
      for (int c = 0; c < NC; ++c, ++gc) {
        if (!__all_sync(0xffffffffu, mbar_wait<500>(bar(B_ACC_FULL), gc & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const bool last = c == NC - 1;
        float sc[2] = {0.0f, 0.0f};
        if (block && valid) {
          const float s_a = a.sa[row * KB + c];
          const float *swp = a.sw + (int64_t(e) * (a.N / 128) + n0 / 128) * KB + c;
          sc[0] = __fmul_rn(s_a, swp[0]);
          sc[1] = __fmul_rn(s_a, swp[KB]);
        }
#pragma unroll 1
        for (int p = 0; p < BN / 32; ++p) {
          uint32_t v[32], u[32];
          tmem_ld32(t_c + 32 * p, v);
          if (c > 0) tmem_ld32(t_r + 32 * p, u);
          tmem_wait_ld();
          const float scp = sc[p >> 2];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float cv = __uint_as_float(v[j]);
            if (!f32acc) {
              const int prev = c > 0 ? int(u[j]) : 0;
              u[j] = uint32_t(prev + __float2int_rn(cv));
            } else {
              const float prev = c > 0 ? __uint_as_float(u[j]) : 0.0f;
              const float add = block ? __fmul_rn(cv, scp) : cv;
              u[j] = __float_as_uint(__fadd_rn(prev, add));
            }
          }
          if (!last) {
            tmem_st32(t_r + 32 * p, u);
          } else if (valid) {
            const int64_t n = n0 + 32 * p;
            if (a.out_type == WQ_OUT_I32) {
              int32_t *o = static_cast<int32_t *>(a.out) + row * a.N + n;
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<uint4 *>(o + j) = make_uint4(u[j], u[j + 1], u[j + 2], u[j + 3]);
            } else {
              uint32_t pk[16];
              const float *swn = a.sw + int64_t(e) * a.N + n;
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float f0, f1;
                if (block) {
                  f0 = __uint_as_float(u[j]);
                  f1 = __uint_as_float(u[j + 1]);
                } else {
                  const float c0 = f32acc ? __uint_as_float(u[j]) : __int2float_rn(int(u[j]));
                  const float c1 = f32acc ? __uint_as_float(u[j + 1]) : __int2float_rn(int(u[j + 1]));
                  f0 = __fmul_rn(__fmul_rn(c0, sa_row), __ldg(swn + j));
                  f1 = __fmul_rn(__fmul_rn(c1, sa_row), __ldg(swn + j + 1));
                }
                pk[j / 2] = pack_bf16x2(f0, f1);
              }
              uint16_t *o = static_cast<uint16_t *>(a.out) + row * a.N + n;
#pragma unroll
              for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<uint4 *>(o + 2 * j) =
                    make_uint4(pk[j], pk[j + 1], pk[j + 2], pk[j + 3]);
            }
          }
        }
        if (!last) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY));
      }
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

bool gemm_tc_supported(const GemmArgs &a) {
  return a.N % BN == 0 && a.K % BK == 0 && a.E * a.N < (int64_t(1) << 31) &&
         a.R < (int64_t(1) << 31) && tma_available();
}

// `gate`: nullptr to always run; otherwise the kernel runs only if *gate != 0.
int launch_gemm_tc(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                   const int32_t *gate, cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  CUtensorMap mA, mW;
  if (!make_tma_2d_u8(&mA, a.A, a.R, a.K, BK, BM) ||
      !make_tma_2d_u8(&mW, a.W, int64_t(a.E) * a.N, a.K, BK, BN))
    return WQ_ERR_LAUNCH;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return WQ_ERR_LAUNCH;
    attr = true;
  }
  const bool f32acc = a.scheme == WQ_SCHEME_BLOCK || a.acc == WQ_ACC_F32;
  const int chunk_stages = f32acc ? 128 / BK : 1024 / BK;
  const int64_t max_items = int64_t(max_tiles) * (a.N / BN);
  const int grid = int(max_items < num_sms() ? max_items : num_sms());
  gemm_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, st>>>(mA, mW, a, tiles, ntiles, gate, chunk_stages);
  return launched(1);
}

}  // namespace wq
