// Grouped W8A8 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// The INT8 products of "[Feature] DeepSeek V3/R1 INT8 Quantization
// (channel-wise)" and of the Meituan article's block-wise scheme, computed
// exactly.  sm_103a has no tcgen05 integer MMA, so every int8 code q (|q| <=
// 127, and -128 also fits) is widened to an fp16 value equal to q (exact: fp16
// holds every integer below 2048) and multiplied by tcgen05.mma kind::f16
// with float32 accumulation in tensor memory.  A product is at most 127^2 =
// 16129, so any sum of at most 1024 products is an integer of magnitude below
// 2^24: every partial sum the tensor core forms is exactly representable, and
// the float32 accumulator over a chunk of at most 1024 K elements holds the
// exact int32 value.  The epilogue drains each chunk and combines it:
//   int32 accumulator:  chunks of 1024 K, run_i32 += int(chunk)   (exact C)
//   fp32 accumulator:   chunks of 128 K,  run_f32 = run_f32 + chunk
//   block scheme:       chunks of 128 K,  run_f32 = run_f32 + chunk * (sa * sw)
// which is the same arithmetic, in the same order, as the definitions in
// include/wq.h.
//
// CTA: 128 rows (one expert's rows) x 256 output channels, K in stages of 64.
//   warp 0     TMA producer: int8 A and W tiles -> int8 staging ring
//   warp 1     TMEM allocator and MMA issuer (one thread)
//   warps 2-5  converters: int8 staging -> fp16, 128-byte swizzled K-major
//   warps 6-9  epilogue: TMEM chunk -> running sum (TMEM) -> dequant -> bf16
// Tensor memory: columns [0,256) chunk accumulator, [256,512) running sum.
// Every wait is bounded (1 s); on expiry the kernel records WQ_ERR_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "wq_common.cuh"

namespace wq {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int S8 = 3, S16 = 3;
constexpr int A8 = BM * BK, B8 = BN * BK;  // int8 tile bytes
constexpr int A16 = 2 * A8, B16 = 2 * B8;  // fp16 tile bytes
constexpr int ST8 = A8 + B8, ST16 = A16 + B16;
constexpr int OFF_F16 = 0;
constexpr int OFF_I8 = OFF_F16 + S16 * ST16;
constexpr int OFF_BAR = OFF_I8 + S8 * ST8;
// barriers
constexpr int B_S8_FULL = 0, B_S8_EMPTY = S8, B_F16_FULL = 2 * S8, B_F16_EMPTY = 2 * S8 + S16,
              B_ACC_FULL = 2 * S8 + 2 * S16, B_ACC_EMPTY = B_ACC_FULL + 1,
              B_MMA_DONE = B_ACC_FULL + 2, NBAR = B_ACC_FULL + 3;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_USED = OFF_ABORT + 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
constexpr int NTHREADS = 320;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s per wait

// instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
// M >> 4 at bit 24
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the 1 s limit passed or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtime();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtime() - t0 > kTimeoutNs) return false;
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), descriptor version 1 (bit 46), layout 2 (bits 61-63)
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

#define WQ_R32(v)                                                                               \
  "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),         \
      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), \
      "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),          \
      "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),          \
      "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
#define WQ_W32(v)                                                                             \
  "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),    \
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),      \
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),    \
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),    \
      "r"(v[29]), "r"(v[30]), "r"(v[31])

// 32 consecutive columns of this warp's 32 lanes (one lane per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : WQ_R32(v)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      WQ_W32(v)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// four int8 codes -> two words of two fp16 values each, exactly:
// u = q + 128 in [0, 255]; fp16 bits 0x6400 | u encode 1024 + u;
// subtracting 1152 (0x6480) leaves q.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const GemmArgs a, const Tile *__restrict__ tiles,
                   const int32_t *__restrict__ ntiles, int chunk_stages) {
  extern __shared__ uint8_t smem_raw[];
  if (int(blockIdx.y) >= ntiles[0]) return;  // uniform over the CTA, before any setup
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_ABORT);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Tile tl = tiles[blockIdx.y];
  const int e = tl.expert;
  const int n0 = int(blockIdx.x) * BN;
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
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
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
      int issued = 0;
      for (int i = 0; i < KT; ++i) {
        const int s = i % S8;
        if (!mbar_wait(bar(B_S8_EMPTY + s), ((i / S8) & 1) ^ 1, abort_flag)) { fail(); break; }
        const uint32_t dst = base + OFF_I8 + uint32_t(s) * ST8;
        mbar_expect_tx(bar(B_S8_FULL + s), ST8);
        tma_load_2d(dst, &tmA, i * BK, tl.row0, bar(B_S8_FULL + s));
        tma_load_2d(dst + A8, &tmW, i * BK, int(int64_t(e) * a.N + n0), bar(B_S8_FULL + s));
        issued = i + 1;
      }
      if (*abort_flag) {
        // let the copies already in flight land before the CTA goes away
        for (int i = issued > S8 ? issued - S8 : 0; i < issued; ++i) {
          const uint64_t t0 = gtime();
          while (!mbar_try(bar(B_S8_FULL + i % S8), (i / S8) & 1) && gtime() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int i = 0; i < KT; ++i) {
        const int ci = i / chunk_stages;
        const bool first = (i % chunk_stages) == 0;
        const bool last = (i % chunk_stages) == chunk_stages - 1 || i == KT - 1;
        if (first && !mbar_wait(bar(B_ACC_EMPTY), (ci & 1) ^ 1, abort_flag)) { fail(); break; }
        const int s = i % S16;
        if (!mbar_wait(bar(B_F16_FULL + s), (i / S16) & 1, abort_flag)) { fail(); break; }
        tc_fence_after();
        const uint32_t a0 = base + OFF_F16 + uint32_t(s) * ST16;
        const uint32_t b0 = a0 + A16;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_f16(tmem, sdesc(a0 + 32u * kk), sdesc(b0 + 32u * kk), (first && kk == 0) ? 0u : 1u);
        mma_commit(bar(B_F16_EMPTY + s));
        if (last) mma_commit(bar(B_ACC_FULL));
      }
      // all MMAs issued by this thread complete before tensor memory is freed
      mma_commit(bar(B_MMA_DONE));
      const uint64_t t0 = gtime();
      while (!mbar_try(bar(B_MMA_DONE), 0) && gtime() - t0 < kTimeoutNs) {
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ converters
    const int t = threadIdx.x - 64;  // 0..127
    for (int i = 0; i < KT; ++i) {
      const int s8 = i % S8, s16 = i % S16;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S8_FULL + s8), (i / S8) & 1, abort_flag))) {
        fail();
        break;
      }
      const uint8_t *src = sm + OFF_I8 + s8 * ST8;
      uint4 v[12];
#pragma unroll
      for (int j = 0; j < 12; ++j)
        v[j] = *reinterpret_cast<const uint4 *>(src + (j * 128 + t) * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S8_EMPTY + s8));
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar(B_F16_EMPTY + s16), ((i / S16) & 1) ^ 1, abort_flag))) {
        fail();
        break;
      }
      uint8_t *dst = sm + OFF_F16 + s16 * ST16;
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const int c = j * 128 + t;  // 16-byte piece: 0..511 of A, 512..1535 of W
        const int cc = c < 512 ? c : c - 512;
        const int row = cc >> 2, part = cc & 3;
        uint8_t *rowp = dst + (c < 512 ? 0 : A16) + row * 128;
        uint4 o0, o1;
        s8x4_to_f16x4(v[j].x, o0.x, o0.y);
        s8x4_to_f16x4(v[j].y, o0.z, o0.w);
        s8x4_to_f16x4(v[j].z, o1.x, o1.y);
        s8x4_to_f16x4(v[j].w, o1.z, o1.w);
        const int sw = row & 7;  // 128-byte swizzle: 16-byte column index ^= row % 8
        *reinterpret_cast<uint4 *>(rowp + (((2 * part) ^ sw) << 4)) = o0;
        *reinterpret_cast<uint4 *>(rowp + (((2 * part + 1) ^ sw) << 4)) = o1;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_F16_FULL + s16));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    const int r = q * 32 + lane;
    const bool valid = r < tl.rows;
    const int64_t row = int64_t(tl.row0) + r;
    const uint32_t t_c = tmem + (uint32_t(q * 32) << 16);
    const uint32_t t_r = t_c + 256;
    const int64_t KB = a.K / 128;
    float sa_row = 0.0f;
    if (valid && !block) sa_row = a.sa[row];
    for (int c = 0; c < NC; ++c) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ACC_FULL), c & 1, abort_flag))) {
        fail();
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
              *reinterpret_cast<uint4 *>(o + 2 * j) = make_uint4(pk[j], pk[j + 1], pk[j + 2], pk[j + 3]);
          }
        }
      }
      if (!last) {
        tmem_wait_st();
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D int8 tensor [rows][K] (K contiguous), box BK x box_rows, no swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(K)};
  cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_tc_supported(const GemmArgs &a) {
  return a.N % BN == 0 && a.K % BK == 0 && a.E * a.N < (int64_t(1) << 31) &&
         a.R < (int64_t(1) << 31) && encode_fn() != nullptr;
}

int launch_gemm_tc(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                   cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  if (max_tiles > 65535) return WQ_ERR_UNSUPPORTED;
  CUtensorMap mA, mW;
  if (!make_map(&mA, a.A, a.R, a.K, BM) || !make_map(&mW, a.W, int64_t(a.E) * a.N, a.K, BN))
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
  dim3 grid(unsigned(a.N / BN), unsigned(max_tiles));
  gemm_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, st>>>(mA, mW, a, tiles, ntiles, chunk_stages);
  return cudaPeekAtLastError() == cudaSuccess ? WQ_OK : WQ_ERR_LAUNCH;
}

}  // namespace wq
