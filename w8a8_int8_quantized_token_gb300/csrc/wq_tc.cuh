// tcgen05 / TMA / mbarrier building blocks shared by the tensor-core GEMM
// kernels of libwq.so (inline PTX for sm_103a).
#pragma once

#include <cuda.h>

#include "wq_common.cuh"

namespace wq {
namespace tc {

constexpr uint64_t kTimeoutNs = 1000000000ull;  // every pipeline wait gives up after 1 s

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
// try_wait that may suspend the thread up to `ns` nanoseconds while the
// phase is incomplete (frees issue slots for busy warps)
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the 1 s limit passed or another role aborted.
template <uint32_t kSleepNs = 0>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtime();
  while (true) {
    if (kSleepNs ? mbar_try_sleep(bar, parity, kSleepNs) : mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtime() - t0 > kTimeoutNs) return false;
  }
}
// Bounded wait with no abort flag (teardown: let in-flight work land).
__device__ __forceinline__ void mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gtime();
  while (!mbar_try(bar, parity) && gtime() - t0 < kTimeoutNs) {
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
// the same copy into the shared memory of every CTA in `mask` (same offset),
// signalling each CTA's barrier at the offset of `bar`
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap *map, int x, int y,
                                               uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy accesses (TMA copies, tcgen05.mma operand reads) that another
// thread starts after a barrier hand-off.  Needed in both directions: after
// writing data an MMA will read, and after reading a slot that TMA is about
// to refill (without it a refill could land before the reads had taken
// their data, an intermittent corruption seen on sm_103a).
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
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, fp16 inputs, fp32 accumulate: A's M
// rows are tensor-memory lanes, its K elements packed two per 32-bit column
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b,
                                           uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
// M >> 4 at bit 24
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
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
// 16 consecutive columns of this warp's 32 lanes (one lane per thread)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
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
// 8 consecutive columns of this warp's 32 lanes (one lane per thread)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}
// The wait for this thread's tensor-memory loads, with the destination
// registers of the last one as operands: the compiler takes their values
// from here on, so a load may stay in flight while other registers are used.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7])
               :
               : "memory");
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


// 16 int8 codes -> 16 fp16 values written as two 16-byte pieces of a row
// of a K-major tile with 128-byte swizzle (16-byte column index ^= row % 8).
// `part` is the 16-element group of the 64-element row.
__device__ __forceinline__ void store_f16_row_piece(uint8_t *rowp, int row, int part, uint4 v) {
  uint4 o0, o1;
  s8x4_to_f16x4(v.x, o0.x, o0.y);
  s8x4_to_f16x4(v.y, o0.z, o0.w);
  s8x4_to_f16x4(v.z, o1.x, o1.y);
  s8x4_to_f16x4(v.w, o1.z, o1.w);
  const int sw = row & 7;
  *reinterpret_cast<uint4 *>(rowp + (((2 * part) ^ sw) << 4)) = o0;
  *reinterpret_cast<uint4 *>(rowp + (((2 * part + 1) ^ sw) << 4)) = o1;
}

// Two float32 products in one packed instruction, each rounded to nearest
// even exactly as a scalar multiply is (no fusion: nothing is added).
__device__ __forceinline__ void fmul2(float &x0, float &x1, float y0, float y1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(x0), "+f"(x1)
      : "f"(y0), "f"(y1));
}
// Two floats -> a bf16 pair (round to nearest even each): lo in bits 0-15
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// arrive (once) on the barrier at this offset in every CTA of `mask` when all
// prior MMAs of this thread complete
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// ---- stores from shared memory ----
// the box at (x, y) of the tensor behind `map` from the row-major box at
// shared address `src`, as one bulk async group member of this thread
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// this thread's bulk groups have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// this thread's bulk groups are complete
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// named barrier `id` over `n` threads
// Eight int4 codes (code j in bits 4j..4j+3, two's complement) -> eight int8
// codes: codes 0-3 in lo, 4-7 in hi (byte i = code i).  The even and odd
// nibbles are masked out per byte, sign-extended as (n ^ 8) - 8 per byte, and
// interleaved back into code order.
__device__ __forceinline__ void s4x8_to_s8x8(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t e = __vsub4((w & 0x0F0F0F0Fu) ^ 0x08080808u, 0x08080808u);         // codes 0,2,4,6
  const uint32_t o = __vsub4(((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u, 0x08080808u);  // codes 1,3,5,7
  lo = __byte_perm(e, o, 0x5140);
  hi = __byte_perm(e, o, 0x7362);
}

// --- distributed shared memory between the two CTAs of a cluster ---------
// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
// arrive on an mbarrier of either CTA of the cluster (address from mapa),
// releasing this thread's earlier shared-memory accesses at cluster scope
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a local barrier that the peer CTA arrives on; acquires the
// peer's released writes.  False if the 1 s limit passed or a role aborted.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag) {
  if (mbar_try_cluster(bar, parity)) return true;
  const uint64_t t0 = gtime();
  while (true) {
    if (mbar_try_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtime() - t0 > kTimeoutNs) return false;
  }
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// named barrier that also returns the AND of every participant's `pred`
__device__ __forceinline__ bool named_sync_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(uint32_t(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

}  // namespace tc

// host side: tensor-map encoder from the driver (no libcuda link needed)
bool make_tma_2d_u8(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_k,
                    int box_rows);
// 2-D 8-bit tensor [rows][K], box 128 x box_rows landing 128-byte swizzled
bool make_tma_2d_u8_sw128(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows);
bool make_tma_2d_u8_sw64(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows);
// 2-D 16-bit tensor [rows][K], box 64 x box_rows landing 128-byte swizzled
bool make_tma_2d_b16_sw128(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K,
                           int box_rows);
// 2-D 16-bit tensor [rows][cols], box box_cols x box_rows, no swizzle
bool make_tma_2d_b16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int box_cols,
                     int box_rows);
bool tma_available();
int num_sms();

}  // namespace wq
