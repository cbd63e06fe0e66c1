// Internal helpers shared by the kernels of libwq.so (sm_103a).
//
// Floating point here is IEEE float32 with explicit round-to-nearest
// intrinsics (__fmul_rn, __fadd_rn, __fdiv_rn): nothing is fused or
// approximated, so every result is reproducible and matches the plain
// definitions stated in include/wq.h.  The library is also compiled with
// -fmad=false as a second guard against contraction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wq.h"

namespace wq {

constexpr int kQMax = 127;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return uint32_t(f_to_bf16(lo)) | (uint32_t(f_to_bf16(hi)) << 16);
}

// 8 bf16 in a uint4 -> 8 floats
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// exp by Cody and Waite's reduction x = n ln2 + r (ln2 split into a
// 16-significant-bit high part and the remainder), the degree-7 Taylor
// polynomial of exp(r) in Horner form, and an exact scaling by
// 2^floor(n/2) * 2^(n - floor(n/2)).  Every step is one float32 operation
// rounded to nearest even.  x >= 89 -> +inf, x <= -104 -> 0, NaN -> NaN.
__device__ __forceinline__ float exp_cw(float x) {
  if (x != x) return x;
  if (x >= 89.0f) return __uint_as_float(0x7f800000u);
  if (x <= -104.0f) return 0.0f;
  const float kLog2e = __uint_as_float(0x3fb8aa3bu);   // nearest float to 1/ln 2
  const float kLn2Hi = __uint_as_float(0x3f317200u);   // floor(ln2 * 2^16) / 2^16
  const float kLn2Lo = __uint_as_float(0x35bfbe8eu);   // nearest float to ln2 - kLn2Hi
  const float c7 = __uint_as_float(0x39500d01u);       // 1/7!
  const float c6 = __uint_as_float(0x3ab60b61u);       // 1/6!
  const float c5 = __uint_as_float(0x3c088889u);       // 1/5!
  const float c4 = __uint_as_float(0x3d2aaaabu);       // 1/4!
  const float c3 = __uint_as_float(0x3e2aaaabu);       // 1/3!
  const float c2 = 0.5f, c1 = 1.0f, c0 = 1.0f;
  float n = rintf(__fmul_rn(x, kLog2e));
  float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  float p = c7;
  p = __fadd_rn(__fmul_rn(p, r), c6);
  p = __fadd_rn(__fmul_rn(p, r), c5);
  p = __fadd_rn(__fmul_rn(p, r), c4);
  p = __fadd_rn(__fmul_rn(p, r), c3);
  p = __fadd_rn(__fmul_rn(p, r), c2);
  p = __fadd_rn(__fmul_rn(p, r), c1);
  p = __fadd_rn(__fmul_rn(p, r), c0);
  int ni = __float2int_rn(n);
  int n1 = ni >> 1;  // floor(n / 2)
  int n2 = ni - n1;
  float s1 = __uint_as_float(uint32_t(n1 + 127) << 23);
  float s2 = __uint_as_float(uint32_t(n2 + 127) << 23);
  return __fmul_rn(__fmul_rn(p, s1), s2);
}

// silu(g) = g / (1 + exp(-g))
__device__ __forceinline__ float silu(float g) {
  return __fdiv_rn(g, __fadd_rn(1.0f, exp_cw(-g)));
}

// silu(g) of every bf16 g whose magnitude lies in [2^-24, 89), of either
// sign, each entry computed with silu() itself, so a lookup returns exactly
// what the formula returns; any other g (smaller, larger, non-finite) takes
// the formula directly.  Outside that range silu is trivial anyway (g / 2,
// g, or -0), and a GEMM output rarely lands there.  Entry k holds the
// positive value with bf16 bits kLo + k, entry kHalf + k its negative.
namespace silu_tab {
constexpr uint32_t kLo = 0x3380u;        // bf16 bits of 2^-24
constexpr uint32_t kHi = 0x42B2u;        // bf16 bits of 89
constexpr int kHalf = int(kHi - kLo);    // entries of each sign
constexpr int kSize = 2 * kHalf;
constexpr int kBytes = kSize * 4;
}  // namespace silu_tab

// entries [i0, kSize) with stride `step` of the table
__device__ __forceinline__ void silu_table_fill(float *tab, int i0, int step) {
  using namespace silu_tab;
  for (int i = i0; i < kSize; i += step) {
    const uint32_t b = i < kHalf ? kLo + uint32_t(i) : (0x8000u | (kLo + uint32_t(i - kHalf)));
    tab[i] = silu(bf16_to_f(uint16_t(b)));
  }
}

// Table index of the bf16 pattern b (bits 0-15), or -1 when b lies outside
// the table
__device__ __forceinline__ int silu_index(uint32_t b) {
  using namespace silu_tab;
  const uint32_t k = (b & 0x7fffu) - kLo;  // wraps (large) below 2^-24
  return k < uint32_t(kHalf) ? int(k + (b >> 15) * uint32_t(kHalf)) : -1;
}

// Quantization scale from an absolute maximum: max(a, 1e-10) / 127.
__device__ __forceinline__ float quant_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, 1e-10f), 127.0f);
}

// One code clamp(rint(x / s), -127, 127), x / s the correctly rounded
// quotient, given rs = __frcp_rn(s) (the correctly rounded reciprocal).
//  * The clamp never binds for finite x: |x| <= amax and s = RN(amax / 127)
//    >= (amax / 127)(1 - 2^-24), so |x / s| <= 127 (1 + 2^-23) and rint gives
//    at most 127 in magnitude.
//  * Only the side of a half-integer on which the quotient falls matters:
//    y = RN(x * rs) = (x / s)(1 + e), |e| <= 2^-23 + 2^-48, lies within
//    1.52e-5 of x / s, which lies within 3.9e-6 (half an ulp below 128) of
//    RN(x / s).  When y is 2^-15 (3.05e-5) or farther from every
//    half-integer, y and RN(x / s) sit strictly inside the same interval
//    between half-integers and round to the same integer; the rare y nearer
//    than that take the exact quotient.
//  * Adding 1.5 * 2^23 rounds a float of magnitude below 2^22 to an integer
//    (to nearest, ties to even) held in the low mantissa bits, so the low
//    byte of the sum is the two's-complement code; subtracting it back gives
//    rint(y) exactly, and y - rint(y) is exact (Sterbenz) for |y| <= 128.
// Returns the sum's bits: the code is the low byte.
__device__ __forceinline__ uint32_t quant_bits(float x, float s, float rs) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  const float y = __fmul_rn(x, rs);
  float t = __fadd_rn(y, kRound);
  if (fabsf(__fsub_rn(y, __fsub_rn(t, kRound))) >= 0.499969482421875f)  // 0.5 - 2^-15
    t = __fadd_rn(__fdiv_rn(x, s), kRound);
  return __float_as_uint(t);
}
// The same code as an int in [-127, 127].
__device__ __forceinline__ int quant_code(float x, float s, float rs) {
  return int(quant_bits(x, s, rs) << 24) >> 24;
}

// Low bytes of four words -> one word (a in byte 0).
__device__ __forceinline__ uint32_t pack_s8x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Packed float32 pairs (.rn.f32x2): each lane rounds to nearest even exactly
// as the scalar instruction does, and nothing is fused unless written as fma.
__device__ __forceinline__ void mul2(float &a0, float &a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float &a0, float &a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
      " add.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
// d = a - b
__device__ __forceinline__ void sub2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " sub.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// acc += x * x for integers x whose every partial sum stays below 2^24 (exact)
__device__ __forceinline__ void sq_acc2(float &a0, float &a1, float x0, float x1) {
  asm("{\n .reg .b64 a, x, d;\n mov.b64 a, {%0, %1};\n mov.b64 x, {%2, %3};\n"
      " fma.rn.f32x2 d, x, x, a;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1));
}
// two floats -> an fp16 pair, lo in bits 0-15 (exact for the integer codes)
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight codes as quant_bits() gives them, the arithmetic in pairs: y = x *
// rs, t = y + 1.5 * 2^23 (its bits: the code in the low byte), r = t - 1.5 *
// 2^23 = rint(y) as a float, and |y - r| checked; when any of the eight lies
// within 2^-15 of one half, all eight take quant_bits() itself.
__device__ __forceinline__ void quant8(const float (&x)[8], float s, float rs, float (&t)[8],
                                       float (&r)[8]) {
  constexpr float kRound = 12582912.0f;        // 1.5 * 2^23
  constexpr float kNear = 0.499969482421875f;  // 0.5 - 2^-15
  float dm = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float y0 = x[e], y1 = x[e + 1];
    mul2(y0, y1, rs, rs);
    t[e] = y0;
    t[e + 1] = y1;
    add2(t[e], t[e + 1], kRound, kRound);
    sub2(r[e], r[e + 1], t[e], t[e + 1], kRound, kRound);
    float d0, d1;
    sub2(d0, d1, y0, y1, r[e], r[e + 1]);
    dm = fmaxf(dm, fmaxf(fabsf(d0), fabsf(d1)));
  }
  if (dm >= kNear) {  // rare
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      t[e] = __uint_as_float(quant_bits(x[e], s, rs));
      r[e] = __fsub_rn(t[e], kRound);
    }
  }
}
// The int8 codes of quant8's t as two words (element 0 in the low byte)
__device__ __forceinline__ uint2 pack_codes8(const float (&t)[8]) {
  return make_uint2(pack_s8x4(__float_as_uint(t[0]), __float_as_uint(t[1]), __float_as_uint(t[2]),
                              __float_as_uint(t[3])),
                    pack_s8x4(__float_as_uint(t[4]), __float_as_uint(t[5]), __float_as_uint(t[6]),
                              __float_as_uint(t[7])));
}
// The fp16 codes of quant8's r as four words
__device__ __forceinline__ uint4 f16_codes8(const float (&r)[8]) {
  return make_uint4(f16x2_rn(r[0], r[1]), f16x2_rn(r[2], r[3]), f16x2_rn(r[4], r[5]),
                    f16x2_rn(r[6], r[7]));
}

__device__ __forceinline__ void set_status(int32_t *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide maximum (blockDim.x a multiple of 32, at most 1024).
__device__ __forceinline__ float block_max(float v, float *red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = (l < nw) ? red[l] : 0.0f;
  return warp_max(r);
}

// A tile of rows that one grouped-GEMM CTA computes.
struct Tile {
  int expert;  // expert index
  int row0;    // first row in A / out
  int rows;    // valid rows (<= the kernel's tile height)
  int pad;
};

}  // namespace wq

// Launchers implemented in the kernel translation units (host side).
namespace wq {
// Adds n to the process-wide count of kernels the library has enqueued and
// returns WQ_OK if the last launch was accepted, else WQ_ERR_LAUNCH.
int launched(int n);
int launch_quant_rows(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group, int8_t *q,
                      float *s, cudaStream_t st);
// the same quantization writing fp16 codes (and, with group 0, row norms)
int launch_quant_rows_f16(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                          uint16_t *q16, float *s, int32_t *norm2, cudaStream_t st);
// FP8 e4m3 weights [N][K] with [N/128][K/128] float32 block scales -> bf16
// (in registers) -> int8 codes with per-row (channel) or per-block scales
int launch_convert_fp8(const uint8_t *w8, const float *s8, int64_t N, int64_t K, int scheme,
                       int8_t *q, float *s, cudaStream_t st);
int launch_quant_weight_block(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *s,
                              cudaStream_t st);
// int4 weights, one scale per row, two codes per byte (low nibble first)
int launch_quant_weight_int4(const uint16_t *w, int64_t N, int64_t K, uint8_t *q4, float *s,
                             cudaStream_t st);
int launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, cudaStream_t st);
size_t align_ws_bytes(int T, int k, int E);
int launch_align(const int32_t *ids, int T, int k, int E, int pad_m, int32_t *counts,
                 int32_t *offsets, int32_t *sorted_pair, int32_t *pair_to_row, void *ws,
                 int32_t *status, cudaStream_t st);
int launch_permute(const int8_t *q, const float *s, int groups, int k, int64_t K,
                   const int32_t *sorted_pair, int64_t R, int8_t *A, float *sa, cudaStream_t st);
int launch_silu_mul_quant(const uint16_t *gu, int64_t R, int64_t I, int group,
                          const int32_t *masked_m, int Mmax, int8_t *hq, float *sh,
                          cudaStream_t st);
int launch_quant_scatter_f16(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                             const int32_t *pair_to_row, int k, int64_t R, uint16_t *A16,
                             float *sa, int32_t *norm2, cudaStream_t st);
int launch_quant_scatter_i8(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                            const int32_t *pair_to_row, int k, int64_t R, int8_t *A, float *sa,
                            cudaStream_t st);
// SiLU-and-mul + re-quantization to int8 codes (one scale per row, rows of
// at most 2048 outputs) that also writes the codes as fp16 values and each
// row's squared norm; WQ_ERR_UNSUPPORTED for wider rows.  zero_gates: the
// GEMM output holds many exact zeros (int4 weights), served on the table path
int launch_silu_mul_quant_dual(const uint16_t *gu, int64_t R, int64_t I, const int32_t *masked_m,
                               int Mmax, int8_t *hq, uint16_t *hq16, float *sh, int32_t *norm2,
                               cudaStream_t st, bool zero_gates = false);
// squared norms of the valid rows of int8 codes A [R][K], and with out16 the
// same codes as fp16 values [R][K] (rows past a masked count untouched)
int launch_row_norm_i8(const int8_t *A, int64_t R, int64_t K, const int32_t *masked_m, int Mmax,
                       int32_t *norm2, cudaStream_t st, uint16_t *out16 = nullptr);
int launch_permute_f16(const int8_t *q, const float *s, int groups, int k, int64_t K,
                       const int32_t *sorted_pair, int64_t R, uint16_t *A16, float *sa,
                       int32_t *norm2, cudaStream_t st);
int launch_silu_mul_quant_f16(const uint16_t *gu, int64_t R, int64_t I, int group,
                              const int32_t *masked_m, int Mmax, uint16_t *hq16, float *sh,
                              int32_t *norm2, cudaStream_t st);
// silu_tab's entries into tab (silu_tab::kSize floats, global memory)
int launch_silu_table(float *tab, cudaStream_t st);
int launch_combine(const uint16_t *y, const int32_t *pair_to_row, const float *w, int T, int k,
                   int64_t H, uint16_t *out, cudaStream_t st);

// Grouped GEMM: segments come from offsets (contiguous) or masked_m (strided).
struct GemmArgs {
  const int8_t *A;           // int8 codes [R][K], or nullptr when A16 is given
  const uint16_t *A16;       // the same codes as fp16 values [R][K] (fast int32 engine)
  const int32_t *a_norm2;    // squared L2 norm of each row of A16 (with A16); with int8 A optional (tc2 reads it instead of summing)
  const float *sa;
  const int8_t *W;
  const float *sw;
  const int32_t *offsets;   // contiguous layout, or nullptr
  const int32_t *masked_m;  // masked layout, or nullptr
  int Mmax;
  int E;
  int64_t R;  // rows of A / out
  int64_t N;
  int64_t K;
  int scheme, acc, out_type;
  void *out;
  void *ws;
  int32_t *status;
  // block scheme, N = 2I gate_up weights: write SiLU-and-mul re-quantized
  // fp16 codes [R][I] and group scales [R][I/128] instead of `out`
  uint16_t *fused_hq16 = nullptr;
  float *fused_sh = nullptr;
  const float *fused_silu_tab = nullptr;  // silu_tab entries (set by the dispatcher)
  int wait_test = 0;  // failure-path test: a wait that nothing completes (block engine)
  int w4 = 0;         // W holds int4 codes, two per byte (low nibble first): [E][N][K/2]
  // the codes of A as fp16 values [R][K] beside the int8 ones (masked layer):
  // the int8-code tensor-core engine then loads its token tiles from here
  // instead of widening them again for every weight block; optional
  const uint16_t *tok16 = nullptr;
};
// The single-pass float32 engines serve both channel-wise accumulator modes.
// In the float32 mode the accumulator is the running sum, over 128-wide K
// tiles in ascending order, of each tile's int32 partial product.  Every
// prefix of that sum is an integer bounded by |a|*|w| (Cauchy-Schwarz); when
// |a|^2*|w|^2 < 2^48 (the bound the engines prove before trusting a tile)
// every conversion and addition is exact, the accumulator equals the int32
// result, and the dequantization (acc*sa)*sw is the same expression in both
// modes.  Tiles the bound does not cover go to the exact recompute, which
// takes each mode's own steps.
inline bool acc_modes_agree(const GemmArgs &a) {
  return a.scheme == WQ_SCHEME_CHANNEL && (a.acc == WQ_ACC_I32 || a.acc == WQ_ACC_F32);
}
// zero_word: two int32 words the builder sets to 0 before the engine runs
// (the exact-recompute flag and an engine's item counter), or nullptr
int launch_build_tiles(const int32_t *offsets, const int32_t *masked_m, int Mmax, int E, int BM,
                       int64_t R, Tile *tiles, int32_t *ntiles, int32_t *zero_word,
                       cudaStream_t st, int small_max = 0, Tile *small = nullptr,
                       int32_t *nsmall = nullptr, const int32_t *gate = nullptr);
size_t gemm_ws_bytes(int64_t R, int E, int Mmax, bool masked, bool silu = false);
int launch_grouped_gemm(const GemmArgs &a, cudaStream_t st);
}  // namespace wq
