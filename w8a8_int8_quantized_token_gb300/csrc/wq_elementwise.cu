// Memory-bound steps of the W8A8 fused-MoE layer: activation and weight
// quantization, top-k routing, permute (scatter by expert), SiLU-and-mul with
// re-quantization, and the weighted combine.  All are coalesced 16-byte
// vector accesses with warp-shuffle reductions for the absolute maxima.
#include "wq_common.cuh"
#include "wq_tc.cuh"

namespace wq {

// ---------------------------------------------------------------------------
// Per-token and per-token-group quantization: one CTA per row, the row held
// in registers (V 16-byte vectors per thread, issued together), one scale
// per row (GV == 0: block-wide absmax) or per group of GV vectors (the GV
// consecutive lanes owning a group reduce with xor shuffles).
// (Meituan INT8 DeepSeek R1 article, 量化技术的探索: online per-token
// activation quantization of the channel-wise scheme, per-token-group
// quantization of the block-wise scheme.)  F16: the codes are written as
// fp16 values (the CTA-pair GEMM engines' input form), and with one scale
// per row also the row's squared norm.
template <int V, int GV, bool F16 = false>
__global__ void __launch_bounds__(1024) quant_row_kernel(const uint16_t *__restrict__ x, int64_t K,
                                                         int64_t ldx, void *__restrict__ q_out,
                                                         float *__restrict__ s,
                                                         int32_t *__restrict__ norm2 = nullptr) {
  __shared__ float red[32];
  __shared__ int redi[32];
  int8_t *q = static_cast<int8_t *>(q_out);
  // one vector of 8 codes: int8 bytes, or fp16 values (exact)
  auto store8 = [&](int64_t row, int idx, uint2 o) {
    if constexpr (F16) {
      uint4 w;
      tc::s8x4_to_f16x4(o.x, w.x, w.y);
      tc::s8x4_to_f16x4(o.y, w.z, w.w);
      reinterpret_cast<uint4 *>(static_cast<uint16_t *>(q_out) + row * K)[idx] = w;
    } else {
      reinterpret_cast<uint2 *>(q + row * K)[idx] = o;
    }
  };
  const int64_t row = blockIdx.x;
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * ldx);
  const int nvec = int(K >> 3);
  uint4 v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nvec) v[i] = __ldcs(xr + idx);
  }
  float a[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    a[i] = 0.0f;
    if (idx < nvec) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) a[i] = fmaxf(a[i], fabsf(f[j]));
    }
  }
  if constexpr (GV == 0) {
    float amax = a[0];
#pragma unroll
    for (int i = 1; i < V; ++i) amax = fmaxf(amax, a[i]);
    amax = block_max(amax, red);
    const float sc = quant_scale(amax);
    const float rs = __frcp_rn(sc);
    int n2 = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int idx = threadIdx.x + i * blockDim.x;
      if (idx < nvec) {
        float f[8];
        unpack8(v[i], f);
        uint2 o;
        o.x = pack_s8x4(quant_bits(f[0], sc, rs), quant_bits(f[1], sc, rs),
                        quant_bits(f[2], sc, rs), quant_bits(f[3], sc, rs));
        o.y = pack_s8x4(quant_bits(f[4], sc, rs), quant_bits(f[5], sc, rs),
                        quant_bits(f[6], sc, rs), quant_bits(f[7], sc, rs));
        store8(row, idx, o);
        if constexpr (F16) n2 = __dp4a(int(o.y), int(o.y), __dp4a(int(o.x), int(o.x), n2));
      }
    }
    if constexpr (F16) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
      const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
      if (l == 0) redi[w] = n2;
      __syncthreads();
      if (threadIdx.x == 0) {
        int t = 0;
        for (int k = 0; k < nw; ++k) t += redi[k];
        norm2[row] = t;
      }
    }
    if (threadIdx.x == 0) s[row] = sc;
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int idx = threadIdx.x + i * blockDim.x;
      float am = a[i];
#pragma unroll
      for (int o = GV / 2; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      if (idx < nvec) {
        const float sc = quant_scale(am);
        const float rs = __frcp_rn(sc);
        float f[8];
        unpack8(v[i], f);
        uint2 o;
        o.x = pack_s8x4(quant_bits(f[0], sc, rs), quant_bits(f[1], sc, rs),
                        quant_bits(f[2], sc, rs), quant_bits(f[3], sc, rs));
        o.y = pack_s8x4(quant_bits(f[4], sc, rs), quant_bits(f[5], sc, rs),
                        quant_bits(f[6], sc, rs), quant_bits(f[7], sc, rs));
        store8(row, idx, o);
        if (idx % GV == 0) s[row * (nvec / GV) + idx / GV] = sc;
      }
    }
  }
}

template <int V, bool F16>
int launch_quant_v(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group, void *q,
                   float *s, int32_t *norm2, cudaStream_t st) {
  const int64_t nvec = K / 8;
  int threads = int((nvec + V - 1) / V);
  threads = ((threads + 31) / 32) * 32;
  switch (group) {
    case 0: quant_row_kernel<V, 0, F16><<<unsigned(T), threads, 0, st>>>(x, K, ldx, q, s, norm2); break;
    case 32: quant_row_kernel<V, 4, F16><<<unsigned(T), threads, 0, st>>>(x, K, ldx, q, s, norm2); break;
    case 64: quant_row_kernel<V, 8, F16><<<unsigned(T), threads, 0, st>>>(x, K, ldx, q, s, norm2); break;
    case 128: quant_row_kernel<V, 16, F16><<<unsigned(T), threads, 0, st>>>(x, K, ldx, q, s, norm2); break;
    case 256: quant_row_kernel<V, 32, F16><<<unsigned(T), threads, 0, st>>>(x, K, ldx, q, s, norm2); break;
    default: return WQ_ERR_UNSUPPORTED;
  }
  return launched(1);
}

// Quantization fused with the permute, scatter form: one CTA per token
// quantizes its row once (the rule of quant_row_kernel) and writes the codes
// (int8, or with F16 as fp16 values), the scale(s) and, with F16 and one
// scale per row, the squared norm to each of the token's k routed rows
// pair_to_row[t * k + j] (a row outside [0, R) is skipped).  Each token is read once and the int8 codes never reach memory
// ("[WIP] feat: support cutlass_moe_fp8 for deepepmoe", review: ep_scatter
// places each token's activations at its experts' rows).
template <int V, int GV, bool F16>
__global__ void __launch_bounds__(1024) quant_scatter_kernel(
    const uint16_t *__restrict__ x, int64_t K, int64_t ldx, const int32_t *__restrict__ pair_to_row,
    int k, int64_t R, void *__restrict__ A_out, float *__restrict__ sa,
    int32_t *__restrict__ norm2) {
  __shared__ float red[32];
  __shared__ int redi[32];
  __shared__ int dst[32];
  const int64_t t = blockIdx.x;
  if (threadIdx.x < k) {
    const int r = pair_to_row[t * k + threadIdx.x];
    dst[threadIdx.x] = r >= 0 && r < R ? r : -1;
  }
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + t * ldx);
  const int nvec = int(K >> 3);
  uint4 v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nvec) v[i] = __ldcs(xr + idx);
  }
  float a[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    a[i] = 0.0f;
    if (idx < nvec) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) a[i] = fmaxf(a[i], fabsf(f[j]));
    }
  }
  float sc[V], rs[V];
  if constexpr (GV == 0) {
    float amax = a[0];
#pragma unroll
    for (int i = 1; i < V; ++i) amax = fmaxf(amax, a[i]);
    amax = block_max(amax, red);  // (its barrier also publishes dst)
#pragma unroll
    for (int i = 0; i < V; ++i) {
      sc[i] = quant_scale(amax);
      rs[i] = __frcp_rn(sc[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float am = a[i];
#pragma unroll
      for (int o = GV / 2; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      sc[i] = quant_scale(am);
      rs[i] = __frcp_rn(sc[i]);
    }
    __syncthreads();  // dst
  }
  uint4 w[V];  // F16: eight fp16 codes; else two words of int8 codes in .x, .y
  int n2 = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nvec) {
      float f[8];
      unpack8(v[i], f);
      const uint32_t lo = pack_s8x4(quant_bits(f[0], sc[i], rs[i]), quant_bits(f[1], sc[i], rs[i]),
                                    quant_bits(f[2], sc[i], rs[i]), quant_bits(f[3], sc[i], rs[i]));
      const uint32_t hi = pack_s8x4(quant_bits(f[4], sc[i], rs[i]), quant_bits(f[5], sc[i], rs[i]),
                                    quant_bits(f[6], sc[i], rs[i]), quant_bits(f[7], sc[i], rs[i]));
      if constexpr (F16) {
        tc::s8x4_to_f16x4(lo, w[i].x, w[i].y);
        tc::s8x4_to_f16x4(hi, w[i].z, w[i].w);
        if constexpr (GV == 0) n2 = __dp4a(int(hi), int(hi), __dp4a(int(lo), int(lo), n2));
      } else {
        w[i] = make_uint4(lo, hi, 0u, 0u);
      }
    }
  }
  for (int j = 0; j < k; ++j) {
    const int64_t r = dst[j];
    if (r < 0) continue;  // CTA-uniform
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int idx = threadIdx.x + i * blockDim.x;
      if (idx < nvec) {
        if constexpr (F16)
          __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(A_out) + r * K) + idx, w[i]);
        else
          __stcs(reinterpret_cast<uint2 *>(static_cast<int8_t *>(A_out) + r * K) + idx,
                 make_uint2(w[i].x, w[i].y));
        if constexpr (GV != 0) {
          if (idx % GV == 0) sa[r * (nvec / GV) + idx / GV] = sc[i];
        }
      }
    }
  }
  if constexpr (GV == 0) {
    if constexpr (F16) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
      const int wi = threadIdx.x >> 5, l = threadIdx.x & 31;
      if (l == 0) redi[wi] = n2;
      __syncthreads();
    }
    if (threadIdx.x < k) {
      const int64_t r = dst[threadIdx.x];
      if (r >= 0) {
        if constexpr (F16) {
          int tot = 0;
          for (int q = 0; q < int(blockDim.x >> 5); ++q) tot += redi[q];
          norm2[r] = tot;
        }
        sa[r] = sc[0];
      }
    }
  }
}

template <int V, bool F16>
int launch_quant_scatter_v(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                           const int32_t *pair_to_row, int k, int64_t R, void *A, float *sa,
                           int32_t *norm2, cudaStream_t st) {
  const int64_t nvec = K / 8;
  int threads = int((nvec + V - 1) / V);
  threads = ((threads + 31) / 32) * 32;
  if (threads < k) threads = ((k + 31) / 32) * 32;
#define WQ_QSC(GV) \
  quant_scatter_kernel<V, GV, F16><<<unsigned(T), threads, 0, st>>>(x, K, ldx, pair_to_row, k, R, A, sa, norm2)
  switch (group) {
    case 0: WQ_QSC(0); break;
    case 32: WQ_QSC(4); break;
    case 64: WQ_QSC(8); break;
    case 128: WQ_QSC(16); break;
    case 256: WQ_QSC(32); break;
    default: return WQ_ERR_UNSUPPORTED;
  }
#undef WQ_QSC
  return launched(1);
}

// k <= 32 destinations per token; rows up to 8192 vectors (K <= 65536)
template <bool F16>
static int launch_quant_scatter_t(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                                  const int32_t *pair_to_row, int k, int64_t R, void *A,
                                  float *sa, int32_t *norm2, cudaStream_t st) {
  if (T == 0 || K == 0) return WQ_OK;
  const int64_t nvec = K / 8;
  if (k < 1 || k > 32 || nvec > 8 * 1024 || T > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  if (group != 0 && K % group) return WQ_ERR_UNSUPPORTED;
  if (nvec <= 2 * 1024) return launch_quant_scatter_v<2, F16>(x, T, K, ldx, group, pair_to_row, k, R, A, sa, norm2, st);
  if (nvec <= 4 * 1024) return launch_quant_scatter_v<4, F16>(x, T, K, ldx, group, pair_to_row, k, R, A, sa, norm2, st);
  return launch_quant_scatter_v<8, F16>(x, T, K, ldx, group, pair_to_row, k, R, A, sa, norm2, st);
}

int launch_quant_scatter_f16(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                             const int32_t *pair_to_row, int k, int64_t R, uint16_t *A16,
                             float *sa, int32_t *norm2, cudaStream_t st) {
  return launch_quant_scatter_t<true>(x, T, K, ldx, group, pair_to_row, k, R, A16, sa, norm2, st);
}

int launch_quant_scatter_i8(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                            const int32_t *pair_to_row, int k, int64_t R, int8_t *A, float *sa,
                            cudaStream_t st) {
  return launch_quant_scatter_t<false>(x, T, K, ldx, group, pair_to_row, k, R, A, sa, nullptr, st);
}

template <bool F16>
int launch_quant_rows_t(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group, void *q,
                        float *s, int32_t *norm2, cudaStream_t st) {
  if (T == 0 || K == 0) return WQ_OK;
  const int64_t nvec = K / 8;
  if (nvec > 8 * 1024 || T > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  if (nvec <= 2 * 1024) return launch_quant_v<2, F16>(x, T, K, ldx, group, q, s, norm2, st);
  if (nvec <= 4 * 1024) return launch_quant_v<4, F16>(x, T, K, ldx, group, q, s, norm2, st);
  return launch_quant_v<8, F16>(x, T, K, ldx, group, q, s, norm2, st);
}

// Rows up to 2048 vectors (K <= 16384) take two vectors per thread (the
// fastest split measured on 7168-wide rows: 40.7 us for 8192 rows, against
// 45 us with 8 per thread and 41 us with 4); longer rows up to 8 per
// thread.  Warps are whole, so the group shuffles always see full warps, and
// a group (GV consecutive vectors, K % group == 0) never straddles the row end.
int launch_quant_rows(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group, int8_t *q,
                      float *s, cudaStream_t st) {
  return launch_quant_rows_t<false>(x, T, K, ldx, group, q, s, nullptr, st);
}

int launch_quant_rows_f16(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                          uint16_t *q16, float *s, int32_t *norm2, cudaStream_t st) {
  return launch_quant_rows_t<true>(x, T, K, ldx, group, q16, s, norm2, st);
}

// ---------------------------------------------------------------------------
// int4 weights for the w4a8 path ("Support DeepSeek-R1 w4a8 low latency
// deepep", Highlights; the page fixes no format, read as symmetric codes per
// output channel): per row a = max|w|, s = max(a, 1e-10) / 7,
// q = clamp(rint(w / s), -7, 7) with the exact quotient's rounding (as
// quant_bits; the clamp never binds, |w / s| <= 7 (1 + 2^-23)), two codes
// per byte with code 2j in the low nibble.  One CTA per row, 8 values a step.
__global__ void __launch_bounds__(256) quant_w4_row_kernel(const uint16_t *__restrict__ w, int64_t K,
                                                           uint8_t *__restrict__ q4,
                                                           float *__restrict__ s) {
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  const uint4 *src = reinterpret_cast<const uint4 *>(w + row * K);
  const int nvec = int(K >> 3);
  float amax = 0.0f;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float f[8];
    unpack8(src[v], f);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
  amax = block_max(amax, red);
  const float sc = __fdiv_rn(fmaxf(amax, 1e-10f), 7.0f);
  const float rs = __frcp_rn(sc);
  uint32_t *dst = reinterpret_cast<uint32_t *>(q4 + row * (K / 2));
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float f[8];
    unpack8(src[v], f);
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) word |= (quant_bits(f[j], sc, rs) & 0xFu) << (4 * j);
    dst[v] = word;
  }
  if (threadIdx.x == 0) s[row] = sc;
}

int launch_quant_weight_int4(const uint16_t *w, int64_t N, int64_t K, uint8_t *q4, float *s,
                             cudaStream_t st) {
  if (N <= 0) return WQ_OK;
  const int64_t nvec = K / 8;
  const int th = nvec >= 256 ? 256 : int((nvec + 31) / 32 * 32);
  quant_w4_row_kernel<<<unsigned(N), th, 0, st>>>(w, K, q4, s);
  return launched(1);
}

// ---------------------------------------------------------------------------
// FP8 (e4m3, one float32 scale per [128,128] block) -> BF16 -> INT8 weight
// conversion (Meituan INT8 article, 量化技术的探索: DeepSeek releases FP8
// weights only, so they are dequantized to BF16 and then quantized to INT8,
// per [128,128] block or per output channel).  Both steps in one pass: the
// bf16 values live only in registers.

// Two e4m3 bytes (sign, 4 exponent bits with bias 7, 3 mantissa bits; no
// infinities) -> their exact values: every e4m3 value is an fp16 value, so
// the hardware conversion to fp16 pairs is exact (byte 0 -> low half).
__device__ __forceinline__ void e4m3x2_values(uint32_t two, float &lo, float &hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(two)));
  lo = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
  hi = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
}

// 16 e4m3 bytes times one block scale, each rounded to float32 then bf16
__device__ __forceinline__ void fp8x16_to_bf16(const uint4 &w, float sc, float (&f)[16]) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v[4];
    e4m3x2_values(words[i] & 0xFFFFu, v[0], v[1]);
    e4m3x2_values(words[i] >> 16, v[2], v[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) f[4 * i + j] = bf16_to_f(f_to_bf16(__fmul_rn(v[j], sc)));
  }
}

__device__ __forceinline__ uint4 codes16(const float (&f)[16], float sc, float rs) {
  uint4 o;
  o.x = pack_s8x4(quant_bits(f[0], sc, rs), quant_bits(f[1], sc, rs), quant_bits(f[2], sc, rs),
                  quant_bits(f[3], sc, rs));
  o.y = pack_s8x4(quant_bits(f[4], sc, rs), quant_bits(f[5], sc, rs), quant_bits(f[6], sc, rs),
                  quant_bits(f[7], sc, rs));
  o.z = pack_s8x4(quant_bits(f[8], sc, rs), quant_bits(f[9], sc, rs), quant_bits(f[10], sc, rs),
                  quant_bits(f[11], sc, rs));
  o.w = pack_s8x4(quant_bits(f[12], sc, rs), quant_bits(f[13], sc, rs), quant_bits(f[14], sc, rs),
                  quant_bits(f[15], sc, rs));
  return o;
}

// channel-wise: one CTA per output row (K/16 threads, 16 bytes each)
__global__ void __launch_bounds__(1024) convert_fp8_row_kernel(const uint8_t *__restrict__ w8,
                                                               const float *__restrict__ s8,
                                                               int64_t K, int8_t *__restrict__ q,
                                                               float *__restrict__ s) {
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  const int c = threadIdx.x;  // 16-byte piece of the row
  const int nchunk = int(K >> 4);
  float f[16];
  float amax = 0.0f;
  if (c < nchunk) {
    const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(w8 + row * K) + c);
    const float sc = s8[(row >> 7) * (K >> 7) + (c >> 3)];
    fp8x16_to_bf16(w, sc, f);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = block_max(amax, red);
  const float sc = quant_scale(amax);
  const float rs = __frcp_rn(sc);
  if (c < nchunk) reinterpret_cast<uint4 *>(q + row * K)[c] = codes16(f, sc, rs);
  if (threadIdx.x == 0) s[row] = sc;
}

// block-wise: one CTA of 256 threads per [128,128] block, 4 pieces each
__global__ void __launch_bounds__(256) convert_fp8_block_kernel(const uint8_t *__restrict__ w8,
                                                                const float *__restrict__ s8,
                                                                int64_t K, int8_t *__restrict__ q,
                                                                float *__restrict__ s) {
  __shared__ float red[32];
  const int64_t kb_n = K >> 7;
  const int64_t nb = blockIdx.x / kb_n, kb = blockIdx.x % kb_n;
  const float sc8 = s8[nb * kb_n + kb];
  float f[4][16];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int p = threadIdx.x + 256 * j;  // piece: row p / 8, 16-byte column p % 8
    const int64_t r = nb * 128 + (p >> 3), col = kb * 128 + (p & 7) * 16;
    const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(w8 + r * K + col));
    fp8x16_to_bf16(w, sc8, f[j]);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[j][i]));
  }
  amax = block_max(amax, red);
  const float sc = quant_scale(amax);
  const float rs = __frcp_rn(sc);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int p = threadIdx.x + 256 * j;
    const int64_t r = nb * 128 + (p >> 3), col = kb * 128 + (p & 7) * 16;
    *reinterpret_cast<uint4 *>(q + r * K + col) = codes16(f[j], sc, rs);
  }
  if (threadIdx.x == 0) s[nb * kb_n + kb] = sc;
}

int launch_convert_fp8(const uint8_t *w8, const float *s8, int64_t N, int64_t K, int scheme,
                       int8_t *q, float *s, cudaStream_t st) {
  if (N == 0 || K == 0) return WQ_OK;
  if (scheme == WQ_SCHEME_CHANNEL) {
    if (K / 16 > 1024 || N > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
    const int threads = int(((K / 16 + 31) / 32) * 32);
    convert_fp8_row_kernel<<<unsigned(N), threads, 0, st>>>(w8, s8, K, q, s);
  } else {
    const int64_t blocks = (N / 128) * (K / 128);
    if (blocks > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
    convert_fp8_block_kernel<<<unsigned(blocks), 256, 0, st>>>(w8, s8, K, q, s);
  }
  return launched(1);
}

// ---------------------------------------------------------------------------
// [128,128] block weight quantization: one CTA of 256 threads per block,
// 8 vectors (64 elements) per thread held in registers.
__global__ void __launch_bounds__(256) quant_wblock_kernel(const uint16_t *__restrict__ w, int64_t K,
                                                           int8_t *__restrict__ q,
                                                           float *__restrict__ s) {
  __shared__ float red[32];
  const int64_t kb_n = K / 128;
  const int64_t nb = blockIdx.x / kb_n, kb = blockIdx.x % kb_n;
  uint4 v[8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + i * 256;  // vector 0..2047 of the block
    const int r = e >> 4, c = e & 15;     // 16 vectors per 128-wide row
    v[i] = __ldcs(reinterpret_cast<const uint4 *>(w + (nb * 128 + r) * K + kb * 128) + c);
    float f[8];
    unpack8(v[i], f);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
  amax = block_max(amax, red);
  const float sc = quant_scale(amax);
  const float rs = __frcp_rn(sc);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + i * 256;
    const int r = e >> 4, c = e & 15;
    float f[8];
    unpack8(v[i], f);
    uint2 o;
    o.x = pack_s8x4(quant_bits(f[0], sc, rs), quant_bits(f[1], sc, rs), quant_bits(f[2], sc, rs),
                    quant_bits(f[3], sc, rs));
    o.y = pack_s8x4(quant_bits(f[4], sc, rs), quant_bits(f[5], sc, rs), quant_bits(f[6], sc, rs),
                    quant_bits(f[7], sc, rs));
    reinterpret_cast<uint2 *>(q + (nb * 128 + r) * K + kb * 128)[c] = o;
  }
  if (threadIdx.x == 0) s[nb * kb_n + kb] = sc;
}

int launch_quant_weight_block(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *s,
                              cudaStream_t st) {
  const int64_t blocks = (N / 128) * (K / 128);
  if (blocks == 0) return WQ_OK;
  if (blocks > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  quant_wblock_kernel<<<unsigned(blocks), 256, 0, st>>>(w, K, q, s);
  return launched(1);
}

// ---------------------------------------------------------------------------
// Top-k routing: one warp per token; lane l holds logits l, l+32, ...
template <int NPER>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T, int E,
                                                    int k, int32_t *__restrict__ ids,
                                                    float *__restrict__ wout) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[NPER];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? logits[int64_t(t) * E + e] : 0.0f;
    if (e >= E) taken |= 1u << i;
  }
  float my_l = 0.0f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    // lane-local best: larger value, then lower expert id
    float bv = 0.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      if (!(taken >> i & 1u)) {
        const int e = lane + 32 * i;
        if (bi == 0x7fffffff || v[i] > bv || (v[i] == bv && e < bi)) { bv = v[i]; bi = e; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool better = (bi == 0x7fffffff) ||
                          (oi != 0x7fffffff && (ov > bv || (ov == bv && oi < bi)));
      if (better) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) { my_l = bv; my_id = bi; }
  }
  const float m = __shfl_sync(0xffffffffu, my_l, 0);
  const float e = lane < k ? exp_cw(__fsub_rn(my_l, m)) : 0.0f;
  float S = 0.0f;
  for (int j = 0; j < k; ++j) S = __fadd_rn(S, __shfl_sync(0xffffffffu, e, j));
  if (lane < k) {
    ids[int64_t(t) * k + lane] = my_id;
    wout[int64_t(t) * k + lane] = __fdiv_rn(e, S);
  }
}

int launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, cudaStream_t st) {
  if (T == 0) return WQ_OK;
  const int blocks = (T + 7) / 8;
  const int nper = (E + 31) / 32;
  if (nper <= 1) route_kernel<1><<<blocks, 256, 0, st>>>(logits, T, E, k, ids, w);
  else if (nper <= 2) route_kernel<2><<<blocks, 256, 0, st>>>(logits, T, E, k, ids, w);
  else if (nper <= 4) route_kernel<4><<<blocks, 256, 0, st>>>(logits, T, E, k, ids, w);
  else if (nper <= 8) route_kernel<8><<<blocks, 256, 0, st>>>(logits, T, E, k, ids, w);
  else if (nper <= 16) route_kernel<16><<<blocks, 256, 0, st>>>(logits, T, E, k, ids, w);
  else route_kernel<32><<<blocks, 256, 0, st>>>(logits, T, E, k, ids, w);
  return launched(1);
}

// ---------------------------------------------------------------------------
// Permute (ep_scatter): one warp per destination row, 16-byte pieces; each
// lane issues all its loads of a batch (the token's codes, usually L2
// resident since a token is read by k rows) before its streaming stores.
constexpr int kPermWarps = 8;  // rows per CTA
constexpr int kPermBatch = 8;  // 16-byte pieces in flight per lane

__global__ void __launch_bounds__(32 * kPermWarps) permute_kernel(
    const int8_t *__restrict__ q, const float *__restrict__ s, int groups, int k, int64_t K,
    const int32_t *__restrict__ sorted_pair, int64_t R, int8_t *__restrict__ A,
    float *__restrict__ sa) {
  const int lane = threadIdx.x & 31;
  const int64_t r = int64_t(blockIdx.x) * kPermWarps + (threadIdx.x >> 5);
  if (r >= R) return;
  const int p = sorted_pair[r];
  const int64_t nvec = K >> 4;
  uint4 *dst = reinterpret_cast<uint4 *>(A + r * K);
  if (p < 0) {
    for (int64_t i = lane; i < nvec; i += 32) __stcs(dst + i, make_uint4(0, 0, 0, 0));
    for (int g = lane; g < groups; g += 32) sa[r * groups + g] = 0.0f;
    return;
  }
  const int64_t tok = p / k;
  const uint4 *src = reinterpret_cast<const uint4 *>(q + tok * K);
  for (int64_t i0 = lane; i0 < nvec; i0 += 32 * kPermBatch) {
    uint4 v[kPermBatch];
#pragma unroll
    for (int u = 0; u < kPermBatch; ++u)
      if (i0 + 32 * u < nvec) v[u] = __ldg(src + i0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kPermBatch; ++u)
      if (i0 + 32 * u < nvec) __stcs(dst + i0 + 32 * u, v[u]);
  }
  for (int g = lane; g < groups; g += 32) sa[r * groups + g] = s[tok * groups + g];
}

// Permute into fp16 codes: A16[r] holds the same integers as the int8 codes
// (2 bytes each), plus the row's squared L2 norm (sum of code^2), the form the
// fast int32 GEMM engine reads.  One CTA per destination row.
__global__ void __launch_bounds__(128) permute_f16_kernel(const int8_t *__restrict__ q,
                                                          const float *__restrict__ s, int groups,
                                                          int k, int64_t K,
                                                          const int32_t *__restrict__ sorted_pair,
                                                          uint16_t *__restrict__ A16,
                                                          float *__restrict__ sa,
                                                          int32_t *__restrict__ norm2) {
  __shared__ int red[4];
  const int64_t r = blockIdx.x;
  const int p = sorted_pair[r];
  const int64_t nvec = K >> 4;  // 16 codes per piece
  uint4 *dst = reinterpret_cast<uint4 *>(A16 + r * K);
  if (p < 0) {
    for (int64_t i = threadIdx.x; i < 2 * nvec; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    for (int g = threadIdx.x; g < groups; g += blockDim.x) sa[r * groups + g] = 0.0f;
    if (threadIdx.x == 0) norm2[r] = 0;
    return;
  }
  const int64_t tok = p / k;
  const uint4 *src = reinterpret_cast<const uint4 *>(q + tok * K);
  int acc = 0;
  for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
    const uint4 v = __ldg(src + i);
    uint4 o0, o1;
    tc::s8x4_to_f16x4(v.x, o0.x, o0.y);
    tc::s8x4_to_f16x4(v.y, o0.z, o0.w);
    tc::s8x4_to_f16x4(v.z, o1.x, o1.y);
    tc::s8x4_to_f16x4(v.w, o1.z, o1.w);
    __stcs(dst + 2 * i, o0);
    __stcs(dst + 2 * i + 1, o1);
    acc = __dp4a(int(v.x), int(v.x), acc);
    acc = __dp4a(int(v.y), int(v.y), acc);
    acc = __dp4a(int(v.z), int(v.z), acc);
    acc = __dp4a(int(v.w), int(v.w), acc);
  }
  for (int g = threadIdx.x; g < groups; g += blockDim.x) sa[r * groups + g] = s[tok * groups + g];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) norm2[r] = red[0] + red[1] + red[2] + red[3];
}

int launch_permute_f16(const int8_t *q, const float *s, int groups, int k, int64_t K,
                       const int32_t *sorted_pair, int64_t R, uint16_t *A16, float *sa,
                       int32_t *norm2, cudaStream_t st) {
  if (R == 0) return WQ_OK;
  if (R > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  permute_f16_kernel<<<unsigned(R), 128, 0, st>>>(q, s, groups, k, K, sorted_pair, A16, sa, norm2);
  return launched(1);
}

int launch_permute(const int8_t *q, const float *s, int groups, int k, int64_t K,
                   const int32_t *sorted_pair, int64_t R, int8_t *A, float *sa, cudaStream_t st) {
  if (R == 0) return WQ_OK;
  if (R > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  const int64_t ctas = (R + kPermWarps - 1) / kPermWarps;
  permute_kernel<<<unsigned(ctas), 32 * kPermWarps, 0, st>>>(q, s, groups, k, K, sorted_pair, R, A,
                                                             sa);
  return launched(1);
}

// ---------------------------------------------------------------------------
// SiLU-and-mul + re-quantization: one CTA per row, V vector pairs per thread.
// F16: write the codes as fp16 values (group mode only).
template <int V, int GV, bool F16 = false>  // GV = 0: one scale per row; else lanes per group
__global__ void __launch_bounds__(1024) silu_mul_quant_kernel(
    const uint16_t *__restrict__ gu, int64_t I, const int32_t *__restrict__ masked_m, int Mmax,
    void *__restrict__ hq_out, float *__restrict__ sh) {
  int8_t *hq = static_cast<int8_t *>(hq_out);
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  if (masked_m != nullptr) {
    const int e = int(row / Mmax), m = int(row % Mmax);
    if (m >= masked_m[e]) return;  // whole CTA leaves together
  }
  const uint4 *g4 = reinterpret_cast<const uint4 *>(gu + row * 2 * I);
  const uint4 *u4 = reinterpret_cast<const uint4 *>(gu + row * 2 * I + I);
  const int nvec = int(I >> 3);
  float h[V][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    float ga[8], ua[8];
    if (idx < nvec) {
      unpack8(__ldcs(g4 + idx), ga);
      unpack8(__ldcs(u4 + idx), ua);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[i][j] = __fmul_rn(silu(ga[j]), ua[j]);
        amax = fmaxf(amax, fabsf(h[i][j]));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) h[i][j] = 0.0f;
    }
  }
  if constexpr (GV == 0) {
    amax = block_max(amax, red);
    const float sc = quant_scale(amax);
    const float rs = __frcp_rn(sc);
    uint2 *dst = reinterpret_cast<uint2 *>(hq + row * I);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int idx = threadIdx.x + i * blockDim.x;
      if (idx < nvec) {
        uint2 o;
        o.x = pack_s8x4(quant_bits(h[i][0], sc, rs), quant_bits(h[i][1], sc, rs), quant_bits(h[i][2], sc, rs),
                        quant_bits(h[i][3], sc, rs));
        o.y = pack_s8x4(quant_bits(h[i][4], sc, rs), quant_bits(h[i][5], sc, rs), quant_bits(h[i][6], sc, rs),
                        quant_bits(h[i][7], sc, rs));
        dst[idx] = o;
      }
    }
    if (threadIdx.x == 0) sh[row] = sc;
  } else {
    static_assert(V == 1, "group mode keeps one vector per thread");
    const int idx = threadIdx.x;
#pragma unroll
    for (int o = GV / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (idx < nvec) {
      const float sc = quant_scale(amax);
      const float rs = __frcp_rn(sc);
      uint2 o;
      o.x = pack_s8x4(quant_bits(h[0][0], sc, rs), quant_bits(h[0][1], sc, rs), quant_bits(h[0][2], sc, rs),
                      quant_bits(h[0][3], sc, rs));
      o.y = pack_s8x4(quant_bits(h[0][4], sc, rs), quant_bits(h[0][5], sc, rs), quant_bits(h[0][6], sc, rs),
                      quant_bits(h[0][7], sc, rs));
      if constexpr (F16) {
        uint4 w;  // the same codes as fp16 values (exact)
        tc::s8x4_to_f16x4(o.x, w.x, w.y);
        tc::s8x4_to_f16x4(o.y, w.z, w.w);
        reinterpret_cast<uint4 *>(static_cast<uint16_t *>(hq_out) + row * I)[idx] = w;
      } else {
        reinterpret_cast<uint2 *>(hq + row * I)[idx] = o;
      }
      if (idx % GV == 0) sh[row * (nvec / GV) + idx / GV] = sc;
    }
  }
}

// SiLU-and-mul + per-row re-quantization writing fp16 codes and the row's
// squared L2 norm (the fast int32 GEMM engine's input form); the arithmetic is
// that of silu_mul_quant_kernel.
template <int V>
__global__ void __launch_bounds__(1024) silu_mul_quant_f16_kernel(
    const uint16_t *__restrict__ gu, int64_t I, const int32_t *__restrict__ masked_m, int Mmax,
    uint16_t *__restrict__ hq16, float *__restrict__ sh, int32_t *__restrict__ norm2) {
  __shared__ float red[32];
  __shared__ int redi[32];
  const int64_t row = blockIdx.x;
  if (masked_m != nullptr) {
    const int e = int(row / Mmax), m = int(row % Mmax);
    if (m >= masked_m[e]) return;  // whole CTA leaves together
  }
  const uint4 *g4 = reinterpret_cast<const uint4 *>(gu + row * 2 * I);
  const uint4 *u4 = reinterpret_cast<const uint4 *>(gu + row * 2 * I + I);
  const int nvec = int(I >> 3);
  float h[V][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    float ga[8], ua[8];
    if (idx < nvec) {
      unpack8(__ldcs(g4 + idx), ga);
      unpack8(__ldcs(u4 + idx), ua);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[i][j] = __fmul_rn(silu(ga[j]), ua[j]);
        amax = fmaxf(amax, fabsf(h[i][j]));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) h[i][j] = 0.0f;
    }
  }
  amax = block_max(amax, red);
  const float sc = quant_scale(amax);
  const float rs = __frcp_rn(sc);
  uint4 *dst = reinterpret_cast<uint4 *>(hq16 + row * I);
  int n2 = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = threadIdx.x + i * blockDim.x;
    if (idx < nvec) {
      int c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = quant_code(h[i][j], sc, rs);
        n2 += c[j] * c[j];
      }
      uint4 o;
      o.x = uint32_t(__half_as_ushort(__int2half_rn(c[0]))) | (uint32_t(__half_as_ushort(__int2half_rn(c[1]))) << 16);
      o.y = uint32_t(__half_as_ushort(__int2half_rn(c[2]))) | (uint32_t(__half_as_ushort(__int2half_rn(c[3]))) << 16);
      o.z = uint32_t(__half_as_ushort(__int2half_rn(c[4]))) | (uint32_t(__half_as_ushort(__int2half_rn(c[5]))) << 16);
      o.w = uint32_t(__half_as_ushort(__int2half_rn(c[6]))) | (uint32_t(__half_as_ushort(__int2half_rn(c[7]))) << 16);
      dst[idx] = o;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (l == 0) redi[w] = n2;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < nw; ++i) t += redi[i];
    norm2[row] = t;
    sh[row] = sc;
  }
}

// ---------------------------------------------------------------------------
// The silu table in global memory (the fused GEMM1 epilogue reads it).
__global__ void __launch_bounds__(256) silu_table_kernel(float *__restrict__ tab) {
  silu_table_fill(tab, int(blockIdx.x * blockDim.x + threadIdx.x), int(gridDim.x * blockDim.x));
}

int launch_silu_table(float *tab, cudaStream_t st) {
  silu_table_kernel<<<unsigned((silu_tab::kSize + 255) / 256), 256, 0, st>>>(tab);
  return launched(1);
}

// SiLU-and-mul + re-quantization, table form (rows of at most 2048 outputs).
// Each CTA first tabulates silu(g) in shared memory (silu_tab: exact by
// construction).  Then WPR warps per row (persistent CTAs loop over rows),
// each warp a contiguous part of VPL 8-element vectors v = i*32 + lane (each
// warp access is 512 contiguous bytes): h = silu(g) * u, the row's or each
// group's absolute maximum (xor shuffles; two warps of a row exchange theirs
// through shared memory behind a named barrier), the codes (int8, or the
// same integers as fp16), the scale, and with one scale per row and norm2
// given the row's squared norm.
//
// Arithmetic in pairs (quant8: packed float32 instructions that round each
// lane as the scalar ones do, so the codes are quant_bits()'s).  fp16 codes
// are the rounded values r converted (exact: |r| <= 127, an integer);
// squared norms are sums of r * r (exact: a lane's sum stays below 2^24).

namespace silu2 {
__device__ __forceinline__ void pair_bar(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}
// silu of the two bf16 gate values of word w from the table; `miss` is set
// when either lies outside it (the entry read is then a stand-in).  ZF: +-0
// is served here too (silu(+-0) = +-0), for GEMM outputs with many exact
// zeros (int4 weights); elsewhere the select costs more than it saves.
template <bool ZF = false>
__device__ __forceinline__ void silu_pair(uint32_t w, const float *tab, float &s0, float &s1,
                                          bool &miss) {
  using namespace silu_tab;
  const uint32_t m0 = w & 0x7fffu, m1 = (w >> 16) & 0x7fffu;
  const uint32_t k0 = m0 - kLo, k1 = m1 - kLo;
  if constexpr (ZF)
    miss |= (k0 >= uint32_t(kHalf) && m0 != 0) | (k1 >= uint32_t(kHalf) && m1 != 0);
  else
    miss |= (k0 >= uint32_t(kHalf)) | (k1 >= uint32_t(kHalf));
  const uint32_t i0 = k0 + ((w >> 15) & 1u) * uint32_t(kHalf);
  const uint32_t i1 = k1 + (w >> 31) * uint32_t(kHalf);
  s0 = tab[min(i0, uint32_t(kSize - 1))];
  s1 = tab[min(i1, uint32_t(kSize - 1))];
  if constexpr (ZF) {
    s0 = m0 == 0 ? __uint_as_float((w & 0x8000u) << 16) : s0;
    s1 = m1 == 0 ? __uint_as_float(w & 0x80000000u) : s1;
  }
}
// silu of a bf16 value outside the table: the formula, except for +-0,
// whose silu is +-0 / 2 = +-0 (an integer GEMM lands on exact zeros often
// enough, more so with int4 weights, to make the formula's cost show)
__device__ __forceinline__ float silu_outside(uint32_t b) {
  return (b & 0x7fffu) == 0 ? __uint_as_float((b & 0x8000u) << 16) : silu(bf16_to_f(uint16_t(b)));
}
}  // namespace silu2

// DUAL (int8 codes, one scale per row): also the same codes as fp16 values
// in hq16, for the int8-code engine's fp16 token form; ZF: zero gates on the
// table path (silu_pair)
template <int VPL, int GV, bool F16, int WPR, bool DUAL = false, bool ZF = false>
__global__ void __launch_bounds__(512, 2) silu_mul_quant_tab_kernel(
    const uint16_t *__restrict__ gu, int64_t R, int64_t I, const int32_t *__restrict__ masked_m,
    int Mmax, void *__restrict__ hq_out, float *__restrict__ sh, int32_t *__restrict__ norm2,
    uint16_t *__restrict__ hq16 = nullptr) {
  using namespace silu2;
  static_assert(!DUAL || (!F16 && GV == 0), "the dual form writes int8 codes, one scale per row");
  static_assert(WPR == 1 || WPR == 2, "one or two warps per row");
  extern __shared__ float tab[];
  __shared__ float xmax[2][16];  // a warp's row maximum for the row's other warp
  __shared__ int xnorm[2][16];   // a warp's squared-norm part, likewise
  silu_table_fill(tab, threadIdx.x, blockDim.x);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = WPR == 2 ? (warp & 1) : 0;
  const int nvec = int(I >> 3);
  const int v0 = part * VPL * 32 + lane;
  const int64_t rstep = int64_t(gridDim.x) * (blockDim.x >> 5) / WPR;
  int par = 0;
  for (int64_t row = (int64_t(blockIdx.x) * (blockDim.x >> 5) + warp) / WPR; row < R;
       row += rstep) {
    if (masked_m != nullptr && int(row % Mmax) >= masked_m[row / Mmax]) continue;  // row-uniform
    const uint4 *g4 = reinterpret_cast<const uint4 *>(gu + row * 2 * I);
    const uint4 *u4 = reinterpret_cast<const uint4 *>(gu + row * 2 * I + I);
    uint4 gv[VPL], uv[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = v0 + i * 32;
      // past the row: gate 1.0 (in the table), up 0, so h = 0
      gv[i] = v < nvec ? __ldcs(g4 + v) : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
      uv[i] = v < nvec ? __ldcs(u4 + v) : make_uint4(0, 0, 0, 0);
    }
    float h[VPL][8];
    bool miss = false;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
      const uint32_t uw[4] = {uv[i].x, uv[i].y, uv[i].z, uv[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float s0, s1;
        silu_pair<ZF>(gw[j], tab, s0, s1, miss);
        mul2(s0, s1, bf16_lo(uw[j]), bf16_hi(uw[j]));
        h[i][2 * j] = s0;
        h[i][2 * j + 1] = s1;
      }
    }
    if (miss) {  // rare: some gate value of this lane lies outside the table; redo those
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int v = v0 + i * 32;
        if (v < nvec) {
          const uint4 g = g4[v], u = u4[v];
          const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (silu_index(gw[j] & 0xffffu) < 0)
              h[i][2 * j] = __fmul_rn(silu_outside(gw[j] & 0xffffu), bf16_lo(uw[j]));
            if (silu_index(gw[j] >> 16) < 0)
              h[i][2 * j + 1] = __fmul_rn(silu_outside(gw[j] >> 16), bf16_hi(uw[j]));
          }
        }
      }
    }
    float am[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      am[i] = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; e += 2) am[i] = fmaxf(am[i], fmaxf(fabsf(h[i][e]), fabsf(h[i][e + 1])));
    }
    float sc = 0.0f, rs = 0.0f;
    if constexpr (GV == 0) {
      float a = am[0];
#pragma unroll
      for (int i = 1; i < VPL; ++i) a = fmaxf(a, am[i]);
      a = warp_max(a);
      if constexpr (WPR == 2) {
        if (lane == 0) xmax[par][warp] = a;
        pair_bar(1 + (warp >> 1));
        a = fmaxf(a, xmax[par][warp ^ 1]);
      }
      sc = quant_scale(a);
      rs = __frcp_rn(sc);
    }
    float n0 = 0.0f, n1 = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = v0 + i * 32;
      if constexpr (GV != 0) {
        float a = am[i];
#pragma unroll
        for (int o = GV / 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        sc = quant_scale(a);
        rs = __frcp_rn(sc);
      }
      float t[8], r[8];
      quant8(h[i], sc, rs, t, r);
      if (v < nvec) {
        if constexpr (F16)
          reinterpret_cast<uint4 *>(static_cast<uint16_t *>(hq_out) + row * I)[v] = f16_codes8(r);
        else
          reinterpret_cast<uint2 *>(static_cast<int8_t *>(hq_out) + row * I)[v] = pack_codes8(t);
        if constexpr (DUAL) reinterpret_cast<uint4 *>(hq16 + row * I)[v] = f16_codes8(r);
        if constexpr (GV == 0) {
          if (norm2 != nullptr) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) sq_acc2(n0, n1, r[e], r[e + 1]);
          }
        }
        if constexpr (GV != 0) {
          if (lane % GV == 0) sh[row * (nvec / GV) + v / GV] = sc;
        }
      }
    }
    if constexpr (GV == 0) {
      if (norm2 != nullptr) {  // (uniform over the launch: both warps of a row take it)
        int n2 = __float2int_rn(__fadd_rn(n0, n1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
        if constexpr (WPR == 2) {
          if (lane == 0) xnorm[par][warp] = n2;
          pair_bar(1 + (warp >> 1));
          n2 += xnorm[par][warp ^ 1];
        }
        if (lane == 0 && part == 0) norm2[row] = n2;
      }
      if (lane == 0 && part == 0) sh[row] = sc;
    }
    par ^= 1;
  }
}

// The table kernel for rows of at most 2048 outputs; returns WQ_ERR_UNSUPPORTED
// for wider rows (the callers then take the block-per-row kernels).
// two CTAs of 16 warps per SM, fewer for short launches (rows of more than
// 1024 outputs take two warps each)
int64_t silu_tab_grid(int64_t R, int64_t nvec) {
  const int64_t rows_per_cta = 16 / (nvec > 128 ? 2 : 1);
  const int64_t grid = (R + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = 2 * int64_t(num_sms());
  return grid > cap ? cap : grid;
}

template <bool F16>
int launch_silu_tab(const uint16_t *gu, int64_t R, int64_t I, int group, const int32_t *masked_m,
                    int Mmax, void *hq, float *sh, int32_t *norm2, cudaStream_t st) {
  const int64_t nvec = I / 8;
  if (nvec > 256) return WQ_ERR_UNSUPPORTED;
  // two CTAs of 16 warps per SM (the table fits the default 48 KB of shared
  // memory), fewer for short launches; rows of more than 1024 outputs take
  // two warps each
  const int64_t grid = silu_tab_grid(R, nvec);
  const size_t smem = silu_tab::kBytes;
#define WQ_SILU_TAB(VPL, GV, WPR)                                                               \
  silu_mul_quant_tab_kernel<VPL, GV, F16, WPR><<<unsigned(grid), 512, smem, st>>>(gu, R, I, masked_m, \
                                                                                  Mmax, hq, sh, norm2)
#define WQ_SILU_TAB_G(VPL, WPR)                    \
  switch (group) {                                 \
    case 0: WQ_SILU_TAB(VPL, 0, WPR); break;       \
    case 32: WQ_SILU_TAB(VPL, 4, WPR); break;      \
    case 64: WQ_SILU_TAB(VPL, 8, WPR); break;      \
    case 128: WQ_SILU_TAB(VPL, 16, WPR); break;    \
    case 256: WQ_SILU_TAB(VPL, 32, WPR); break;    \
    default: return WQ_ERR_UNSUPPORTED;            \
  }
  if (nvec <= 32) {
    WQ_SILU_TAB_G(1, 1)
  } else if (nvec <= 64) {
    WQ_SILU_TAB_G(2, 1)
  } else if (nvec <= 128) {
    WQ_SILU_TAB_G(4, 1)
  } else {
    WQ_SILU_TAB_G(4, 2)
  }
#undef WQ_SILU_TAB_G
#undef WQ_SILU_TAB
  return launched(1);
}

// int8 codes, one scale per row, the codes again as fp16 values and each
// row's squared norm (table kernel only: rows of at most 2048 outputs)
int launch_silu_mul_quant_dual(const uint16_t *gu, int64_t R, int64_t I, const int32_t *masked_m,
                               int Mmax, int8_t *hq, uint16_t *hq16, float *sh, int32_t *norm2,
                               cudaStream_t st, bool zero_gates) {
  if (R == 0 || I == 0) return WQ_OK;
  const int64_t nvec = I / 8;
  if (R > 0x7fffffff || nvec > 256 || I % 8) return WQ_ERR_UNSUPPORTED;
  const unsigned grid = unsigned(silu_tab_grid(R, nvec));
  const size_t smem = silu_tab::kBytes;
#define WQ_SILU_DUAL(VPL, WPR)                                                                   \
  do {                                                                                          \
    if (zero_gates)                                                                             \
      silu_mul_quant_tab_kernel<VPL, 0, false, WPR, true, true><<<grid, 512, smem, st>>>(         \
          gu, R, I, masked_m, Mmax, hq, sh, norm2, hq16);                                       \
    else                                                                                        \
      silu_mul_quant_tab_kernel<VPL, 0, false, WPR, true><<<grid, 512, smem, st>>>(               \
          gu, R, I, masked_m, Mmax, hq, sh, norm2, hq16);                                       \
  } while (0)
  if (nvec <= 32) WQ_SILU_DUAL(1, 1);
  else if (nvec <= 64) WQ_SILU_DUAL(2, 1);
  else if (nvec <= 128) WQ_SILU_DUAL(4, 1);
  else WQ_SILU_DUAL(4, 2);
#undef WQ_SILU_DUAL
  return launched(1);
}

int launch_silu_mul_quant_f16(const uint16_t *gu, int64_t R, int64_t I, int group,
                              const int32_t *masked_m, int Mmax, uint16_t *hq16, float *sh,
                              int32_t *norm2, cudaStream_t st) {
  if (R == 0 || I == 0) return WQ_OK;
  if (R > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  const int64_t nvec = I / 8;
  if (nvec <= 256) return launch_silu_tab<true>(gu, R, I, group, masked_m, Mmax, hq16, sh, norm2, st);
  auto rnd = [](int64_t t) { int v = int(((t + 31) / 32) * 32); return v < 32 ? 32 : v; };
  if (group != 0) {  // per-group scales, fp16 codes, no norms
    if (nvec > 1024) return WQ_ERR_UNSUPPORTED;
    const int th = rnd(nvec);
    switch (group) {
      case 32: silu_mul_quant_kernel<1, 4, true><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq16, sh); break;
      case 64: silu_mul_quant_kernel<1, 8, true><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq16, sh); break;
      case 128: silu_mul_quant_kernel<1, 16, true><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq16, sh); break;
      case 256: silu_mul_quant_kernel<1, 32, true><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq16, sh); break;
      default: return WQ_ERR_UNSUPPORTED;
    }
    return launched(1);
  }
  if (nvec <= 1024) {
    silu_mul_quant_f16_kernel<1><<<unsigned(R), rnd(nvec), 0, st>>>(gu, I, masked_m, Mmax, hq16, sh, norm2);
  } else if (nvec <= 4096) {
    silu_mul_quant_f16_kernel<4><<<unsigned(R), rnd((nvec + 3) / 4), 0, st>>>(gu, I, masked_m, Mmax, hq16, sh, norm2);
  } else {
    return WQ_ERR_UNSUPPORTED;
  }
  return launched(1);
}


int launch_silu_mul_quant(const uint16_t *gu, int64_t R, int64_t I, int group,
                          const int32_t *masked_m, int Mmax, int8_t *hq, float *sh,
                          cudaStream_t st) {
  if (R == 0 || I == 0) return WQ_OK;
  if (R > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  const int64_t nvec = I / 8;
  if (nvec <= 256) return launch_silu_tab<false>(gu, R, I, group, masked_m, Mmax, hq, sh, nullptr, st);
  auto rnd = [](int64_t t) { int v = int(((t + 31) / 32) * 32); return v < 32 ? 32 : v; };
  if (group == 0) {
    if (nvec <= 1024) {
      silu_mul_quant_kernel<1, 0><<<unsigned(R), rnd(nvec), 0, st>>>(gu, I, masked_m, Mmax, hq, sh);
    } else if (nvec <= 4096) {
      silu_mul_quant_kernel<4, 0><<<unsigned(R), rnd((nvec + 3) / 4), 0, st>>>(gu, I, masked_m, Mmax, hq, sh);
    } else {
      return WQ_ERR_UNSUPPORTED;
    }
  } else {
    if (nvec > 1024) return WQ_ERR_UNSUPPORTED;
    const int th = rnd(nvec);
    switch (group) {
      case 32: silu_mul_quant_kernel<1, 4><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq, sh); break;
      case 64: silu_mul_quant_kernel<1, 8><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq, sh); break;
      case 128: silu_mul_quant_kernel<1, 16><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq, sh); break;
      case 256: silu_mul_quant_kernel<1, 32><<<unsigned(R), th, 0, st>>>(gu, I, masked_m, Mmax, hq, sh); break;
      default: return WQ_ERR_UNSUPPORTED;
    }
  }
  return launched(1);
}

// ---------------------------------------------------------------------------
// Squared L2 norm of each int8 row (sum of code^2, exact: at most
// 127^2 * 65536 < 2^31), one warp per row; with masked_m, rows past their
// expert's valid count are skipped.  With W16 the warp also writes the row's
// codes as fp16 values (exact), for the int8-code tensor-core engine to load
// as token tiles.
template <bool W16>
__global__ void __launch_bounds__(256) row_norm_i8_kernel(const int8_t *__restrict__ A, int64_t R,
                                                          int64_t K, const int32_t *__restrict__ masked_m,
                                                          int Mmax, int32_t *__restrict__ norm2,
                                                          uint16_t *__restrict__ out16) {
  const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  if (masked_m != nullptr && int(row % Mmax) >= masked_m[row / Mmax]) return;  // warp-uniform
  // 8-code units: lane l takes units l, l + 32, ... (8-byte loads, 256
  // contiguous bytes a warp; 16-byte fp16 stores, 512 contiguous bytes)
  const uint2 *a = reinterpret_cast<const uint2 *>(A + row * K);
  uint4 *o = W16 ? reinterpret_cast<uint4 *>(out16 + row * K) : nullptr;
  const int n8 = int(K >> 3);
  constexpr int U = 8;  // loads a lane keeps in flight
  int n = 0;
  for (int i0 = lane; i0 < n8; i0 += 32 * U) {
    uint2 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      v[u] = i0 + 32 * u < n8 ? __ldg(a + i0 + 32 * u) : make_uint2(0, 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      n = __dp4a(int(v[u].x), int(v[u].x), n);
      n = __dp4a(int(v[u].y), int(v[u].y), n);
      if constexpr (W16) {
        const int i = i0 + 32 * u;
        if (i < n8) {
          uint4 f;
          tc::s8x4_to_f16x4(v[u].x, f.x, f.y);
          tc::s8x4_to_f16x4(v[u].y, f.z, f.w);
          o[i] = f;
        }
      }
    }
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o2);
  if (lane == 0) norm2[row] = n;
}

int launch_row_norm_i8(const int8_t *A, int64_t R, int64_t K, const int32_t *masked_m, int Mmax,
                       int32_t *norm2, cudaStream_t st, uint16_t *out16) {
  if (R == 0) return WQ_OK;
  if (K % 16 || K > 65536 || (R + 7) / 8 > 0x7fffffff) return WQ_ERR_UNSUPPORTED;
  if (out16 != nullptr)
    row_norm_i8_kernel<true><<<unsigned((R + 7) / 8), 256, 0, st>>>(A, R, K, masked_m, Mmax, norm2,
                                                                   out16);
  else
    row_norm_i8_kernel<false><<<unsigned((R + 7) / 8), 256, 0, st>>>(A, R, K, masked_m, Mmax,
                                                                    norm2, nullptr);
  return launched(1);
}

// ---------------------------------------------------------------------------
// Weighted combine (the gather after the down GEMM): blockIdx.x = token,
// blockIdx.y = slice of its row.  A thread loads its 16-byte piece of all k
// routed rows first (KMAX >= k, so the loads are independent and in flight
// together), then sums w_j * y_j in j order, as the method writes it.
template <int KMAX>
__global__ void __launch_bounds__(128) combine_kernel(const uint16_t *__restrict__ y,
                                                      const int32_t *__restrict__ p2r,
                                                      const float *__restrict__ w, int k,
                                                      int64_t H, uint16_t *__restrict__ out) {
  const int64_t t = blockIdx.x;
  const int64_t nvec = H >> 3;
  int rows[KMAX];
  float wt[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    rows[j] = j < k ? p2r[t * k + j] : -1;
    wt[j] = j < k ? w[t * k + j] : 0.0f;
  }
  for (int64_t i = int64_t(blockIdx.y) * blockDim.x + threadIdx.x; i < nvec;
       i += int64_t(gridDim.y) * blockDim.x) {
    uint4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (rows[j] >= 0) v[j] = __ldcs(reinterpret_cast<const uint4 *>(y + int64_t(rows[j]) * H) + i);
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (rows[j] < 0) continue;
      float f[8];
      unpack8(v[j], f);
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = __fadd_rn(acc[c], __fmul_rn(wt[j], f[c]));
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4 *>(out + t * H)[i] = o;
  }
}

int launch_combine(const uint16_t *y, const int32_t *pair_to_row, const float *w, int T, int k,
                   int64_t H, uint16_t *out, cudaStream_t st) {
  if (T == 0 || H == 0) return WQ_OK;
  if (k > 32) return WQ_ERR_UNSUPPORTED;
  // few tokens: split each row over several CTAs so that about four CTAs per
  // SM are in flight
  const int64_t nvec = H >> 3;
  int64_t splits = (int64_t(4) * num_sms() + T - 1) / T;
  const int64_t max_splits = (nvec + 127) / 128;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  const dim3 grid{unsigned(T), unsigned(splits), 1u};
  if (k <= 8)
    combine_kernel<8><<<grid, 128, 0, st>>>(y, pair_to_row, w, k, H, out);
  else if (k <= 16)
    combine_kernel<16><<<grid, 128, 0, st>>>(y, pair_to_row, w, k, H, out);
  else
    combine_kernel<32><<<grid, 128, 0, st>>>(y, pair_to_row, w, k, H, out);
  return launched(1);
}

}  // namespace wq
