// Grouped W8A8 GEMM, CUDA-core engine: dp4a int8 dot products into exact
// int32 sums per 128-wide K tile, then the dequantization epilogues of
// "[Feature] DeepSeek V3/R1 INT8 Quantization (channel-wise)" (int32 or fp32
// accumulator) and of the Meituan article's block-wise scheme.
//
// Tile: 64 rows x 64 output channels x 128 K, 256 threads, 4x4 outputs per
// thread.  Serves the shapes the tensor-core engines do not take (output
// width not a multiple of 256 in the chunked modes) and is their exact
// fallback there.
#include "wq_tc.cuh"

namespace wq {

constexpr int kSBM = 64, kSBN = 64, kSBK = 128;

// 16 codes stored as fp16 values (32 bytes) -> 16 int8 codes (16 bytes)
__device__ __forceinline__ uint4 f16codes_to_s8(const uint4 &lo, const uint4 &hi) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int a = __half2int_rn(__ushort_as_half(uint16_t(w[2 * i] & 0xffffu)));
    const int b = __half2int_rn(__ushort_as_half(uint16_t(w[2 * i] >> 16)));
    const int c = __half2int_rn(__ushort_as_half(uint16_t(w[2 * i + 1] & 0xffffu)));
    const int d = __half2int_rn(__ushort_as_half(uint16_t(w[2 * i + 1] >> 16)));
    o[i] = pack_s8x4(a, b, c, d);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Persistent over (64-row tile, 64-channel tile) items.  kA16: A holds fp16
// codes (a.A16) instead of int8 codes (a.A).
template <bool kA16>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a, const Tile *__restrict__ tiles,
                                                        const int32_t *__restrict__ ntiles,
                                                        const int32_t *__restrict__ gate) {
  __shared__ int32_t As[kSBM][kSBK / 4 + 1];
  __shared__ int32_t Ws[kSBN][kSBK / 4 + 1];
  if (gate != nullptr && *gate == 0) return;
  const int n_nt = int(a.N / kSBN);
  const int items = ntiles[0] * n_nt;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
  const Tile tl = tiles[it / n_nt];
  const int e = tl.expert;
  const int64_t n0 = int64_t(it % n_nt) * kSBN;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t K = a.K, N = a.N;
  const int KT = int(K / kSBK);
  const int8_t *Wb = a.W + (int64_t(e) * N + n0) * K;
  const int8_t *Ab = kA16 ? nullptr : a.A + int64_t(tl.row0) * K;
  const uint16_t *Ab16 = kA16 ? a.A16 + int64_t(tl.row0) * K : nullptr;
  const bool block = a.scheme == WQ_SCHEME_BLOCK;
  const bool f32acc = block || a.acc == WQ_ACC_F32;

  int32_t ci[4][4];
  float cf[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { ci[i][j] = 0; cf[i][j] = 0.0f; }

  for (int kt = 0; kt < KT; ++kt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int idx = tid + h * 256;  // 512 16-byte pieces per operand tile
      const int r = idx >> 3, c = idx & 7;
      uint4 va = make_uint4(0, 0, 0, 0);
      if (r < tl.rows) {
        if (kA16) {
          const uint4 *p16 =
              reinterpret_cast<const uint4 *>(Ab16 + int64_t(r) * K + int64_t(kt) * kSBK) + 2 * c;
          va = f16codes_to_s8(__ldg(p16), __ldg(p16 + 1));
        } else {
          va = __ldg(reinterpret_cast<const uint4 *>(Ab + int64_t(r) * K + int64_t(kt) * kSBK) + c);
        }
      }
      const uint4 vw =
          __ldg(reinterpret_cast<const uint4 *>(Wb + int64_t(r) * K + int64_t(kt) * kSBK) + c);
      As[r][c * 4 + 0] = int32_t(va.x); As[r][c * 4 + 1] = int32_t(va.y);
      As[r][c * 4 + 2] = int32_t(va.z); As[r][c * 4 + 3] = int32_t(va.w);
      Ws[r][c * 4 + 0] = int32_t(vw.x); Ws[r][c * 4 + 1] = int32_t(vw.y);
      Ws[r][c * 4 + 2] = int32_t(vw.z); Ws[r][c * 4 + 3] = int32_t(vw.w);
    }
    __syncthreads();
    int32_t part[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part[i][j] = f32acc ? 0 : ci[i][j];
#pragma unroll 8
    for (int kw = 0; kw < kSBK / 4; ++kw) {
      int32_t av[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[ty + 16 * i][kw];
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = Ws[tx + 16 * j][kw];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = __dp4a(av[i], wv[j], part[i][j]);
    }
    if (!f32acc) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) ci[i][j] = part[i][j];
    } else if (!block) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) cf[i][j] = __fadd_rn(cf[i][j], __int2float_rn(part[i][j]));
    } else {
      // a 64-wide tile lies inside one 128-wide weight block
      const int64_t KB = K / 128;
      const float swb = a.sw[(int64_t(e) * (N / 128) + n0 / 128) * KB + kt];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = ty + 16 * i;
        const float sar = r < tl.rows ? a.sa[int64_t(tl.row0 + r) * KB + kt] : 0.0f;
        const float sc = __fmul_rn(sar, swb);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          cf[i][j] = __fadd_rn(cf[i][j], __fmul_rn(__int2float_rn(part[i][j]), sc));
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 16 * i;
    if (r >= tl.rows) continue;
    const int64_t row = tl.row0 + r;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (a.out_type == WQ_OUT_I32) {
        static_cast<int32_t *>(a.out)[row * N + n] = ci[i][j];
        continue;
      }
      float v;
      if (block) {
        v = cf[i][j];
      } else {
        const float acc = f32acc ? cf[i][j] : __int2float_rn(ci[i][j]);
        v = __fmul_rn(__fmul_rn(acc, a.sa[row]), a.sw[int64_t(e) * N + n]);
      }
      static_cast<uint16_t *>(a.out)[row * N + n] = f_to_bf16(v);
    }
  }
  __syncthreads();  // the next item overwrites As / Ws
  }
}

// `gate`: nullptr to always run; otherwise the kernel runs only if *gate != 0.
int launch_gemm_simt(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                     const int32_t *gate, cudaStream_t st) {
  if (max_tiles <= 0) return WQ_OK;
  const int64_t max_items = int64_t(max_tiles) * (a.N / kSBN);
  const int64_t cap = int64_t(8) * num_sms();
  const unsigned grid = unsigned(max_items < cap ? max_items : cap);
  if (a.A16 != nullptr) gemm_simt_kernel<true><<<grid, 256, 0, st>>>(a, tiles, ntiles, gate);
  else gemm_simt_kernel<false><<<grid, 256, 0, st>>>(a, tiles, ntiles, gate);
  return launched(1);
}

}  // namespace wq
