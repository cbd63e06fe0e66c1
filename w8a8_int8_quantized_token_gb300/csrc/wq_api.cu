// C ABI of libwq.so: host-side argument checks, workspace carving and the
// composition of the layer's steps on one stream.  Declarations and the
// contract of every entry point are in include/wq.h.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "wq_common.cuh"

namespace wq {
int launch_gemm_simt(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                     const int32_t *gate, cudaStream_t st);
int launch_gemm_tc(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                   const int32_t *gate, cudaStream_t st);
bool gemm_tc_supported(const GemmArgs &a);
int launch_gemm_tc2(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    int32_t *redo, cudaStream_t st);
bool gemm_tc2_supported(const GemmArgs &a);
int gemm_tc2_tile_rows(const GemmArgs &a);
int launch_gemm_tc4(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    int32_t *redo, cudaStream_t st);
bool gemm_tc4_supported(const GemmArgs &a);
int launch_gemm_tc5(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    int32_t *redo, cudaStream_t st);
bool gemm_tc5_supported(const GemmArgs &a);
int gemm_tc5_tile_rows(const GemmArgs &a);
int launch_gemm_small(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                      cudaStream_t st);
int launch_gemm_tc6(const GemmArgs &a, const Tile *tiles, const int32_t *ntiles, int max_tiles,
                    cudaStream_t st);
bool gemm_tc6_supported(const GemmArgs &a);
int gemm_tc6_tile_rows();
bool gemm_small_supported(const GemmArgs &a);
int gemm_small_max_rows();
}  // namespace wq

using namespace wq;

namespace {

constexpr int kMaxDevices = 64;
int g_dev_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ_ERR_DEVICE;
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return WQ_ERR_DEVICE;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_dev_ok[dev] == 1 ? WQ_OK : WQ_ERR_DEVICE;
}

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
inline size_t rup(size_t v) { return (v + 255) & ~size_t(255); }

// Sequential carving of a caller workspace into 256-byte aligned pieces.
struct Carver {
  char *base;
  size_t used = 0;
  explicit Carver(void *p) : base(static_cast<char *>(p)) {}
  template <class T>
  T *take(size_t count) {
    T *p = reinterpret_cast<T *>(base ? base + used : nullptr);
    used += rup(count * sizeof(T));
    return p;
  }
};

#define WQ_TRY(expr)              \
  do {                            \
    int _rc = (expr);             \
    if (_rc != WQ_OK) return _rc; \
  } while (0)

int group_ok(int g) { return g == 32 || g == 64 || g == 128 || g == 256; }

int64_t gemm_max_tiles(int64_t R, int E, int Mmax, bool masked, int BM) {
  if (masked) return int64_t(E) * ((Mmax + BM - 1) / BM);
  return (R + BM - 1) / BM + E;
}

}  // namespace

namespace wq {

std::atomic<uint64_t> g_launches{0};

int launched(int n) {
  g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed);
  return cudaPeekAtLastError() == cudaSuccess ? WQ_OK : WQ_ERR_LAUNCH;
}

// Workspace of one grouped GEMM: four tile lists (64-row tiles for the
// CUDA-core engine, 128-row tiles for the chunked tensor-core engine, 256-row
// token tiles for the single-pass engines, and the small-token engine's
// tiles: at most one per expert), each with its count, and the flag the
// single-pass engines raise when a tile needs the exact recompute.
struct GemmWs {
  Tile *t64, *t128, *t256, *tsm;
  int32_t *n64, *n128, *n256, *nsm, *redo;
  int64_t m64, m128, m256, msm;
  float *silu;     // silu_tab entries for the fused GEMM1 epilogue, or nullptr
  int32_t *anorm;  // masked layout: the rows' squared norms, or nullptr
  size_t bytes;
};

GemmWs carve_gemm_ws(void *ws, int64_t R, int E, int Mmax, bool masked, bool silu = false) {
  GemmWs w;
  Carver c(ws);
  w.m64 = gemm_max_tiles(R, E, Mmax, masked, 64);
  w.m128 = gemm_max_tiles(R, E, Mmax, masked, 128);
  w.m256 = gemm_max_tiles(R, E, Mmax, masked, 256);
  w.t64 = c.take<Tile>(size_t(w.m64));
  w.n64 = c.take<int32_t>(1);
  w.t128 = c.take<Tile>(size_t(w.m128));
  w.n128 = c.take<int32_t>(1);
  w.t256 = c.take<Tile>(size_t(w.m256));
  w.n256 = c.take<int32_t>(1);
  w.msm = E;
  w.tsm = c.take<Tile>(size_t(w.msm));
  w.nsm = c.take<int32_t>(1);
  w.redo = c.take<int32_t>(2);  // recompute flag, then an engine's item counter
  w.silu = silu ? c.take<float>(silu_tab::kSize) : nullptr;
  w.anorm = masked ? c.take<int32_t>(size_t(R)) : nullptr;
  w.bytes = c.used;
  return w;
}

size_t gemm_ws_bytes(int64_t R, int E, int Mmax, bool masked, bool silu) {
  return carve_gemm_ws(nullptr, R, E, Mmax, masked, silu).bytes;
}

// A second stream per device, on which the small-token engine runs beside
// the tensor-core engine of the same GEMM launch.  Both engines are
// persistent, write disjoint rows and never wait on each other; the second
// one to start takes the SMs the first leaves idle (the tensor-core engine
// claims its items from a counter, so CTAs that start late take fewer).
// Fork and join go through events, so the pair records into a CUDA graph
// like any other stream work; the stream and events are created on first
// use, outside any capture, else both engines run one after the other.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[kMaxDevices];

template <class Side, class Main>
int fork_join(cudaStream_t st, Side &&side, Main &&main) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_side_mu);  // one fork/join pair at a time
  SideStream &sd = g_side[dev];
  if (sd.s == nullptr) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    SideStream n;
    const bool made = cudaStreamIsCapturing(st, &cs) == cudaSuccess &&
                      cs == cudaStreamCaptureStatusNone &&
                      cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) == cudaSuccess &&
                      cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) == cudaSuccess;
    if (!made) {
      cudaGetLastError();
      if (n.join) cudaEventDestroy(n.join);
      if (n.fork) cudaEventDestroy(n.fork);
      if (n.s) cudaStreamDestroy(n.s);
      WQ_TRY(side(st));
      return main(st);
    }
    sd = n;
  }
  if (cudaEventRecord(sd.fork, st) != cudaSuccess || cudaStreamWaitEvent(sd.s, sd.fork, 0) != cudaSuccess)
    return WQ_ERR_LAUNCH;
  const int rs = side(sd.s);
  if (cudaEventRecord(sd.join, sd.s) != cudaSuccess) return WQ_ERR_LAUNCH;
  const int rm = rs == WQ_OK ? main(st) : rs;
  if (cudaStreamWaitEvent(st, sd.join, 0) != cudaSuccess) return WQ_ERR_LAUNCH;
  return rm;
}

int launch_grouped_gemm(const GemmArgs &a, cudaStream_t st) {
  const bool masked = a.masked_m != nullptr;
  GemmWs w = carve_gemm_ws(a.ws, a.R, a.E, a.Mmax, masked, a.fused_hq16 != nullptr);
  const int32_t *gate = nullptr;
  if (a.w4) {
    // int4 weights (two codes a byte): the int8-code engine unpacks and widens
    // them on chip.  With |w| <= 7 and |a| <= 127, ||a||^2 ||w||^2 <=
    // 127^2 * 7^2 * K^2 < 2^48 for K <= 16384, so every float32 partial sum
    // is an exact integer, the engine's check always passes and no recompute
    // follows.  Remainders of at most 16 rows go to the small-token engine,
    // which reads the packed codes (half the bytes of int8 weights).
    if (a.A == nullptr || a.K > 16384 || !gemm_tc2_supported(a)) return WQ_ERR_UNSUPPORTED;
    const bool small = gemm_small_supported(a);
    const int rows = gemm_tc2_tile_rows(a);
    Tile *t = rows == 64 ? w.t64 : w.t256;
    int32_t *n = rows == 64 ? w.n64 : w.n256;
    const int64_t m = rows == 64 ? w.m64 : w.m256;
    WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, rows, a.R, t, n, w.redo, st,
                              small ? gemm_small_max_rows() : 0, w.tsm, w.nsm));
    auto tc2 = [&](cudaStream_t s) { return launch_gemm_tc2(a, t, n, int(m), w.redo, s); };
    if (!small) return tc2(st);
    if (rows == 64) {  // few rows per expert: the small-token engine does nearly all
      WQ_TRY(launch_gemm_small(a, w.tsm, w.nsm, int(w.msm), st));
      return tc2(st);
    }
    return fork_join(
        st, [&](cudaStream_t s) { return launch_gemm_small(a, w.tsm, w.nsm, int(w.msm), s); }, tc2);
  }
  if (a.A16 != nullptr && a.scheme == WQ_SCHEME_BLOCK) {
    // block-wise on fp16 codes: every K block's sum is exact in float32, so
    // the CTA-pair block engine needs no check and no recompute
    if (!gemm_tc6_supported(a)) return WQ_ERR_UNSUPPORTED;
    WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, gemm_tc6_tile_rows(), a.R,
                              w.t128, w.n128, nullptr, st));
    if (a.fused_hq16 == nullptr) return launch_gemm_tc6(a, w.t128, w.n128, int(w.m128), st);
    // the fused epilogue looks silu up in a table of the workspace
    WQ_TRY(launch_silu_table(w.silu, st));
    GemmArgs f = a;
    f.fused_silu_tab = w.silu;
    return launch_gemm_tc6(f, w.t128, w.n128, int(w.m128), st);
  }
  if (a.A16 != nullptr) {
    // fp16-stored codes: the CTA-pair engine, then the CUDA-core engine reading
    // fp16 codes as its exact recompute (it exits at once when *redo == 0)
    // K >= 1024: the tensor-memory-weights engine (one item of up to 320 or
    // 384 tokens per expert and weight block, so an expert a little above 256
    // rows streams its weights once; its drain is not overlapped with the
    // next item's MMAs but takes twelve warps); shorter K: the double-buffered
    // shared-memory engine
    if (a.K >= 1024 && gemm_tc5_supported(a)) {
      // token tiles of up to 320 or 384 rows (fit the 256-row list's capacity)
      WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, gemm_tc5_tile_rows(a), a.R,
                                w.t256, w.n256, w.redo, st));
      WQ_TRY(launch_gemm_tc5(a, w.t256, w.n256, int(w.m256), w.redo, st));
    } else {
      if (!gemm_tc4_supported(a)) return WQ_ERR_UNSUPPORTED;
      WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, 256, a.R, w.t256, w.n256,
                                w.redo, st));
      WQ_TRY(launch_gemm_tc4(a, w.t256, w.n256, int(w.m256), w.redo, st));
    }
    WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, 64, a.R, w.t64, w.n64, nullptr,
                              st, 0, nullptr, nullptr, w.redo));
    return launch_gemm_simt(a, w.t64, w.n64, int(w.m64), w.redo, st);
  }
  // Segment remainders of at most 16 rows (all of a decode batch's experts,
  // the ragged tail of larger ones) go to the small-token engine, which reads
  // int8 weights without widening and is exact in every mode.
  const bool small = gemm_small_supported(a);
  const int small_max = small ? gemm_small_max_rows() : 0;
  if (gemm_tc2_supported(a)) {
    // single-pass engine; it raises *redo for any tile whose float32 sums it
    // cannot prove exact, and the chunked engine below then recomputes the
    // whole launch (it exits at once when *redo == 0)
    const int rows = gemm_tc2_tile_rows(a);  // 64 (few rows per expert) or 256
    Tile *t = rows == 64 ? w.t64 : w.t256;
    int32_t *n = rows == 64 ? w.n64 : w.n256;
    const int64_t m = rows == 64 ? w.m64 : w.m256;
    WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, rows, a.R, t, n, w.redo, st,
                              small_max, w.tsm, w.nsm));
    // masked layout, channel scheme, 256-token tiles: the valid rows' squared
    // norms once per launch (unless given), so that the engine's converters,
    // which widen each token stage again for every weight block, need not
    // sum them for the exactness check.  This pass runs before the fork: on
    // the engine's own stream, beside the small-token engine, the masked
    // layer took 0.703 ms instead of 0.684.
    GemmArgs an = a;
    if (rows == 256 && w.anorm != nullptr && an.a_norm2 == nullptr &&
        a.scheme == WQ_SCHEME_CHANNEL) {
      WQ_TRY(launch_row_norm_i8(a.A, a.R, a.K, a.masked_m, a.Mmax, w.anorm, st));
      an.a_norm2 = w.anorm;
    }
    auto tc2 = [&](cudaStream_t s) { return launch_gemm_tc2(an, t, n, int(m), w.redo, s); };
    if (small && rows == 64) {  // few rows per expert: the small-token engine does nearly all
      WQ_TRY(launch_gemm_small(a, w.tsm, w.nsm, int(w.msm), st));
      WQ_TRY(tc2(st));
    } else if (small)
      WQ_TRY(fork_join(
          st, [&](cudaStream_t s) { return launch_gemm_small(a, w.tsm, w.nsm, int(w.msm), s); },
          tc2));
    else
      WQ_TRY(tc2(st));
    gate = w.redo;
  }
  if (gemm_tc_supported(a)) {
    // as the gated recompute it covers every row; on its own it leaves the
    // small remainders to the small-token engine
    const bool split = small && gate == nullptr;
    WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, 128, a.R, w.t128, w.n128,
                              nullptr, st, split ? small_max : 0, w.tsm, w.nsm, gate));
    if (split) WQ_TRY(launch_gemm_small(a, w.tsm, w.nsm, int(w.msm), st));
    return launch_gemm_tc(a, w.t128, w.n128, int(w.m128), gate, st);
  }
  WQ_TRY(launch_build_tiles(a.offsets, a.masked_m, a.Mmax, a.E, 64, a.R, w.t64, w.n64, nullptr,
                            st, 0, nullptr, nullptr, gate));
  return launch_gemm_simt(a, w.t64, w.n64, int(w.m64), gate, st);
}

}  // namespace wq

extern "C" {

int wq_init(int device) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return WQ_ERR_DEVICE;
  if (cudaSetDevice(device) != cudaSuccess) return WQ_ERR_DEVICE;
  return check_device();
}

uint64_t wq_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char *wq_status_string(int code) {
  switch (code) {
    case WQ_OK: return "ok";
    case WQ_ERR_INVALID_ARG: return "invalid argument";
    case WQ_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case WQ_ERR_DEVICE: return "no compute capability 10.3 device";
    case WQ_ERR_LAUNCH: return "CUDA launch or copy failed";
    case WQ_ERR_WORKSPACE: return "workspace too small";
    case WQ_ERR_INDEX: return "index out of range (device)";
    case WQ_ERR_TIMEOUT: return "pipeline wait timed out (device)";
    default: return "unknown status";
  }
}

int wq_quantize_per_token(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int8_t *q,
                          float *s, wq_stream_t stream) {
  if (T < 0 || K < 0 || ldx < K) return WQ_ERR_INVALID_ARG;
  if (T == 0 || K == 0) return WQ_OK;
  if (!x || !q || !s) return WQ_ERR_INVALID_ARG;
  if (K % 8 || ldx % 8 || !al16(x) || !al8(q)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_quant_rows(x, T, K, ldx, 0, q, s, stream);
}

int wq_quantize_per_token_group(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, int group,
                                int8_t *q, float *s, wq_stream_t stream) {
  if (T < 0 || K < 0 || ldx < K) return WQ_ERR_INVALID_ARG;
  if (!group_ok(group)) return WQ_ERR_UNSUPPORTED;
  if (T == 0 || K == 0) return WQ_OK;
  if (!x || !q || !s) return WQ_ERR_INVALID_ARG;
  if (K % group || ldx % 8 || !al16(x) || !al8(q)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_quant_rows(x, T, K, ldx, group, q, s, stream);
}

int wq_convert_fp8_weights(const uint8_t *w8, const float *s8, int64_t N, int64_t K, int scheme,
                           int8_t *q, float *s, wq_stream_t stream) {
  if (N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
  if (scheme != WQ_SCHEME_CHANNEL && scheme != WQ_SCHEME_BLOCK) return WQ_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return WQ_OK;
  if (!w8 || !s8 || !q || !s) return WQ_ERR_INVALID_ARG;
  if (N % 128 || K % 128 || !al16(w8) || !al16(q)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_convert_fp8(w8, s8, N, K, scheme, q, s, stream);
}

int wq_quantize_weight_block(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *s,
                             wq_stream_t stream) {
  if (N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return WQ_OK;
  if (!w || !q || !s) return WQ_ERR_INVALID_ARG;
  if (N % 128 || K % 128 || !al16(w) || !al8(q)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_quant_weight_block(w, N, K, q, s, stream);
}

int wq_route_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                  wq_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return WQ_ERR_INVALID_ARG;
  if (T == 0) return WQ_OK;
  if (!logits || !ids || !w) return WQ_ERR_INVALID_ARG;
  WQ_TRY(check_device());
  return launch_route(logits, T, E, k, ids, w, stream);
}

size_t wq_moe_align_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return align_ws_bytes(T, k, E);
}

int wq_moe_align(const int32_t *ids, int T, int k, int E, int pad_m, int32_t *counts,
                 int32_t *offsets, int32_t *sorted_pair, int32_t *pair_to_row, void *ws,
                 size_t ws_bytes, int32_t *status, wq_stream_t stream) {
  if (T < 0 || k < 1 || E < 1 || E > 4096 || pad_m < 1 || pad_m > 1024) return WQ_ERR_INVALID_ARG;
  if (int64_t(T) * k + int64_t(E) * (pad_m - 1) >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  if (!counts || !offsets || (T > 0 && (!ids || !sorted_pair || !pair_to_row)))
    return WQ_ERR_INVALID_ARG;
  if (ws_bytes < align_ws_bytes(T, k, E) || (T > 0 && !ws)) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  return launch_align(ids, T, k, E, pad_m, counts, offsets, sorted_pair, pair_to_row, ws, status,
                      stream);
}

int wq_moe_permute(const int8_t *q, const float *s, int groups, int T, int k, int64_t K,
                   const int32_t *sorted_pair, int64_t R, int8_t *A, float *sa,
                   wq_stream_t stream) {
  if (groups < 1 || T < 0 || k < 1 || K < 0 || R < 0) return WQ_ERR_INVALID_ARG;
  if (R == 0) return WQ_OK;
  if (!sorted_pair || !A || !sa || (T > 0 && (!q || !s))) return WQ_ERR_INVALID_ARG;
  if (K % 16 || !al16(q) || !al16(A)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_permute(q, s, groups, k, K, sorted_pair, R, A, sa, stream);
}

static int check_gemm_common(const int8_t *W, const float *sw, int E, int64_t N, int64_t K,
                             int scheme, int acc, int out_type, const void *out) {
  if (E < 1 || N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
  if (scheme != WQ_SCHEME_CHANNEL && scheme != WQ_SCHEME_BLOCK) return WQ_ERR_INVALID_ARG;
  if (acc != WQ_ACC_I32 && acc != WQ_ACC_F32) return WQ_ERR_INVALID_ARG;
  if (out_type != WQ_OUT_BF16 && out_type != WQ_OUT_I32) return WQ_ERR_INVALID_ARG;
  if (out_type == WQ_OUT_I32 && (scheme != WQ_SCHEME_CHANNEL || acc != WQ_ACC_I32))
    return WQ_ERR_INVALID_ARG;
  if (!W || !sw || !out) return WQ_ERR_INVALID_ARG;
  if (N % 128 || K % 128 || N == 0 || K == 0) return WQ_ERR_UNSUPPORTED;
  if (!al16(W) || !al16(out)) return WQ_ERR_UNSUPPORTED;
  return WQ_OK;
}

size_t wq_grouped_gemm_workspace_size(int64_t R, int E) {
  if (R < 0 || E < 1) return 0;
  return gemm_ws_bytes(R, E, 0, false);
}

}  // extern "C"

namespace wq {
// The host-side argument checks of the grouped GEMM on int8 codes, shared by
// the workspace entry point and the allocation-free one (which must reject
// the same calls with the same codes).  WQ_OK with R == 0 means "nothing to
// do".
int check_grouped_gemm_args(const int8_t *A, const float *sa, const int8_t *W, const float *sw,
                            const int32_t *offsets, int E, int64_t R, int64_t N, int64_t K,
                            int scheme, int acc, int out_type, const void *out) {
  if (R < 0 || E > 4096) return WQ_ERR_INVALID_ARG;
  if (R == 0) return WQ_OK;
  WQ_TRY(check_gemm_common(W, sw, E, N, K, scheme, acc, out_type, out));
  if (!A || !sa || !offsets) return WQ_ERR_INVALID_ARG;
  if (!al16(A)) return WQ_ERR_UNSUPPORTED;
  if (R >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  return WQ_OK;
}
}  // namespace wq

extern "C" {

int wq_grouped_gemm_w8a8(const int8_t *A, const float *sa, const int8_t *W, const float *sw,
                         const int32_t *offsets, int E, int64_t R, int64_t N, int64_t K,
                         int scheme, int acc, int out_type, void *out, void *ws, size_t ws_bytes,
                         int32_t *status, wq_stream_t stream) {
  WQ_TRY(check_grouped_gemm_args(A, sa, W, sw, offsets, E, R, N, K, scheme, acc, out_type, out));
  if (R == 0) return WQ_OK;
  if (ws_bytes < gemm_ws_bytes(R, E, 0, false) || !ws) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  GemmArgs a{A, nullptr, nullptr, sa, W, sw, offsets, nullptr, 0, E, R, N, K, scheme, acc, out_type, out, ws, status};
  return launch_grouped_gemm(a, stream);
}

int wq_moe_permute_f16(const int8_t *q, const float *s, int groups, int T, int k, int64_t K,
                       const int32_t *sorted_pair, int64_t R, uint16_t *A16, float *sa,
                       int32_t *norm2, wq_stream_t stream) {
  if (groups < 1 || T < 0 || k < 1 || K < 0 || R < 0) return WQ_ERR_INVALID_ARG;
  if (R == 0) return WQ_OK;
  if (!sorted_pair || !A16 || !sa || !norm2 || (T > 0 && (!q || !s))) return WQ_ERR_INVALID_ARG;
  if (K % 16 || !al16(q) || !al16(A16)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_permute_f16(q, s, groups, k, K, sorted_pair, R, A16, sa, norm2, stream);
}

int wq_silu_mul_quant_f16(const uint16_t *gu, int64_t R, int64_t I, int group, uint16_t *hq16,
                          float *sh, int32_t *norm2, wq_stream_t stream) {
  if (R < 0 || I < 0) return WQ_ERR_INVALID_ARG;
  if (group != 0 && !group_ok(group)) return WQ_ERR_UNSUPPORTED;
  if (R == 0 || I == 0) return WQ_OK;
  if (!gu || !hq16 || !sh || (group == 0 && !norm2)) return WQ_ERR_INVALID_ARG;
  if (I % 8 || (group && I % group) || !al16(gu) || !al16(hq16)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_silu_mul_quant_f16(gu, R, I, group, nullptr, 0, hq16, sh, norm2, stream);
}

int wq_grouped_gemm_w8a8_f16codes(const uint16_t *A16, const int32_t *a_norm2, const float *sa,
                                  const int8_t *W, const float *sw, const int32_t *offsets, int E,
                                  int64_t R, int64_t N, int64_t K, int scheme, int acc,
                                  int out_type, void *out, void *ws, size_t ws_bytes,
                                  int32_t *status, wq_stream_t stream) {
  if (R < 0 || E > 4096) return WQ_ERR_INVALID_ARG;
  if (R == 0) return WQ_OK;
  WQ_TRY(check_gemm_common(W, sw, E, N, K, scheme, acc, out_type, out));
  const bool blk = scheme == WQ_SCHEME_BLOCK;
  if (!A16 || (!blk && !a_norm2) || !sa || !offsets) return WQ_ERR_INVALID_ARG;
  if (!al16(A16) || N % 256 || K > 65536 || (blk && K % 128)) return WQ_ERR_UNSUPPORTED;
  if (R >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  if (ws_bytes < gemm_ws_bytes(R, E, 0, false) || !ws) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  GemmArgs a{nullptr, A16, a_norm2, sa, W, sw, offsets, nullptr, 0, E, R, N, K, scheme,
             acc, out_type, out, ws, status};
  return launch_grouped_gemm(a, stream);
}

int wq_selftest_wait_timeout(const uint16_t *A16, const float *sa, const int8_t *W, const float *sw,
                             const int32_t *offsets, int E, int64_t R, int64_t N, int64_t K,
                             void *out, void *ws, size_t ws_bytes, int32_t *status,
                             wq_stream_t stream) {
  if (R <= 0 || E < 1 || E > 4096 || !status) return WQ_ERR_INVALID_ARG;
  WQ_TRY(check_gemm_common(W, sw, E, N, K, WQ_SCHEME_BLOCK, WQ_ACC_F32, WQ_OUT_BF16, out));
  if (!A16 || !sa || !offsets) return WQ_ERR_INVALID_ARG;
  if (!al16(A16) || N % 256 || K > 65536 || R >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  if (ws_bytes < gemm_ws_bytes(R, E, 0, false) || !ws) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  GemmArgs a{nullptr, A16, nullptr, sa, W, sw, offsets, nullptr, 0, E, R, N, K, WQ_SCHEME_BLOCK,
             WQ_ACC_F32, WQ_OUT_BF16, out, ws, status};
  a.wait_test = 1;
  return launch_grouped_gemm(a, stream);
}

size_t wq_grouped_gemm_silu_quant_workspace_size(int64_t R, int E) {
  if (R < 0 || E < 1) return 0;
  return gemm_ws_bytes(R, E, 0, false, true);
}

int wq_grouped_gemm_w8a8_silu_quant_f16codes(const uint16_t *A16, const float *sa, const int8_t *W13,
                                             const float *sw13, const int32_t *offsets, int E,
                                             int64_t R, int64_t I, int64_t K, int scheme,
                                             uint16_t *hq16, float *sh, void *ws, size_t ws_bytes,
                                             int32_t *status, wq_stream_t stream) {
  if (R < 0 || E > 4096 || I <= 0) return WQ_ERR_INVALID_ARG;
  if (scheme == WQ_SCHEME_CHANNEL) return WQ_ERR_UNSUPPORTED;  // needs the whole row's maximum
  if (R == 0) return WQ_OK;
  WQ_TRY(check_gemm_common(W13, sw13, E, 2 * I, K, scheme, WQ_ACC_F32, WQ_OUT_BF16, hq16));
  if (!A16 || !sa || !offsets || !sh) return WQ_ERR_INVALID_ARG;
  if (!al16(A16) || I % 128 || K > 65536) return WQ_ERR_UNSUPPORTED;
  if (R >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  if (ws_bytes < gemm_ws_bytes(R, E, 0, false, true) || !ws) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  GemmArgs a{nullptr, A16, nullptr, sa, W13, sw13, offsets, nullptr, 0, E, R, 2 * I, K, scheme,
             WQ_ACC_F32, WQ_OUT_BF16, nullptr, ws, status};
  a.fused_hq16 = hq16;
  a.fused_sh = sh;
  return launch_grouped_gemm(a, stream);
}

int wq_quantize_per_token_f16(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, uint16_t *q16,
                              float *s, int32_t *norm2, wq_stream_t stream) {
  if (T < 0 || K < 0 || ldx < K) return WQ_ERR_INVALID_ARG;
  if (T == 0 || K == 0) return WQ_OK;
  if (!x || !q16 || !s || !norm2) return WQ_ERR_INVALID_ARG;
  if (K % 8 || ldx % 8 || !al16(x) || !al16(q16)) return WQ_ERR_UNSUPPORTED;
  if (K > 65536) return WQ_ERR_UNSUPPORTED;  // squared norms stay below 2^31
  WQ_TRY(check_device());
  return launch_quant_rows_f16(x, T, K, ldx, 0, q16, s, norm2, stream);
}

int wq_quantize_permute(const uint16_t *x, int64_t T, int64_t K, int group,
                        const int32_t *pair_to_row, int k, int64_t R, int8_t *A, float *sa,
                        wq_stream_t stream) {
  if (T < 0 || K < 0 || k < 1 || k > 32 || R < 0) return WQ_ERR_INVALID_ARG;
  if (group != 0 && group != 32 && group != 64 && group != 128 && group != 256)
    return WQ_ERR_INVALID_ARG;
  if (T == 0 || K == 0 || R == 0) return WQ_OK;
  if (!x || !pair_to_row || !A || !sa) return WQ_ERR_INVALID_ARG;
  if (K % 8 || (group != 0 && K % group) || !al16(x) || !al16(A)) return WQ_ERR_UNSUPPORTED;
  if (K > 65536) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_quant_scatter_i8(x, T, K, K, group, pair_to_row, k, R, A, sa, stream);
}

int wq_quantize_permute_f16(const uint16_t *x, int64_t T, int64_t K, int group,
                            const int32_t *pair_to_row, int k, int64_t R, uint16_t *A16,
                            float *sa, int32_t *norm2, wq_stream_t stream) {
  if (T < 0 || K < 0 || k < 1 || k > 32 || R < 0) return WQ_ERR_INVALID_ARG;
  if (group != 0 && group != 32 && group != 64 && group != 128 && group != 256)
    return WQ_ERR_INVALID_ARG;
  if (T == 0 || K == 0 || R == 0) return WQ_OK;
  if (!x || !pair_to_row || !A16 || !sa || (group == 0 && !norm2)) return WQ_ERR_INVALID_ARG;
  if (K % 8 || (group != 0 && K % group) || !al16(x) || !al16(A16)) return WQ_ERR_UNSUPPORTED;
  if (K > 65536) return WQ_ERR_UNSUPPORTED;  // squared norms stay below 2^31
  WQ_TRY(check_device());
  return launch_quant_scatter_f16(x, T, K, K, group, pair_to_row, k, R, A16, sa, norm2, stream);
}

size_t wq_grouped_gemm_masked_workspace_size(int E, int Mmax) {
  if (E < 1 || Mmax < 0) return 0;
  return gemm_ws_bytes(int64_t(E) * Mmax, E, Mmax, true);
}

int wq_grouped_gemm_w8a8_masked(const int8_t *A, const float *sa, const int32_t *masked_m, int E,
                                int Mmax, const int8_t *W, const float *sw, int64_t N, int64_t K,
                                int scheme, int acc, int out_type, void *out, void *ws,
                                size_t ws_bytes, int32_t *status, wq_stream_t stream) {
  if (Mmax < 0 || E > 4096) return WQ_ERR_INVALID_ARG;
  if (Mmax == 0) return WQ_OK;
  WQ_TRY(check_gemm_common(W, sw, E, N, K, scheme, acc, out_type, out));
  if (!A || !sa || !masked_m) return WQ_ERR_INVALID_ARG;
  if (!al16(A)) return WQ_ERR_UNSUPPORTED;
  const int64_t R = int64_t(E) * Mmax;
  if (R >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  if (ws_bytes < gemm_ws_bytes(R, E, Mmax, true) || !ws) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  GemmArgs a{A, nullptr, nullptr, sa, W, sw, nullptr, masked_m, Mmax, E, R, N, K, scheme, acc, out_type, out, ws,
             status};
  return launch_grouped_gemm(a, stream);
}

int wq_silu_mul_quant(const uint16_t *gu, int64_t R, int64_t I, int group, int8_t *hq, float *sh,
                      wq_stream_t stream) {
  if (R < 0 || I < 0) return WQ_ERR_INVALID_ARG;
  if (group != 0 && !group_ok(group)) return WQ_ERR_UNSUPPORTED;
  if (R == 0 || I == 0) return WQ_OK;
  if (!gu || !hq || !sh) return WQ_ERR_INVALID_ARG;
  if (I % 8 || (group && I % group) || !al16(gu) || !al8(hq)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_silu_mul_quant(gu, R, I, group, nullptr, 0, hq, sh, stream);
}

int wq_moe_combine(const uint16_t *y, const int32_t *pair_to_row, const float *w, int T, int k,
                   int64_t H, uint16_t *out, wq_stream_t stream) {
  if (T < 0 || k < 1 || H < 0) return WQ_ERR_INVALID_ARG;
  if (T == 0 || H == 0) return WQ_OK;
  if (!y || !pair_to_row || !w || !out) return WQ_ERR_INVALID_ARG;
  if (k > 32 || H % 8 || !al16(y) || !al16(out)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_combine(y, pair_to_row, w, T, k, H, out, stream);
}

// ---------------------------------------------------------------------------
// The layer

namespace {

struct FwdBufs {
  int32_t *ids;
  float *w;
  int8_t *q;
  float *s;
  int32_t *counts, *offsets, *sorted_pair, *pair_to_row;
  void *align_ws;
  int8_t *A;  // int8 codes, or fp16 codes (the buffer holds either)
  float *sa;
  int32_t *anorm;
  uint16_t *gu;
  int8_t *hq;  // int8 codes, or fp16 codes
  float *sh;
  int32_t *hnorm;
  uint16_t *y;
  void *gemm_ws;
  size_t gemm_ws_bytes;
};

size_t carve_forward(void *ws, int T, int H, int I, int E, int k, int scheme, FwdBufs *b) {
  Carver c(ws);
  const int64_t R = int64_t(T) * k;
  const int64_t g1 = scheme == WQ_SCHEME_BLOCK ? H / 128 : 1;
  const int64_t g2 = scheme == WQ_SCHEME_BLOCK ? I / 128 : 1;
  FwdBufs t;
  t.ids = c.take<int32_t>(R);
  t.w = c.take<float>(R);
  t.q = c.take<int8_t>(size_t(T) * H);
  t.s = c.take<float>(size_t(T) * g1);
  t.counts = c.take<int32_t>(E);
  t.offsets = c.take<int32_t>(E + 1);
  t.sorted_pair = c.take<int32_t>(R);
  t.pair_to_row = c.take<int32_t>(R);
  t.align_ws = c.take<char>(align_ws_bytes(T, k, E));
  t.A = c.take<int8_t>(size_t(R) * H * 2);
  t.sa = c.take<float>(size_t(R) * g1);
  t.anorm = c.take<int32_t>(size_t(R));
  t.gu = c.take<uint16_t>(size_t(R) * 2 * I);
  t.hq = c.take<int8_t>(size_t(R) * I * 2);
  t.sh = c.take<float>(size_t(R) * g2);
  t.hnorm = c.take<int32_t>(size_t(R));
  t.y = c.take<uint16_t>(size_t(R) * H);
  t.gemm_ws_bytes = gemm_ws_bytes(R, E, 0, false);
  t.gemm_ws = c.take<char>(t.gemm_ws_bytes);
  if (b) *b = t;
  return c.used;
}

int check_forward_shape(int T, int H, int I, int E, int k, int scheme, int acc) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E)
    return WQ_ERR_INVALID_ARG;
  if (scheme != WQ_SCHEME_CHANNEL && scheme != WQ_SCHEME_BLOCK) return WQ_ERR_INVALID_ARG;
  if (acc != WQ_ACC_I32 && acc != WQ_ACC_F32) return WQ_ERR_INVALID_ARG;
  if (H % 128 || I % 128) return WQ_ERR_UNSUPPORTED;
  if (int64_t(T) * k >= (int64_t(1) << 31) / 2) return WQ_ERR_UNSUPPORTED;
  return WQ_OK;
}

int run_forward(const uint16_t *x, const float *logits, const int8_t *W13, const float *sw13,
                const int8_t *W2, const float *sw2, int T, int H, int I, int E, int k, int scheme,
                int acc, uint16_t *out, const FwdBufs &b, int32_t *status, cudaStream_t st) {
  const int64_t R = int64_t(T) * k;
  const bool blk = scheme == WQ_SCHEME_BLOCK;
  WQ_TRY(launch_route(logits, T, E, k, b.ids, b.w, st));
  WQ_TRY(launch_align(b.ids, T, k, E, 1, b.counts, b.offsets, b.sorted_pair, b.pair_to_row,
                      b.align_ws, status, st));
  // with many rows per expert and widths that are multiples of 256 the
  // activation codes travel as fp16 values (the CTA-pair GEMM engines; row
  // norms for the channel-wise exactness check); otherwise int8 codes
  GemmArgs probe{nullptr, reinterpret_cast<const uint16_t *>(b.A), b.anorm, b.sa, W13, sw13,
                 b.offsets, nullptr, 0, E, R, int64_t(2) * I, H, scheme, acc, WQ_OUT_BF16, b.gu,
                 b.gemm_ws, status};
  // (with few rows per expert the GEMMs stream weights from HBM and the
  // int8 path's 64-token engine with its deeper weight ring is faster)
  const bool f16 = (2 * I) % 256 == 0 && H % 256 == 0 && R > int64_t(64) * E &&
                   (blk ? gemm_tc6_supported(probe) : gemm_tc4_supported(probe));
  if (f16) {
    uint16_t *A16 = reinterpret_cast<uint16_t *>(b.A);
    uint16_t *hq16 = reinterpret_cast<uint16_t *>(b.hq);
    // each token quantized once and written to its k rows (no int8 copy)
    WQ_TRY(launch_quant_scatter_f16(x, T, H, H, blk ? 128 : 0, b.pair_to_row, k, R, A16, b.sa,
                                    b.anorm, st));
    GemmArgs f1{nullptr, A16, b.anorm, b.sa, W13, sw13, b.offsets, nullptr, 0, E, R,
                int64_t(2) * I, H, scheme, acc, WQ_OUT_BF16, b.gu, b.gemm_ws, status};
    // (the block scheme's fused gate_up -> SiLU-and-mul -> re-quantization
    // entry computes the same codes; on the converter-bound block engine its
    // epilogue costs more than this separate memory-bound pass)
    WQ_TRY(launch_grouped_gemm(f1, st));
    WQ_TRY(launch_silu_mul_quant_f16(b.gu, R, I, blk ? 128 : 0, nullptr, 0, hq16, b.sh, b.hnorm,
                                     st));
    GemmArgs f2{nullptr, hq16, b.hnorm, b.sh, W2, sw2, b.offsets, nullptr, 0, E, R, H, I, scheme,
                acc, WQ_OUT_BF16, b.y, b.gemm_ws, status};
    WQ_TRY(launch_grouped_gemm(f2, st));
    return launch_combine(b.y, b.pair_to_row, b.w, T, k, H, out, st);
  }
  WQ_TRY(launch_quant_scatter_i8(x, T, H, H, blk ? 128 : 0, b.pair_to_row, k, R, b.A, b.sa, st));
  GemmArgs g1{b.A, nullptr, nullptr, b.sa, W13, sw13, b.offsets, nullptr, 0, E, R, int64_t(2) * I, H, scheme, acc,
              WQ_OUT_BF16, b.gu, b.gemm_ws, status};
  WQ_TRY(launch_grouped_gemm(g1, st));
  WQ_TRY(launch_silu_mul_quant(b.gu, R, I, blk ? 128 : 0, nullptr, 0, b.hq, b.sh, st));
  GemmArgs g2{b.hq, nullptr, nullptr, b.sh, W2, sw2, b.offsets, nullptr, 0, E, R, H, I, scheme, acc,
              WQ_OUT_BF16, b.y, b.gemm_ws, status};
  WQ_TRY(launch_grouped_gemm(g2, st));
  return launch_combine(b.y, b.pair_to_row, b.w, T, k, H, out, st);
}

}  // namespace

size_t wq_moe_forward_workspace_size(int T, int H, int I, int E, int k, int scheme) {
  if (check_forward_shape(T, H, I, E, k, scheme, WQ_ACC_I32) != WQ_OK) return 0;
  return carve_forward(nullptr, T, H, I, E, k, scheme, nullptr);
}

int wq_moe_forward(const uint16_t *x, const float *logits, const int8_t *W13, const float *sw13,
                   const int8_t *W2, const float *sw2, int T, int H, int I, int E, int k,
                   int scheme, int acc, uint16_t *out, void *ws, size_t ws_bytes,
                   int32_t *status, wq_stream_t stream) {
  WQ_TRY(check_forward_shape(T, H, I, E, k, scheme, acc));
  if (T == 0) return WQ_OK;
  if (!x || !logits || !W13 || !sw13 || !W2 || !sw2 || !out) return WQ_ERR_INVALID_ARG;
  if (!al16(x) || !al16(out) || !al16(W13) || !al16(W2)) return WQ_ERR_UNSUPPORTED;
  FwdBufs b;
  const size_t need = carve_forward(ws, T, H, I, E, k, scheme, &b);
  if (!ws || ws_bytes < need || !al16(ws)) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  return run_forward(x, logits, W13, sw13, W2, sw2, T, H, I, E, k, scheme, acc, out, b, status,
                     stream);
}

namespace {
// The device address of a host buffer that is mapped into the device's
// address space (pinned host memory), else nullptr.
const void *host_mapping(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}
}  // namespace

size_t wq_moe_forward_host_workspace_size(int T, int H, int I, int E, int k, int scheme) {
  const size_t inner = wq_moe_forward_workspace_size(T, H, I, E, k, scheme);
  if (inner == 0) return 0;
  return inner + rup(size_t(T) * H * 2) + rup(size_t(T) * E * 4) + rup(size_t(T) * H * 2);
}

int wq_moe_forward_host(const uint16_t *x_host, const float *logits_host, const int8_t *W13,
                        const float *sw13, const int8_t *W2, const float *sw2, int T, int H, int I,
                        int E, int k, int scheme, int acc, uint16_t *out_host, void *ws,
                        size_t ws_bytes, int32_t *status, wq_stream_t stream) {
  WQ_TRY(check_forward_shape(T, H, I, E, k, scheme, acc));
  if (T == 0) return WQ_OK;
  if (!x_host || !logits_host || !W13 || !sw13 || !W2 || !sw2 || !out_host)
    return WQ_ERR_INVALID_ARG;
  if (!al16(W13) || !al16(W2)) return WQ_ERR_UNSUPPORTED;
  if (!ws || !al16(ws) || ws_bytes < wq_moe_forward_host_workspace_size(T, H, I, E, k, scheme))
    return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  Carver c(ws);
  uint16_t *x = c.take<uint16_t>(size_t(T) * H);
  float *logits = c.take<float>(size_t(T) * E);
  uint16_t *out = c.take<uint16_t>(size_t(T) * H);
  FwdBufs b;
  carve_forward(c.base + c.used, T, H, I, E, k, scheme, &b);
  // Pinned host buffers are mapped into the device's address space: then the
  // quantization kernel reads x, the router reads the logits and the combine
  // writes the output across the CPU-GPU link themselves (each is the only
  // kernel touching that buffer), with no staging copies.
  const void *xm = host_mapping(x_host), *lm = host_mapping(logits_host),
             *om = host_mapping(out_host);
  if (xm && lm && om && al16(xm) && al16(om))
    return run_forward(static_cast<const uint16_t *>(xm), static_cast<const float *>(lm), W13, sw13,
                       W2, sw2, T, H, I, E, k, scheme, acc,
                       static_cast<uint16_t *>(const_cast<void *>(om)), b, status, stream);
  if (cudaMemcpyAsync(x, x_host, size_t(T) * H * 2, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return WQ_ERR_LAUNCH;
  if (cudaMemcpyAsync(logits, logits_host, size_t(T) * E * 4, cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return WQ_ERR_LAUNCH;
  WQ_TRY(run_forward(x, logits, W13, sw13, W2, sw2, T, H, I, E, k, scheme, acc, out, b, status,
                     stream));
  if (cudaMemcpyAsync(out_host, out, size_t(T) * H * 2, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return WQ_ERR_LAUNCH;
  return WQ_OK;
}

// ---------------------------------------------------------------------------
// Dense W8A8 linear ("Norm Linear")

namespace {

struct LinBufs {
  int32_t *offsets;
  void *q;  // int8 codes, or the same codes as fp16
  float *s;
  int32_t *norm;
  void *gws;
  size_t gws_bytes;
};

size_t carve_linear(void *ws, int64_t T, int64_t K, int scheme, LinBufs *b) {
  Carver c(ws);
  LinBufs t;
  const int64_t g = scheme == WQ_SCHEME_BLOCK ? K / 128 : 1;
  t.offsets = c.take<int32_t>(2);
  t.q = c.take<uint16_t>(size_t(T) * K);
  t.s = c.take<float>(size_t(T) * g);
  t.norm = c.take<int32_t>(size_t(T));
  t.gws_bytes = gemm_ws_bytes(T, 1, 0, false);
  t.gws = c.take<char>(t.gws_bytes);
  if (b) *b = t;
  return c.used;
}

__global__ void linear_offsets_kernel(int32_t *offsets, int32_t T) {
  offsets[0] = 0;
  offsets[1] = T;
}

int check_linear_shape(int64_t T, int64_t K, int64_t N, int scheme, int acc) {
  if (T < 0 || K <= 0 || N <= 0) return WQ_ERR_INVALID_ARG;
  if (scheme != WQ_SCHEME_CHANNEL && scheme != WQ_SCHEME_BLOCK) return WQ_ERR_INVALID_ARG;
  if (acc != WQ_ACC_I32 && acc != WQ_ACC_F32) return WQ_ERR_INVALID_ARG;
  if (K % 128 || N % 128 || K > 65536) return WQ_ERR_UNSUPPORTED;
  if (T >= (int64_t(1) << 31) / 2) return WQ_ERR_UNSUPPORTED;
  return WQ_OK;
}

}  // namespace

size_t wq_linear_w8a8_workspace_size(int64_t T, int64_t K, int64_t N, int scheme) {
  if (check_linear_shape(T, K, N, scheme, WQ_ACC_I32) != WQ_OK) return 0;
  return carve_linear(nullptr, T, K, scheme, nullptr);
}

int wq_linear_w8a8(const uint16_t *x, int64_t T, int64_t K, int64_t ldx, const int8_t *W,
                   const float *sw, int64_t N, int scheme, int acc, uint16_t *out, void *ws,
                   size_t ws_bytes, int32_t *status, wq_stream_t stream) {
  WQ_TRY(check_linear_shape(T, K, N, scheme, acc));
  if (ldx < K) return WQ_ERR_INVALID_ARG;
  if (T == 0) return WQ_OK;
  if (!x || !W || !sw || !out) return WQ_ERR_INVALID_ARG;
  if (ldx % 8 || !al16(x) || !al16(W) || !al16(out)) return WQ_ERR_UNSUPPORTED;
  LinBufs b;
  const size_t need = carve_linear(ws, T, K, scheme, &b);
  if (!ws || !al16(ws) || ws_bytes < need) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  const bool blk = scheme == WQ_SCHEME_BLOCK;
  linear_offsets_kernel<<<1, 1, 0, stream>>>(b.offsets, int32_t(T));
  WQ_TRY(launched(1));
  // many rows and N a multiple of 256: fp16 codes for the CTA-pair engines
  // (the quantizer writes them directly, with row norms for the channel-wise
  // exactness check); otherwise int8 codes (few rows: the small-token engine)
  GemmArgs probe{nullptr, static_cast<const uint16_t *>(b.q), b.norm, b.s, W, sw, b.offsets,
                 nullptr, 0, 1, T, N, K, scheme, acc, WQ_OUT_BF16, out, b.gws, status};
  const bool f16 = N % 256 == 0 && T > 64 &&
                   (blk ? gemm_tc6_supported(probe) : gemm_tc4_supported(probe));
  if (f16) {
    WQ_TRY(launch_quant_rows_f16(x, T, K, ldx, blk ? 128 : 0, static_cast<uint16_t *>(b.q), b.s,
                                 b.norm, stream));
    return launch_grouped_gemm(probe, stream);
  }
  WQ_TRY(launch_quant_rows(x, T, K, ldx, blk ? 128 : 0, static_cast<int8_t *>(b.q), b.s, stream));
  GemmArgs g{static_cast<const int8_t *>(b.q), nullptr, nullptr, b.s, W, sw, b.offsets, nullptr, 0,
             1, T, N, K, scheme, acc, WQ_OUT_BF16, out, b.gws, status};
  return launch_grouped_gemm(g, stream);
}

// ---------------------------------------------------------------------------
// Masked layout

namespace {

// The fp16 token form of the int8-code engine serves the masked layer when
// the engine takes 256-token tiles (more than 64 rows per expert buffer; the
// same rule as gemm_tc2_tile_rows) on the channel scheme, K within its range.
bool masked_tok16(int scheme, int Mmax, int H, int I) {
  return scheme == WQ_SCHEME_CHANNEL && Mmax > 64 && H <= 65536 && I <= 65536;
}

size_t carve_masked(void *ws, int E, int Mmax, int H, int I, int scheme, uint16_t **gu,
                    int8_t **hq, float **sh, void **gws, size_t *gws_bytes,
                    int32_t **norm = nullptr, uint16_t **t16 = nullptr) {
  Carver c(ws);
  const int64_t R = int64_t(E) * Mmax;
  const int64_t g2 = scheme == WQ_SCHEME_BLOCK ? I / 128 : 1;
  uint16_t *a = c.take<uint16_t>(size_t(R) * 2 * I);
  int8_t *b = c.take<int8_t>(size_t(R) * I);
  float *d = c.take<float>(size_t(R) * g2);
  const size_t gb = gemm_ws_bytes(R, E, Mmax, true);
  void *g = c.take<char>(gb);
  // fp16 token form: a GEMM input's valid rows as fp16 codes (x for GEMM1,
  // then h for GEMM2, in the same buffer) and their squared norms
  const bool f16t = masked_tok16(scheme, Mmax, H, I);
  int32_t *n2 = f16t ? c.take<int32_t>(size_t(R)) : nullptr;
  uint16_t *t = f16t ? c.take<uint16_t>(size_t(R) * size_t(H > I ? H : I)) : nullptr;
  if (gu) { *gu = a; *hq = b; *sh = d; *gws = g; *gws_bytes = gb; }
  if (norm) *norm = n2;
  if (t16) *t16 = t;
  return c.used;
}

}  // namespace

namespace wq {
// The masked layer on W8A8 weights, or (w4) on int4 weights packed two per
// byte: GEMM1 -> SiLU-mul + re-quantization -> GEMM2 on the valid rows.
int forward_masked(const int8_t *a, const float *sa, const int32_t *masked_m, int E, int Mmax,
                   const int8_t *W13, const float *sw13, const int8_t *W2, const float *sw2, int H,
                   int I, int scheme, int acc, bool w4, uint16_t *y, void *ws, size_t ws_bytes,
                   int32_t *status, cudaStream_t stream) {
  if (E < 1 || E > 4096 || Mmax < 0 || H <= 0 || I <= 0) return WQ_ERR_INVALID_ARG;
  if (scheme != WQ_SCHEME_CHANNEL && scheme != WQ_SCHEME_BLOCK) return WQ_ERR_INVALID_ARG;
  if (acc != WQ_ACC_I32 && acc != WQ_ACC_F32) return WQ_ERR_INVALID_ARG;
  if (H % 128 || I % 128) return WQ_ERR_UNSUPPORTED;
  if (Mmax == 0) return WQ_OK;
  if (!a || !sa || !masked_m || !W13 || !sw13 || !W2 || !sw2 || !y) return WQ_ERR_INVALID_ARG;
  if (!al16(a) || !al16(y) || !al16(W13) || !al16(W2)) return WQ_ERR_UNSUPPORTED;
  if (int64_t(E) * Mmax >= (int64_t(1) << 31) / 2) return WQ_ERR_UNSUPPORTED;
  uint16_t *gu;
  int8_t *hq;
  float *sh;
  void *gws;
  size_t gwsb;
  int32_t *norm;
  uint16_t *t16;
  const size_t need =
      carve_masked(ws, E, Mmax, H, I, scheme, &gu, &hq, &sh, &gws, &gwsb, &norm, &t16);
  if (!ws || !al16(ws) || ws_bytes < need) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  const int64_t R = int64_t(E) * Mmax;
  // Channel scheme, 256-token tiles: before each GEMM one pass writes the
  // valid rows' codes as fp16 values and their squared norms, so that the
  // int8-code engine loads fp16 token tiles instead of widening each again for
  // every weight block, and (int8 weights) need not sum their norms for its
  // exactness check.  The small-token engine beside it reads the int8 codes.
  const bool f16t = masked_tok16(scheme, Mmax, H, I);
  if (f16t) WQ_TRY(launch_row_norm_i8(a, R, H, masked_m, Mmax, norm, stream, t16));
  GemmArgs g1{a, nullptr, nullptr, sa, W13, sw13, nullptr, masked_m, Mmax, E, R, int64_t(2) * I,
              H, scheme, acc, WQ_OUT_BF16, gu, gws, status};
  g1.w4 = w4 ? 1 : 0;
  if (f16t) {
    g1.tok16 = t16;
    g1.a_norm2 = w4 ? nullptr : norm;
  }
  WQ_TRY(launch_grouped_gemm(g1, stream));
  // GEMM1 has finished with the fp16 rows and norms (same stream): h's
  // replace them, written by the SiLU pass itself (rows of at most 2048
  // outputs), else by the widening pass after it
  int rc = WQ_ERR_UNSUPPORTED;
  if (f16t) rc = launch_silu_mul_quant_dual(gu, R, I, masked_m, Mmax, hq, t16, sh, norm, stream, w4);
  if (rc != WQ_OK && rc != WQ_ERR_UNSUPPORTED) return rc;
  if (rc != WQ_OK) {
    WQ_TRY(launch_silu_mul_quant(gu, R, I, scheme == WQ_SCHEME_BLOCK ? 128 : 0, masked_m, Mmax, hq,
                                 sh, stream));
    if (f16t) WQ_TRY(launch_row_norm_i8(hq, R, I, masked_m, Mmax, norm, stream, t16));
  }
  GemmArgs g2{hq, nullptr, nullptr, sh, W2, sw2, nullptr, masked_m, Mmax, E, R,
              H, I, scheme, acc, WQ_OUT_BF16, y, gws, status};
  g2.w4 = w4 ? 1 : 0;
  if (f16t) {
    g2.tok16 = t16;
    g2.a_norm2 = w4 ? nullptr : norm;
  }
  return launch_grouped_gemm(g2, stream);
}
}  // namespace wq


size_t wq_moe_forward_masked_workspace_size(int E, int Mmax, int H, int I, int scheme) {
  if (E < 1 || Mmax < 0 || H <= 0 || I <= 0) return 0;
  return carve_masked(nullptr, E, Mmax, H, I, scheme, nullptr, nullptr, nullptr, nullptr, nullptr);
}

int wq_moe_forward_masked(const int8_t *a, const float *sa, const int32_t *masked_m, int E,
                          int Mmax, const int8_t *W13, const float *sw13, const int8_t *W2,
                          const float *sw2, int H, int I, int scheme, int acc, uint16_t *y,
                          void *ws, size_t ws_bytes, int32_t *status, wq_stream_t stream) {
  return wq::forward_masked(a, sa, masked_m, E, Mmax, W13, sw13, W2, sw2, H, I, scheme, acc, false,
                            y, ws, ws_bytes, status, stream);
}

int wq_quantize_weight_int4(const uint16_t *w, int64_t N, int64_t K, uint8_t *q4, float *s,
                            wq_stream_t stream) {
  if (N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return WQ_OK;
  if (!w || !q4 || !s) return WQ_ERR_INVALID_ARG;
  if (K % 8 || !al16(w) || (reinterpret_cast<uintptr_t>(q4) & 3u)) return WQ_ERR_UNSUPPORTED;
  if (N >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  WQ_TRY(check_device());
  return launch_quant_weight_int4(w, N, K, q4, s, stream);
}

int wq_grouped_gemm_w4a8_masked(const int8_t *A, const float *sa, const int32_t *masked_m, int E,
                                int Mmax, const uint8_t *W4, const float *s4, int64_t N,
                                int64_t K, int out_type, void *out, void *ws, size_t ws_bytes,
                                int32_t *status, wq_stream_t stream) {
  if (Mmax < 0 || E > 4096) return WQ_ERR_INVALID_ARG;
  if (Mmax == 0) return WQ_OK;
  WQ_TRY(check_gemm_common(reinterpret_cast<const int8_t *>(W4), s4, E, N, K, WQ_SCHEME_CHANNEL,
                           WQ_ACC_I32, out_type, out));
  if (!A || !sa || !masked_m) return WQ_ERR_INVALID_ARG;
  if (!al16(A) || K > 16384 || int64_t(E) * Mmax >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  const int64_t R = int64_t(E) * Mmax;
  if (ws_bytes < gemm_ws_bytes(R, E, Mmax, true) || !ws) return WQ_ERR_WORKSPACE;
  WQ_TRY(check_device());
  GemmArgs g{A, nullptr, nullptr, sa, reinterpret_cast<const int8_t *>(W4), s4, nullptr, masked_m,
             Mmax, E, R, N, K, WQ_SCHEME_CHANNEL, WQ_ACC_I32, out_type, out, ws, status};
  g.w4 = 1;
  return launch_grouped_gemm(g, stream);
}

size_t wq_moe_forward_masked_w4a8_workspace_size(int E, int Mmax, int H, int I) {
  return wq_moe_forward_masked_workspace_size(E, Mmax, H, I, WQ_SCHEME_CHANNEL);
}

int wq_moe_forward_masked_w4a8(const int8_t *a, const float *sa, const int32_t *masked_m, int E,
                               int Mmax, const uint8_t *W13, const float *s13, const uint8_t *W2,
                               const float *s2, int H, int I, uint16_t *y, void *ws,
                               size_t ws_bytes, int32_t *status, wq_stream_t stream) {
  if (H > 16384 || I > 16384) return WQ_ERR_UNSUPPORTED;
  return wq::forward_masked(a, sa, masked_m, E, Mmax, reinterpret_cast<const int8_t *>(W13), s13,
                            reinterpret_cast<const int8_t *>(W2), s2, H, I, WQ_SCHEME_CHANNEL,
                            WQ_ACC_I32, true, y, ws, ws_bytes, status, stream);
}

}  // extern "C"
