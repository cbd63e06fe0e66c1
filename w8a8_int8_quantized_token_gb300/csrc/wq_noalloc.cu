// Grouped W8A8 GEMM for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at run time: a plug-in running inside
// a host framework that owns the device's whole memory pool and gives its
// plug-ins no allocator, or a latency-bound serving loop where cudaMalloc's
// implicit device synchronisation (and its possible failure) is not
// acceptable once the loop has started.  For them this file keeps the grouped
// GEMM's scratch (tile lists, tile counts, the exact-recompute flag) in a
// static device array instead of a caller workspace.
//
// The array is a module global: every GPU that loads libwq.so holds
// WQ_NOALLOC_SCRATCH_BYTES of it until the process exits.  Its device address
// is looked up once per device, on the first call made with that device
// current, and cached in an atomic slot per device (host threads that make
// their first calls at the same time each look it up and store the same
// value).  All calls on a device share the one array and it keeps the last
// call's contents: each call rewrites the tile lists and counts and zeroes
// the recompute flag before its kernels read them, and calls whose kernels
// overlap on the GPU (different streams or threads) race on it.
#include <atomic>

#include "wq_common.cuh"

namespace wq {
int check_grouped_gemm_args(const int8_t *A, const float *sa, const int8_t *W, const float *sw,
                            const int32_t *offsets, int E, int64_t R, int64_t N, int64_t K,
                            int scheme, int acc, int out_type, const void *out);
}

namespace {

__device__ __align__(256) unsigned char g_gemm_scratch[WQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];  // device address of g_gemm_scratch, per device

// Device address of the scratch array on the current device (looked up on
// the first call for that device).
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ_ERR_DEVICE;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return WQ_ERR_LAUNCH;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return WQ_OK;
}

}  // namespace

extern "C" int wq_grouped_gemm_w8a8_noalloc(const int8_t *A, const float *sa, const int8_t *W,
                                            const float *sw, const int32_t *offsets, int E,
                                            int64_t R, int64_t N, int64_t K, int scheme, int acc,
                                            int out_type, void *out, int32_t *status,
                                            wq_stream_t stream) {
  // the workspace entry point's argument checks first, so both reject a bad
  // call with the same code; then the scratch limit
  const int arg = wq::check_grouped_gemm_args(A, sa, W, sw, offsets, E, R, N, K, scheme, acc,
                                              out_type, out);
  if (arg != WQ_OK) return arg;
  if (R == 0) return WQ_OK;
  const size_t need = wq_grouped_gemm_workspace_size(R, E);
  if (need == 0 || need > size_t(WQ_NOALLOC_SCRATCH_BYTES)) return WQ_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != WQ_OK) return rc;
  return wq_grouped_gemm_w8a8(A, sa, W, sw, offsets, E, R, N, K, scheme, acc, out_type, out,
                              scratch, size_t(WQ_NOALLOC_SCRATCH_BYTES), status, stream);
}
