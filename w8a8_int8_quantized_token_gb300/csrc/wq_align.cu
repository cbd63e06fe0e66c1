// Expert alignment: counts, offsets (cumulative with a leading zero, as the
// cutlass_moe_fp8 review for DeepEP asks), and the stable permutation of the
// (token, slot) pairs by expert.  Deterministic: a counting sort whose ranks
// come from ordered scans and warp match masks, never from atomic order.
//
// Also the grouped GEMM's tile list: per expert segment, ceil(rows/BM)
// tiles, longest first.
#include "wq_common.cuh"

namespace wq {

constexpr int kAlignChunk = 256;  // pairs per chunk

static inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

size_t align_ws_bytes(int T, int k, int E) {
  const int64_t P = int64_t(T) * k;
  const int64_t chunks = (P + kAlignChunk - 1) / kAlignChunk;
  return size_t(align_up(chunks * E * 4, 256));
}

// 1) per-chunk expert histogram (shared-memory counts; order-free)
__global__ void __launch_bounds__(kAlignChunk) align_hist_kernel(const int32_t *__restrict__ ids,
                                                                 int64_t P, int E,
                                                                 int32_t *__restrict__ hist,
                                                                 int32_t *status) {
  extern __shared__ int32_t cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t p = int64_t(blockIdx.x) * kAlignChunk + threadIdx.x;
  if (p < P) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else set_status(status, WQ_ERR_INDEX);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[int64_t(blockIdx.x) * E + e] = cnt[e];
}

// 2) one CTA. Warps own contiguous chunk ranges, lanes own experts, so
//    every access to hist is a coalesced row piece. Per tile of 128
//    experts: the warps' sums, their exclusive scan down the 32 warps in
//    shared memory (-> counts), then each warp rewrites its rows with the
//    running prefix. Then the padded counts are scanned over experts
//    (-> offsets) and added to every row: hist[c][e] becomes the first row
//    of chunk c's pairs of expert e.
__global__ void __launch_bounds__(1024) align_scan_kernel(int32_t *__restrict__ hist, int chunks,
                                                          int E, int pad_m,
                                                          int32_t *__restrict__ counts,
                                                          int32_t *__restrict__ offsets) {
  constexpr int TE = 128, J = TE / 32;
  __shared__ int32_t part[32][TE];
  __shared__ int32_t scan[1024];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_warp = (chunks + 31) / 32;
  const int c0 = min(chunks, warp * per_warp), c1 = min(chunks, c0 + per_warp);
  for (int eb = 0; eb < E; eb += TE) {
    int acc[J];
#pragma unroll
    for (int j = 0; j < J; ++j) acc[j] = 0;
    for (int c = c0; c < c1; ++c) {
      const int32_t *row = hist + int64_t(c) * E + eb;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (eb + lane + 32 * j < E) acc[j] += row[lane + 32 * j];
    }
#pragma unroll
    for (int j = 0; j < J; ++j) part[warp][lane + 32 * j] = acc[j];
    __syncthreads();
    if (threadIdx.x < TE) {
      int run = 0;
      for (int w = 0; w < 32; ++w) {
        const int v = part[w][threadIdx.x];
        part[w][threadIdx.x] = run;
        run += v;
      }
      if (eb + int(threadIdx.x) < E) counts[eb + threadIdx.x] = run;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < J; ++j) acc[j] = part[warp][lane + 32 * j];
    for (int c = c0; c < c1; ++c) {
      int32_t *row = hist + int64_t(c) * E + eb;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (eb + lane + 32 * j < E) {
          const int v = row[lane + 32 * j];
          row[lane + 32 * j] = acc[j];
          acc[j] += v;
        }
    }
    __syncthreads();  // part is reused by the next tile
  }
  // padded counts of this thread's experts, block-wide exclusive scan
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per;
  int local = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) local += (counts[e] + pad_m - 1) / pad_m * pad_m;
  scan[threadIdx.x] = local;
  __syncthreads();
  for (int o = 1; o < int(blockDim.x); o <<= 1) {  // inclusive Hillis-Steele scan
    const int v = threadIdx.x >= unsigned(o) ? scan[threadIdx.x - o] : 0;
    __syncthreads();
    scan[threadIdx.x] += v;
    __syncthreads();
  }
  int base = scan[threadIdx.x] - local;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    offsets[e] = base;
    base += (counts[e] + pad_m - 1) / pad_m * pad_m;
  }
  if (threadIdx.x == blockDim.x - 1) offsets[E] = scan[threadIdx.x];
  __syncthreads();
  for (int c = c0; c < c1; ++c)
    for (int e = lane; e < E; e += 32) hist[int64_t(c) * E + e] += offsets[e];
}

// 3) one warp per chunk walks its pairs in order, 32 at a time; a pair's row
//    is its chunk base + the pairs of the same expert already placed + its
//    rank among equal lanes below it (match mask).
__global__ void __launch_bounds__(32) align_scatter_kernel(const int32_t *__restrict__ ids,
                                                           int64_t P, int E,
                                                           const int32_t *__restrict__ hist,
                                                           int32_t *__restrict__ sorted_pair,
                                                           int32_t *__restrict__ pair_to_row) {
  extern __shared__ int32_t cur[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cur[e] = hist[int64_t(blockIdx.x) * E + e];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  for (int step = 0; step < kAlignChunk / 32; ++step) {
    const int64_t p = int64_t(blockIdx.x) * kAlignChunk + step * 32 + lane;
    int e = -1;
    if (p < P) {
      e = ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int row = cur[e] + __popc(same & lt);
      sorted_pair[row] = int32_t(p);
      pair_to_row[p] = row;
    } else if (p < P) {
      pair_to_row[p] = -1;
    }
    __syncwarp();
    if (e >= 0 && (same & lt) == 0) cur[e] += __popc(same);  // group leader advances
    __syncwarp();
  }
}

int launch_align(const int32_t *ids, int T, int k, int E, int pad_m, int32_t *counts,
                 int32_t *offsets, int32_t *sorted_pair, int32_t *pair_to_row, void *ws,
                 int32_t *status, cudaStream_t st) {
  const int64_t P = int64_t(T) * k;
  const int64_t cap = P + int64_t(E) * (pad_m - 1);
  const int chunks = int((P + kAlignChunk - 1) / kAlignChunk);
  int32_t *hist = static_cast<int32_t *>(ws);
  if (cap > 0 && cudaMemsetAsync(sorted_pair, 0xff, size_t(cap) * 4, st) != cudaSuccess)
    return WQ_ERR_LAUNCH;
  const size_t smem = size_t(E) * 4;
  if (chunks > 0) {
    align_hist_kernel<<<chunks, kAlignChunk, smem, st>>>(ids, P, E, hist, status);
  }
  align_scan_kernel<<<1, 1024, 0, st>>>(hist, chunks, E, pad_m, counts, offsets);
  if (chunks > 0) {
    align_scatter_kernel<<<chunks, 32, smem, st>>>(ids, P, E, hist, sorted_pair, pair_to_row);
  }
  return launched(chunks > 0 ? 3 : 1);
}

// ---------------------------------------------------------------------------
// Tile list of the grouped GEMM.  Segment e: rows [offsets[e], offsets[e+1])
// (contiguous layout) or [e*Mmax, e*Mmax + clamp(masked_m[e], 0, Mmax))
// (masked layout).  A segment of len rows gives floor(len / BM) full tiles
// and, for a remainder of rem rows, one more tile: in the small list when
// 0 < rem <= small_max (a small list is given), else in the main list.
// The main list is ordered longest first, so that persistent engines that
// hand items out in order finish with their shortest ones: first the
// experts with full tiles (BM rows), in expert order, each followed at once
// by its own partial tile (the tiles of one expert stay adjacent, so the
// engines read that expert's weights from DRAM once and from L2 for the
// other tiles), then the partial tiles of the other experts by row count,
// descending (equal counts in arbitrary order: the tiles write disjoint
// rows, so the order changes no result).  ntiles[0] / nsmall[0] = numbers
// written.
constexpr int kMaxTileRows = 384;

// Inclusive prefix sums of a and b over the 1024 threads of the block (warp
// shuffles, then one warp over the 32 warp totals); ta / tb: the totals.
__device__ __forceinline__ void block_scan2(int &a, int &b, int &ta, int &tb) {
  __shared__ int wa[32], wb[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) {
      a += ya;
      b += yb;
    }
  }
  if (lane == 31) {
    wa[warp] = a;
    wb[warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    int x = wa[lane], y = wb[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(0xffffffffu, x, o), yy = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) {
        x += xa;
        y += yy;
      }
    }
    wa[lane] = x;
    wb[lane] = y;
  }
  __syncthreads();
  if (warp > 0) {
    a += wa[warp - 1];
    b += wb[warp - 1];
  }
  ta = wa[31];
  tb = wb[31];
  __syncthreads();  // wa / wb free for the next call
}

__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t *__restrict__ offsets,
                                                           const int32_t *__restrict__ masked_m,
                                                           int Mmax, int E, int BM, int64_t R,
                                                           Tile *__restrict__ tiles,
                                                           int32_t *__restrict__ ntiles,
                                                           int32_t *__restrict__ zero_word,
                                                           int small_max,
                                                           Tile *__restrict__ small,
                                                           int32_t *__restrict__ nsmall,
                                                           const int32_t *__restrict__ gate) {
  // the list of a gated exact recompute: not needed unless its flag is set
  if (gate != nullptr && *gate == 0) return;
  __shared__ int32_t hist[kMaxTileRows + 1];  // partial main tiles by row count, then cursors
  if (zero_word != nullptr && threadIdx.x < 2) zero_word[threadIdx.x] = 0;  // flag, item counter
  for (int i = threadIdx.x; i <= kMaxTileRows; i += blockDim.x) hist[i] = 0;
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per;
  const bool split = small != nullptr && small_max > 0;
  auto seg = [&](int e, int &r0, int &len) {
    if (masked_m) {
      int m = masked_m[e];
      m = m < 0 ? 0 : (m > Mmax ? Mmax : m);
      r0 = e * Mmax;
      len = m;
    } else {
      // clamp to [0, R): the tile list can never outgrow ceil(R/BM) + E
      int64_t a = offsets[e], b = offsets[e + 1];
      a = a < 0 ? 0 : (a > R ? R : a);
      b = b < a ? a : (b > R ? R : b);
      r0 = int(a);
      len = int(b - a);
    }
  };
  // full tiles, the remainder, and whether it goes to the small list
  auto plan = [&](int len, int &nfull, int &rem, bool &to_small) {
    nfull = len / BM;
    rem = len - nfull * BM;
    to_small = split && rem > 0 && rem <= small_max;
  };
  __syncthreads();
  int local = 0, local_s = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    int r0, len, nfull, rem;
    bool ts;
    seg(e, r0, len);
    plan(len, nfull, rem, ts);
    const bool part_main = rem > 0 && !ts;
    local += nfull + (nfull > 0 && part_main ? 1 : 0);  // beside its full tiles
    if (nfull == 0 && part_main) atomicAdd(&hist[rem], 1);
    local_s += ts ? 1 : 0;
  }
  int incl = local, incl_s = local_s, nfull_total, nsmall_total;
  block_scan2(incl, incl_s, nfull_total, nsmall_total);  // (the histogram is complete too)
  // first position of the partial tiles of each row count, longest first:
  // thread i takes row count BM - 1 - i (BM <= 384 < 1024)
  const int rc = BM - 1 - int(threadIdx.x);
  int c = rc >= 1 ? hist[rc] : 0, unused = 0, npart, unused_t;
  const int c0 = c;
  block_scan2(c, unused, npart, unused_t);
  if (rc >= 1) hist[rc] = nfull_total + c - c0;
  if (threadIdx.x == 0) {
    ntiles[0] = nfull_total + npart;
    if (split) nsmall[0] = nsmall_total;
  }
  __syncthreads();
  int t = incl - local, ts_i = incl_s - local_s;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    int r0, len, nfull, rem;
    bool ts;
    seg(e, r0, len);
    plan(len, nfull, rem, ts);
    for (int m = 0; m < nfull; ++m) {
      Tile tl;
      tl.expert = e;
      tl.row0 = r0 + m * BM;
      tl.rows = BM;
      tl.pad = 0;
      tiles[t++] = tl;
    }
    if (rem > 0) {
      Tile tl;
      tl.expert = e;
      tl.row0 = r0 + nfull * BM;
      tl.rows = rem;
      tl.pad = 0;
      if (ts) small[ts_i++] = tl;
      else if (nfull > 0) tiles[t++] = tl;
      else tiles[atomicAdd(&hist[rem], 1)] = tl;
    }
  }
}

int launch_build_tiles(const int32_t *offsets, const int32_t *masked_m, int Mmax, int E, int BM,
                       int64_t R, Tile *tiles, int32_t *ntiles, int32_t *zero_word,
                       cudaStream_t st, int small_max, Tile *small, int32_t *nsmall,
                       const int32_t *gate) {
  if (BM < 1 || BM > kMaxTileRows) return WQ_ERR_UNSUPPORTED;
  build_tiles_kernel<<<1, 1024, 0, st>>>(offsets, masked_m, Mmax, E, BM, R, tiles, ntiles,
                                         zero_word, small_max, small, nsmall, gate);
  return launched(1);
}

}  // namespace wq
