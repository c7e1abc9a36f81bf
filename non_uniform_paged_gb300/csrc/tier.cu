// Tiered KV placement: promoted-page fetch with in-place block reuse.
//
// Source: "FlexiCache: Leveraging Temporal Stability of Attention Heads for
// Efficient KV Cache Management (MLSys 2026)" (paper-review page), "Core
// method / Tiered KV placement" (a stable head keeps only its top-K pages on
// the GPU, the rest in host memory; at a rerank only the newly promoted pages
// move host -> GPU), "System engineering / Block Allocator" (physical blocks
// are reclaimed and reassigned in place at rerank time) and "KV transfer"
// (a custom kernel reads pinned host KV directly through unified addressing).
//
// One CTA per re-ranked (request, KV head) row.  A stable row owns K GPU blocks
// (slot_block[row][k]); slot_page[row][k] is the page a block holds (-1: none).
// With the new ascending selection sel[row][0..K): a block whose page left the
// selection is freed; the pages that entered it take the freed blocks, the
// lowest promoted page the lowest freed slot; each promoted page is copied from
// the pinned host copy (read through its device-mapped address over
// NVLink-C2C / PCIe) into its block, and kept pages are not touched.  The
// decode list pt_ids[row][k] is then the block holding sel[row][k].  An
// unstable row holds all its pages in GPU memory: its list is dense_base[row]
// + sel[row][k].
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

namespace {

using namespace tgk;

constexpr int kMaxTierPages = 16384;  // pages per row the shared-memory bitmaps cover
constexpr int kMaxTierK = 1024;

struct TierArgs {
  const int32_t *rows;        // [n_rows] row numbers b*H + h to process
  int n_rows;
  const uint8_t *unstable;    // [H] of this layer
  int H, n_pages, K;
  const int32_t *sel;         // [total][K] ascending
  int32_t *slot_page;         // [total][K]
  const int32_t *slot_block;  // [total][K]
  const int64_t *dense_base;  // [total] first pool page of an unstable row's dense region
  const uint4 *host_kv;       // [total][n_pages][page_vec] pinned host, device-mapped
  uint4 *pool;                // [pool_pages][page_vec]
  int64_t pool_pages;
  int page_vec;               // 16-byte vectors per page
  int64_t total_rows;
  int32_t *pt_ids;            // [total][K] decode lists (output)
  int64_t *promoted;          // [1] pages copied (optional, accumulated)
  int32_t *status;
  int slices;                 // copy units per row (kCopy)
};

// What a launch of the kernel does with each listed row
constexpr int kWhole = 0;   // lists, copy, new block table and decode list
constexpr int kCopy = 1;    // lists and 1/slices of the copy (the row's state is not changed)
constexpr int kCommit = 2;  // lists from the old block table, then the new table and decode list

// NT threads per CTA: 256 for a copy on the decode's stream, 64 (at most 64 registers a
// thread: 4096 registers and 16 KB of shared memory a CTA) for a background copy whose CTAs
// stay resident beside a decode or score CTA on the same SM
template <int NT, int MODE>
__global__ void __launch_bounds__(NT, 65536 / (NT * 64)) tier_promote_kernel(const TierArgs a) {
  constexpr int kThreads = NT;
  constexpr int U = NT == 64 ? 5 : 4;  // host reads in flight per thread
  __shared__ uint32_t in_sel[kMaxTierPages / 32];   // page is in the new selection
  __shared__ uint32_t resident[kMaxTierPages / 32]; // page is held by one of the row's blocks
  __shared__ int32_t freed[kMaxTierK];              // slots to reuse, ascending
  __shared__ int32_t incoming[kMaxTierK];           // promoted pages, ascending
  __shared__ int32_t blk_of[kMaxTierK];             // block holding sel[k]
  __shared__ int n_freed, n_in;
  const int tid = threadIdx.x;
  const int words = (a.n_pages + 31) / 32;
  const int units = MODE == kCopy ? a.n_rows * a.slices : a.n_rows;
  for (int i = blockIdx.x; i < units; i += gridDim.x) {
    const int ri = MODE == kCopy ? i / a.slices : i, slice = MODE == kCopy ? i % a.slices : 0;
    const int64_t row = a.rows[ri];
    if (row < 0 || row >= a.total_rows) {
      if (tid == 0 && slice == 0) report(a.status, TG_STATUS_BAD_INPUT);
      continue;  // uniform over the CTA
    }
    const int32_t *srow = a.sel + row * a.K;
    int32_t *prow = a.pt_ids + row * a.K;
    if (a.unstable[row % a.H]) {  // all pages on the GPU
      if (MODE != kCopy)
        for (int k = tid; k < a.K; k += kThreads) prow[k] = (int32_t)(a.dense_base[row] + srow[k]);
      continue;
    }
    int32_t *spage = a.slot_page + row * a.K;
    const int32_t *sblock = a.slot_block + row * a.K;
    for (int w = tid; w < words; w += kThreads) in_sel[w] = resident[w] = 0u;
    if (tid == 0) n_freed = n_in = 0;
    __syncthreads();
    for (int k = tid; k < a.K; k += kThreads) {
      const int p = srow[k];
      if (p >= 0 && p < a.n_pages) atomicOr(&in_sel[p >> 5], 1u << (p & 31));
      const int r = spage[k];
      if (r >= 0 && r < a.n_pages) atomicOr(&resident[r >> 5], 1u << (r & 31));
    }
    __syncthreads();
    // freed slots (page gone from the selection, or empty) and incoming pages, each listed in
    // ascending order by a CTA-wide prefix count
    for (int base = 0; base < a.K; base += kThreads) {
      const int k = base + tid;
      bool f = false, in = false;
      int p = -1;
      if (k < a.K) {
        const int r = spage[k];
        f = r < 0 || r >= a.n_pages || !((in_sel[r >> 5] >> (r & 31)) & 1u);
        p = srow[k];
        in = p >= 0 && p < a.n_pages && !((resident[p >> 5] >> (p & 31)) & 1u);
      }
      const int nf = __syncthreads_count(f), ni = __syncthreads_count(in);
      // rank within this chunk: ballots per warp, warp totals through shared memory
      __shared__ int wf[kThreads / 32], wi[kThreads / 32];
      const int lane = tid & 31, warp = tid >> 5;
      const uint32_t bf = __ballot_sync(0xffffffffu, f), bi = __ballot_sync(0xffffffffu, in);
      if (lane == 0) {
        wf[warp] = __popc(bf);
        wi[warp] = __popc(bi);
      }
      __syncthreads();
      int of = 0, oi = 0;
      for (int w = 0; w < warp; ++w) {
        of += wf[w];
        oi += wi[w];
      }
      const uint32_t lt = (1u << lane) - 1u;
      if (f) freed[n_freed + of + __popc(bf & lt)] = k;
      if (in) incoming[n_in + oi + __popc(bi & lt)] = p;
      __syncthreads();
      if (tid == 0) {
        n_freed += nf;
        n_in += ni;
      }
      __syncthreads();
    }
    const int moves = min(n_freed, n_in);  // equal for a valid selection of K distinct pages
    if (n_freed != n_in && tid == 0 && MODE != kCopy) report(a.status, TG_STATUS_BAD_INPUT);
    // copy every promoted page into the block of its freed slot: the CTA's threads stride over
    // the (page, 16-byte vector) pairs (all of them, or this slice's share), U independent host
    // reads in flight per thread
    const int64_t all = MODE == kCommit ? 0 : (int64_t)moves * a.page_vec;
    const int64_t lo = MODE == kCopy ? all * slice / a.slices : 0;
    const int64_t total = MODE == kCopy ? all * (slice + 1) / a.slices : all;
    auto vec_src = [&](int64_t e, uint4 *&dst) -> const uint4 * {
      const int m = (int)(e / a.page_vec), v = (int)(e % a.page_vec);
      const int64_t blk = sblock[freed[m]];
      if (blk < 0 || blk >= a.pool_pages) {
        dst = nullptr;
        return nullptr;
      }
      dst = a.pool + blk * (int64_t)a.page_vec + v;
      return a.host_kv + (row * a.n_pages + incoming[m]) * (int64_t)a.page_vec + v;
    };
    bool bad_block = false;
    for (int64_t e0 = lo + tid; e0 < total; e0 += U * kThreads) {
      uint4 val[U];
      uint4 *dst[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = e0 + (int64_t)u * kThreads;
        dst[u] = nullptr;
        if (e < total) {
          const uint4 *src = vec_src(e, dst[u]);
          if (src) val[u] = __ldcv(src);
          else bad_block = true;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (dst[u]) *dst[u] = val[u];
    }
    if (bad_block) report(a.status, TG_STATUS_BAD_PAGE);
    __syncthreads();
    if (MODE == kCopy) continue;  // (the shared tables are rebuilt for the next unit)
    for (int m = tid; m < moves; m += kThreads) spage[freed[m]] = incoming[m];
    if (tid == 0 && a.promoted && moves) atomicAdd(reinterpret_cast<unsigned long long *>(a.promoted), (unsigned long long)moves);
    __syncthreads();
    // decode list: for each selected page (ascending), the block that now holds it
    for (int k = tid; k < a.K; k += kThreads) blk_of[k] = -1;
    __syncthreads();
    for (int k = tid; k < a.K; k += kThreads) {
      const int r = spage[k];
      if (r < 0 || r >= a.n_pages) continue;
      int lo = 0, hi = a.K;  // position of page r in the ascending selection
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (srow[mid] < r) lo = mid + 1;
        else hi = mid;
      }
      if (lo < a.K && srow[lo] == r) blk_of[lo] = sblock[k];
    }
    __syncthreads();
    for (int k = tid; k < a.K; k += kThreads) prow[k] = blk_of[k];
    __syncthreads();  // the shared tables are rebuilt for the next row
  }
}

}  // namespace

namespace {
int promote_launch(const char *name, int threads, tg_stream_t stream, int n_rows, const int32_t *rows,
                   int grid_limit, const uint8_t *unstable, int batch, int H, int n_pages, int K, const int32_t *sel,
                   int32_t *slot_page, const int32_t *slot_block, const int64_t *dense_base, const void *host_kv,
                   int page_bytes, void *pool, int64_t pool_pages, int32_t *pt_ids, int64_t *promoted,
                   int32_t *dev_status) {
  if (n_rows < 0 || batch < 0 || H <= 0 || n_pages < 1 || K < 1 || K > n_pages)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: bad sizes", name);
  if (n_pages > kMaxTierPages || K > kMaxTierK)
    return tgi::fail(TG_ERR_SHAPE, "%s: n_pages <= %d and K <= %d", name, kMaxTierPages, kMaxTierK);
  if (page_bytes <= 0 || page_bytes % 16) return tgi::fail(TG_ERR_SHAPE, "%s: page_bytes %% 16 != 0", name);
  if (n_rows == 0) return tgi::ok();
  if (!rows || !unstable || !sel || !slot_page || !slot_block || !dense_base || !host_kv || !pool || !pt_ids)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: NULL pointer argument", name);
  if ((reinterpret_cast<uintptr_t>(host_kv) | reinterpret_cast<uintptr_t>(pool)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: host_kv and pool must be 16-byte aligned", name);
  // the kernel reads host_kv directly: pinned host memory through its device-mapped address,
  // other host memory only where the device reads pageable memory itself (Grace: through the
  // host page tables over NVLink-C2C)
  const void *host_dev = nullptr;
  cudaPointerAttributes pa;
  cudaError_t he = cudaPointerGetAttributes(&pa, host_kv);
  if (he == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer) {
    host_dev = pa.devicePointer;
  } else {
    cudaGetLastError();  // clear the error of a failed query
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) == cudaSuccess && pageable &&
        (he != cudaSuccess || pa.type == cudaMemoryTypeUnregistered))
      host_dev = host_kv;
  }
  if (!host_dev)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: host_kv is neither pinned host memory nor readable "
                                         "pageable memory on this device", name);
  TierArgs a;
  a.rows = rows;
  a.n_rows = n_rows;
  a.unstable = unstable;
  a.H = H;
  a.n_pages = n_pages;
  a.K = K;
  a.sel = sel;
  a.slot_page = slot_page;
  a.slot_block = slot_block;
  a.dense_base = dense_base;
  a.host_kv = static_cast<const uint4 *>(host_dev);
  a.pool = static_cast<uint4 *>(pool);
  a.pool_pages = pool_pages;
  a.page_vec = page_bytes / 16;
  a.total_rows = (int64_t)batch * H;
  a.pt_ids = pt_ids;
  a.promoted = promoted;
  a.status = dev_status;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  a.slices = 1;
  if (threads == 64) {
    // background: the copy in slices over up to one small CTA per SM, then the tables
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
    int cap = grid_limit > 0 && grid_limit < sms ? grid_limit : sms;
    a.slices = (cap + n_rows - 1) / n_rows;
    const int64_t units = (int64_t)n_rows * a.slices;
    const int grid = (int)(units < cap ? units : cap);
    tier_promote_kernel<64, kCopy><<<grid, 64, 0, st>>>(a);
    tier_promote_kernel<64, kCommit><<<n_rows < cap ? n_rows : cap, 64, 0, st>>>(a);
  } else {
    const int grid = grid_limit > 0 ? (n_rows < grid_limit ? n_rows : grid_limit) : n_rows;
    tier_promote_kernel<256, kWhole><<<grid, 256, 0, st>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  return tgi::ok();
}
}  // namespace

extern "C" int tg_tier_promote(tg_stream_t stream, int n_rows, const int32_t *rows, int grid_limit,
                               const uint8_t *unstable, int batch, int H, int n_pages, int K, const int32_t *sel,
                               int32_t *slot_page, const int32_t *slot_block, const int64_t *dense_base,
                               const void *host_kv, int page_bytes, void *pool, int64_t pool_pages,
                               int32_t *pt_ids, int64_t *promoted, int32_t *dev_status) {
  return promote_launch("tg_tier_promote", 256, stream, n_rows, rows, grid_limit, unstable, batch, H, n_pages, K,
                        sel, slot_page, slot_block, dense_base, host_kv, page_bytes, pool, pool_pages, pt_ids,
                        promoted, dev_status);
}

extern "C" int tg_tier_promote_background(tg_stream_t stream, int n_rows, const int32_t *rows, int grid_limit,
                                          const uint8_t *unstable, int batch, int H, int n_pages, int K,
                                          const int32_t *sel, int32_t *slot_page, const int32_t *slot_block,
                                          const int64_t *dense_base, const void *host_kv, int page_bytes,
                                          void *pool, int64_t pool_pages, int32_t *pt_ids, int64_t *promoted,
                                          int32_t *dev_status) {
  return promote_launch("tg_tier_promote_background", 64, stream, n_rows, rows, grid_limit, unstable, batch, H,
                        n_pages, K, sel, slot_page, slot_block, dense_base, host_kv, page_bytes, pool, pool_pages,
                        pt_ids, promoted, dev_status);
}
