// Quest-style page scoring and per-KV-head top-K page selection, plus the
// per-page min/max key vectors it reads.
//
// Source: "FlexiCache: Leveraging Temporal Stability of Attention Heads for
// Efficient KV Cache Management (MLSys 2026)" (paper-review page):
//  "Core method / Sparse decode" -- every KV head attends only to its top-K
//  pages; a page is ranked by the min-max key bound of max q.k;
//  "Assumption 2" -- the min/max vectors form a MinMax cache resident on the
//  GPU, separate from the KV pages.
//
// Score of page p for KV head h: max over its g query heads j of
//   sum_d max(q_jd * mn_pd, q_jd * mx_pd)
// in float32, in one fixed order so the selection is reproducible: d is cut
// into 16 slices of d/16, each summed left to right; the 16 slice sums are then
// added pairwise (j, j+8), (j, j+4), (j, j+2), (j, j+1).  bf16 x bf16 products
// are exact in float32, and since mn <= mx exactly one of q+ mx and q- mn is
// nonzero (q+ = max(q, 0), q- = min(q, 0)), so two fused multiply-adds per
// element add exactly what multiply-max-add adds.
//
// Two kernels per call:
//  * page_score_kernel: the (request, KV head, page) units of the whole call
//    form one flat sequence (the MinMax rows are contiguous), split evenly over
//    one persistent CTA per SM and, inside it, over its warps.  Each warp
//    streams its contiguous range through its own ring of 1-D bulk copies; each
//    half warp scores its pages with lane j owning slice j; f32x2 FMAs pair two
//    query heads of one page (2 <= g <= 4 at d = 128, g = 2 at d = 256) or two
//    pages (g = 1), and wider groups use scalar FMAs, each chain in the fixed
//    order below.  The 16 slice sums are combined by an
//    xor butterfly that also spreads the g heads over the lanes (every add is
//    one of the fixed pairs; a + b == b + a in float32).  Scores go to the
//    workspace as order-preserving keys.
//  * page_select_warp_kernel (rows of up to 1024 pages: one warp per (request,
//    KV head), keys in registers) or page_select_kernel (longer rows: one CTA,
//    keys in shared memory): an exact radix select of the K-th largest key, then
//    an ascending sweep (ties to the lower page).
#include "block_select.cuh"
#include "score_body.cuh"

#include <cuda_runtime.h>

#include <algorithm>

namespace {

using namespace tgk;

template <int D, int GQ>
__global__ void __launch_bounds__(ScoreCfg<D>::NW * 32, 1) page_score_kernel(const ScoreArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  score_body<D, GQ>(a, smem);
}

// One CTA per (request, KV head): top-K of the row's keys, ascending, ties to the lower page.
__global__ void __launch_bounds__(kSelThreads) page_select_kernel(const uint32_t *keys, const int32_t *rows,
                                                                  int64_t total_rows, int n_pages, int K,
                                                                  int32_t *sel, int32_t *pt_ids,
                                                                  const int64_t *dense_base) {
  extern __shared__ uint32_t skeys[];  // [n_pages]
  __shared__ int hist[256];
  __shared__ int scan[33];
  __shared__ int sel_scratch[4];
  const int row = blockIdx.x, tid = threadIdx.x;  // list position
  const int64_t out_row = rows ? (int64_t)__ldcg(rows + row) : row;  // checked by the score kernel
  // the keys are written by the score kernel just before this one
  griddep_wait();
  if (out_row < 0 || out_row >= total_rows) return;
  const uint32_t *rk = keys + (size_t)row * n_pages;
  for (int i = tid; i < n_pages; i += kSelThreads) skeys[i] = __ldcg(rk + i);
  __syncthreads();
  uint32_t T;
  int need_eq;
  block_radix_select<kSelThreads>(n_pages, K, [&](int i) { return skeys[i]; }, hist, sel_scratch, T, need_eq);
  int taken = 0, eq_seen = 0;
  for (int c0 = 0; c0 < n_pages && taken < K; c0 += kSelThreads) {
    const int p = c0 + tid;
    const uint32_t key = p < n_pages ? skeys[p] : 0u;
    const bool gt = p < n_pages && key > T, eq = p < n_pages && key == T;
    int eq_total, sel_total;
    const int eq_rank = eq_seen + block_excl_count<kSelThreads>(eq, scan, eq_total);
    const bool take = gt || (eq && eq_rank < need_eq);
    const int k = taken + block_excl_count<kSelThreads>(take, scan, sel_total);
    if (take) {
      sel[(size_t)out_row * K + k] = p;
      if (pt_ids) pt_ids[(size_t)out_row * K + k] = (int32_t)((dense_base ? dense_base[out_row] : out_row * n_pages) + p);
    }
    taken += sel_total;
    eq_seen += eq_total;
  }
}

cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  return at;
}

template <int D, int GQ>
cudaError_t launch_score(const ScoreArgs &a, cudaStream_t s) {
  using CF = ScoreCfg<D>;
  auto fn = page_score_kernel<D, GQ>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, CF::NW * 32, CF::SMEM);
  if (e != cudaSuccess) return e;
  // one wave of persistent CTAs; no more CTAs than give each warp a full stage
  const int64_t want = (a.units + CF::NW * CF::SP - 1) / (CF::NW * CF::SP);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)std::max(1, per_sm) * sms, want));
  // may start while the previous kernel in the stream finishes (it reads only q and MinMax
  // before that kernel is done, and writes only keys, which no other kernel reads then)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(CF::NW * 32);
  cfg.dynamicSmemBytes = (size_t)CF::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

template <int D>
cudaError_t launch_score_d(const ScoreArgs &a, cudaStream_t s) {
  if (a.g <= 1) return launch_score<D, 1>(a, s);
  if (a.g <= 2) return launch_score<D, 2>(a, s);
  if (a.g <= 4) return launch_score<D, 4>(a, s);
  return launch_score<D, 8>(a, s);
}

cudaError_t launch_select(const uint32_t *keys, const int32_t *rows, int64_t total_rows, int n_rows, int n_pages,
                          int K, int32_t *sel, int32_t *pt_ids, const int64_t *dense_base, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(page_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMaxPages * 4);
  if (e != cudaSuccess) return e;
  // launched early behind the score kernel; it waits for it before reading the keys.  It
  // does not let the next kernel start early, so a decode launch that reads the page
  // lists written here always sees them complete
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(n_rows);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = (size_t)n_pages * 4;
  return cudaLaunchKernelEx(&cfg, page_select_kernel, keys, rows, total_rows, n_pages, K, sel, pt_ids, dense_base);
}

// minmax[b][h][p][0][:] = min over the page's valid keys, [1][:] = max (exact in bf16)
__global__ void build_minmax_kernel(const uint16_t *K, uint16_t *mm, int N, int P, int d, int n_pages,
                                    long long total) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (row, page, 2-element chunk)
  if (e >= total) return;
  const int c = (int)(e % (d / 2));
  const long long rp = e / (d / 2);
  const int p = (int)(rp % n_pages);
  const long long row = rp / n_pages;
  const int t0 = p * P, t1 = min(N, t0 + P);
  const uint32_t *src = reinterpret_cast<const uint32_t *>(K + ((size_t)row * N + t0) * d) + c;
  float mn0 = INFINITY, mn1 = INFINITY, mx0 = -INFINITY, mx1 = -INFINITY;
  // the page's rows are independent loads: unrolled so that they are all in flight
#pragma unroll 16
  for (int t = t0; t < t1; ++t, src += d / 2) {
    const uint32_t v = *src;
    mn0 = fminf(mn0, bf16_lo(v));
    mx0 = fmaxf(mx0, bf16_lo(v));
    mn1 = fminf(mn1, bf16_hi(v));
    mx1 = fmaxf(mx1, bf16_hi(v));
  }
  // values are bf16 already: take the upper 16 bits back unchanged
  uint32_t *dst = reinterpret_cast<uint32_t *>(mm + (((size_t)row * n_pages + p) * 2) * d) + c;
  dst[0] = (__float_as_uint(mn0) >> 16) | (__float_as_uint(mn1) & 0xffff0000u);
  dst[d / 2] = (__float_as_uint(mx0) >> 16) | (__float_as_uint(mx1) & 0xffff0000u);
}

}  // namespace

extern "C" int tg_page_score_workspace(int batch, int H, int n_pages, int64_t *workspace_bytes) {
  if (!workspace_bytes) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_workspace: NULL workspace_bytes");
  if (batch < 0 || H <= 0 || n_pages < 1) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_workspace: bad sizes");
  // page keys, then one page counter and one ready flag per (request, KV head)
  *workspace_bytes =
      tgi::align_up((int64_t)batch * H * n_pages * 4, 256) + 2 * tgi::align_up((int64_t)batch * H * 4, 256);
  return tgi::ok();
}

namespace {
int score_topk(const char *fn, tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K, int n_rows,
               const int32_t *rows, const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
               const int64_t *dense_base, void *workspace, int64_t workspace_bytes, uint32_t flags,
               int32_t *dev_status) {
  if (flags & ~TG_SCORE_LET_NEXT_START) return tgi::fail(TG_ERR_INVALID_ARG, "%s: unknown flags 0x%x", fn, flags);
  if (batch < 0 || H <= 0 || g < 1 || g > 8) return tgi::fail(TG_ERR_INVALID_ARG, "%s: bad batch/H/g", fn);
  if (d != 128 && d != 256) return tgi::fail(TG_ERR_SHAPE, "%s: d=%d (128 or 256)", fn, d);
  if (n_pages < 1 || n_pages > kMaxPages || K < 1 || K > n_pages)
    return tgi::fail(TG_ERR_SHAPE, "%s: need 1 <= K=%d <= n_pages=%d <= %d", fn, K, n_pages, kMaxPages);
  if (n_rows < 0 || (int64_t)n_rows > (int64_t)batch * H)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: n_rows=%d outside [0, batch*H]", fn, n_rows);
  if (batch == 0 || n_rows == 0) return tgi::ok();
  if (!q || !minmax || !sel || !workspace) return tgi::fail(TG_ERR_INVALID_ARG, "%s: NULL q/minmax/sel/workspace", fn);
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(minmax) | reinterpret_cast<uintptr_t>(workspace)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: q, minmax and workspace must be 16-byte aligned", fn);
  if ((int64_t)batch * H * n_pages > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "%s: page ids overflow int32", fn);
  const int64_t keys_bytes = tgi::align_up((int64_t)batch * H * n_pages * 4, 256);
  const int64_t need = keys_bytes + tgi::align_up((int64_t)batch * H * 4, 256);
  if (workspace_bytes < need)
    return tgi::fail(TG_ERR_CAPACITY, "%s: workspace %lld < %lld bytes", fn, (long long)workspace_bytes, (long long)need);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  ScoreArgs a;
  a.q = q;
  a.minmax = minmax;
  a.keys = reinterpret_cast<uint32_t *>(ws);
  a.row_cnt = reinterpret_cast<int32_t *>(ws + keys_bytes);
  a.sel = sel;
  a.pt_ids = pt_ids;
  a.status = dev_status;
  a.rows = rows;
  a.total_rows = (int64_t)batch * H;
  a.units = (int64_t)n_rows * n_pages;
  a.g = g;
  a.n_pages = n_pages;
  a.K = K;
  a.fused = n_pages <= 32 * kWarpKeysMax;
  a.let_next = (flags & TG_SCORE_LET_NEXT_START) != 0;
  a.dense_base = dense_base;
  a.row_ready = nullptr;
  a.epoch = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = d == 128 ? launch_score_d<128>(a, s) : launch_score_d<256>(a, s);
  if (e == cudaSuccess && !a.fused)
    e = launch_select(a.keys, rows, a.total_rows, n_rows, n_pages, K, sel, pt_ids, dense_base, s);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return tgi::ok();
}
}  // namespace

extern "C" int tg_page_score_topk(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                                  const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
                                  void *workspace, int64_t workspace_bytes, uint32_t flags, int32_t *dev_status) {
  return score_topk("tg_page_score_topk", stream, batch, H, g, d, n_pages, K, batch * H, nullptr, q, minmax, sel,
                    pt_ids, nullptr, workspace, workspace_bytes, flags, dev_status);
}

extern "C" int tg_page_score_topk_rows(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                                       int n_rows, const int32_t *rows, const uint16_t *q, const uint16_t *minmax,
                                       int32_t *sel, int32_t *pt_ids, const int64_t *dense_base, void *workspace,
                                       int64_t workspace_bytes, uint32_t flags, int32_t *dev_status) {
  if (n_rows > 0 && !rows) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_topk_rows: NULL rows");
  return score_topk("tg_page_score_topk_rows", stream, batch, H, g, d, n_pages, K, n_rows, rows, q, minmax, sel,
                    pt_ids, dense_base, workspace, workspace_bytes, flags, dev_status);
}

extern "C" int tg_build_minmax(tg_stream_t stream, int batch, int H, int N, int P, int d, const uint16_t *K,
                               uint16_t *minmax, int32_t *dev_status) {
  (void)dev_status;
  if (batch < 0 || H <= 0 || N <= 0 || P <= 0 || d <= 0 || d % 2)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_build_minmax: bad sizes");
  if (batch == 0) return tgi::ok();
  if (!K || !minmax) return tgi::fail(TG_ERR_INVALID_ARG, "tg_build_minmax: NULL K/minmax");
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(minmax)) & 3)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_build_minmax: K and minmax must be 4-byte aligned");
  const int n_pages = (N + P - 1) / P;
  const long long total = (long long)batch * H * n_pages * (d / 2);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_build_minmax: too large");
  build_minmax_kernel<<<(unsigned)blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(K, minmax, N, P, d,
                                                                                                n_pages, total);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_build_minmax: %s", cudaGetErrorString(e));
  return tgi::ok();
}
