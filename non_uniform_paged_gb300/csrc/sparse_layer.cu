// One sparse decode layer in one persistent kernel: Quest page scores, per-KV-head top-K
// pages, and flash decoding over them.
//
// Source: "FlexiCache: Leveraging Temporal Stability of Attention Heads for
// Efficient KV Cache Management (MLSys 2026)" (paper-review page), "Core method /
// Sparse decode" (every head attends only to its top-K pages, ranked by the
// Quest min-max bound).
//
// The layer's three steps run as two phases of one cooperative launch (every CTA
// resident, one per SM):
//  * score phase: the page-score body (flat split of all (request, head, page)
//    units; the warp that completes a row selects its top K) -- each selected row
//    also raises its ready flag to this call's epoch (release store);
//  * decode phase: the same CTAs reuse their shared memory for the split-KV decode
//    body of the plan; each CTA waits (bounded, acquire loads) for the flags of the
//    rows its work items read, then streams their pages.
// Compared with two kernels, the decode starts without a launch or a drained grid,
// and a CTA whose rows are selected decodes while other rows are still being
// selected.  The arithmetic is the two kernels': the results are bit-identical.
#include "decode_body.cuh"
#include "score_body.cuh"

#include <algorithm>

namespace {

constexpr int kD = 128;

// Launched with the decode body's threads; the score phase streams on its first ScoreCfg::NW
// warps, and the rest join its barriers and row selections.
template <int GQ>
__global__ void __launch_bounds__(Layout<kD>::THREADS, 1)
    sparse_layer_kernel(const __grid_constant__ CUtensorMap pool_map, const ScoreArgs sa, const DecodeArgs da) {
  static_assert(ScoreCfg<kD>::NW <= Layout<kD>::THREADS / 32, "the score phase runs on the decode's warps");
  extern __shared__ __align__(1024) uint8_t smem[];
  score_body<kD, GQ>(sa, smem);
  __syncthreads();
  // the score phase's mbarriers return to plain shared memory before the decode phase reuses it
  constexpr int kBars = ScoreCfg<kD>::NW * ScoreCfg<kD>::R;
  if (threadIdx.x < kBars) mbar_inval(reinterpret_cast<uint64_t *>(smem + ScoreCfg<kD>::RING) + threadIdx.x);
  __syncthreads();
  decode_body<kD>(&pool_map, da, smem);
}

template <int GQ>
int launch_fused(const char *fn_name, const CUtensorMap &map, const ScoreArgs &sa, const DecodeArgs &da, int grid,
                 cudaStream_t s) {
  auto fn = sparse_layer_kernel<GQ>;
  const int smem = std::max(ScoreCfg<kD>::SMEM, Layout<kD>::smem_bytes(da.g));
  const int threads = Layout<kD>::THREADS;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: %s", fn_name, cudaGetErrorString(e));
  // the decode phase waits for rows other CTAs select: every CTA must be resident at once
  if ((int64_t)per_sm * sms < grid)
    return tgi::fail(TG_ERR_SHAPE, "%s: the plan's %d CTAs exceed the %d that can be resident together", fn_name, grid,
                     per_sm * sms);
  void *params[] = {const_cast<CUtensorMap *>(&map), const_cast<ScoreArgs *>(&sa), const_cast<DecodeArgs *>(&da)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(fn), params);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: launch failed: %s", fn_name, cudaGetErrorString(e));
  return TG_OK;
}

}  // namespace

extern "C" int tg_sparse_layer(tg_stream_t stream, const void *plan_host, const void *plan_dev, int n_pages, int K,
                               int n_rows, const int32_t *rows, const uint8_t *due, int64_t wait_limit_ns,
                               const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
                               void *score_ws, int64_t score_ws_bytes, int epoch, const uint16_t *pool,
                               int64_t pool_pages, const int64_t *pt_off, float scale, void *workspace,
                               int64_t workspace_bytes, uint16_t *out, float *lse, int32_t *dev_status) {
  const char *fn_name = "tg_sparse_layer";
  if (!plan_host || !plan_dev || !q || !minmax || !sel || !pt_ids || !score_ws || !pool || !pt_off || !workspace ||
      !out)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_sparse_layer: NULL pointer argument");
  const tg_plan_header *hd;
  const tg_plan_layer *lt;
  int rc = check_decode_call(fn_name, plan_host, plan_dev, 0, q, pool, scale, &hd, &lt);
  if (rc) return rc;
  const int batch = hd->batch, H = hd->H, g = hd->H_q / hd->H;
  if (hd->d != kD || hd->H_p != 1 || g < 1 || g > 8)
    return tgi::fail(TG_ERR_SHAPE, "tg_sparse_layer: needs a plan of d=%d, H_p=1 page lists, g <= 8", kD);
  if (n_pages < 1 || n_pages > 32 * kWarpKeysMax || K < 1 || K > n_pages)
    return tgi::fail(TG_ERR_SHAPE, "tg_sparse_layer: need 1 <= K=%d <= n_pages=%d <= %d", K, n_pages,
                     32 * kWarpKeysMax);
  if (epoch < 1) return tgi::fail(TG_ERR_INVALID_ARG, "tg_sparse_layer: epoch must be >= 1");
  if (wait_limit_ns < 0) return tgi::fail(TG_ERR_INVALID_ARG, "tg_sparse_layer: wait_limit_ns < 0");
  if (rows && (n_rows < 0 || (int64_t)n_rows > (int64_t)batch * H))
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_sparse_layer: n_rows=%d outside [0, batch*H]", n_rows);
  if (rows && !due) return tgi::fail(TG_ERR_INVALID_ARG, "tg_sparse_layer: a row list needs its due map");
  if ((int64_t)batch * H * n_pages > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_sparse_layer: page ids overflow int32");
  const int64_t nrow_total = (int64_t)batch * H;
  const int32_t *rows_list = rows;
  const int64_t keys_bytes = tgi::align_up(nrow_total * n_pages * 4, 256), cnt_bytes = tgi::align_up(nrow_total * 4, 256);
  if (score_ws_bytes < keys_bytes + 2 * cnt_bytes)
    return tgi::fail(TG_ERR_CAPACITY, "tg_sparse_layer: score workspace %lld < %lld bytes", (long long)score_ws_bytes,
                     (long long)(keys_bytes + 2 * cnt_bytes));
  if (workspace_bytes < hd->workspace_bytes)
    return tgi::fail(TG_ERR_CAPACITY, "tg_sparse_layer: workspace %lld < %lld bytes", (long long)workspace_bytes,
                     (long long)hd->workspace_bytes);
  if (((reinterpret_cast<uintptr_t>(minmax) | reinterpret_cast<uintptr_t>(score_ws)) & 15) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_sparse_layer: minmax and score workspace 16-byte, workspace 256-byte aligned");
  CUtensorMap map;
  rc = make_pool_map(&map, pool, pool_pages, hd, fn_name);
  if (rc) return rc;
  uint8_t *sws = static_cast<uint8_t *>(score_ws);
  int32_t *ready = reinterpret_cast<int32_t *>(sws + keys_bytes + cnt_bytes);
  ScoreArgs sa;
  sa.q = q;
  sa.minmax = minmax;
  sa.keys = reinterpret_cast<uint32_t *>(sws);
  sa.row_cnt = reinterpret_cast<int32_t *>(sws + keys_bytes);
  sa.sel = sel;
  sa.pt_ids = pt_ids;
  sa.status = dev_status;
  sa.rows = rows_list;
  sa.total_rows = nrow_total;
  sa.units = (rows_list ? (int64_t)n_rows : nrow_total) * n_pages;
  sa.g = g;
  sa.n_pages = n_pages;
  sa.K = K;
  sa.fused = 1;
  sa.let_next = 0;
  sa.dense_base = nullptr;
  sa.row_ready = ready;
  sa.epoch = epoch;
  DecodeArgs da = decode_args(hd, lt, plan_dev, static_cast<uint8_t *>(workspace), q, out, lse, pt_off, pt_ids,
                              pool_pages, scale, dev_status, nullptr);
  da.row_ready = ready;
  da.row_due = rows_list ? due : nullptr;
  if (wait_limit_ns > 0) da.wait_ns = (uint64_t)wait_limit_ns;
  da.epoch = epoch;
  da.wait_tables = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (g <= 1) return launch_fused<1>(fn_name, map, sa, da, hd->N_CTA, s);
  if (g <= 2) return launch_fused<2>(fn_name, map, sa, da, hd->N_CTA, s);
  if (g <= 4) return launch_fused<4>(fn_name, map, sa, da, hd->N_CTA, s);
  return launch_fused<8>(fn_name, map, sa, da, hd->N_CTA, s);
}
