// Split-KV flash decoding over the ragged (head-wise non-uniform) page pool,
// with the log-sum-exp merge fused in.
//
// Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
// Multi-turn LLM Serving" (paper-review page), 3.2 Ragged Paging (group pages
// of H_p x 2 x P x d elements) and 3.3 AOT Load Balancing (one launch of N_CTA
// CTAs per layer, each CTA given an equal share of its group's retained tokens
// by the static split map); "FlexiCache ... (MLSys 2026)" (paper-review page),
// "Core method / Sparse decode" (flash decoding restricted to per-head page
// lists).
//
// Design (GB300):
//  * One persistent CTA per SM slot: NW streaming warps and NE epilogue warps.
//    The CTA walks its work items (pieces of one (request, KV head) run); inside
//    an item, 16-token tiles go round-robin to the streaming warps.
//  * Each warp owns an R-stage ring in shared memory.  Its lane 0 streams the
//    K and V rows of a tile with 2-D TMA loads (128-byte swizzle) that complete
//    on the stage's mbarrier; the warp waits with a time limit.
//  * Q.K^T and P.V run on the tensor cores as bf16 m16n8k16 MMAs with float32
//    accumulation: S^T[16 tokens x 8] = K[16 x d] . Q^T[d x 8] (the g <= 8
//    query heads of the KV head are the N columns), then O^T[d x 8] +=
//    V^T[d x 16] . P^T[16 x 8].  movmatrix turns the S^T accumulator into the
//    P^T operand without shared memory.  Online softmax in base 2.
//  * At the end of an item each streaming warp hands its (m, l, O) to the
//    epilogue warps through a double-buffered shared-memory slot and streams
//    on.  The epilogue merges the warps' states: a run finished by one CTA is
//    normalised and written directly; a run shared by several CTAs leaves a
//    float32 partial in the workspace, and the last CTA to finish (atomic
//    counter, no waiting) merges all partials and resets the counter.  Pieces
//    of shared runs are processed first, so their merges overlap streaming.
#include "decode_body.cuh"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

namespace {

using namespace tgk;

template <int D>
__global__ void __launch_bounds__(Layout<D>::THREADS, 1)
    ragged_decode_kernel(const __grid_constant__ CUtensorMap pool_map, const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  decode_body<D>(&pool_map, a, smem_raw);
}

template <int D>
void *kernel_ptr() {
  return reinterpret_cast<void *>(&ragged_decode_kernel<D>);
}

int kernel_config(int d, int g, void **fn, int *threads, int *smem) {
  if (d == 128) {
    *fn = kernel_ptr<128>();
    *threads = Layout<128>::THREADS;
    *smem = Layout<128>::smem_bytes(g);
  } else if (d == 256) {
    *fn = kernel_ptr<256>();
    *threads = Layout<256>::THREADS;
    *smem = Layout<256>::smem_bytes(g);
  } else {
    return tgi::fail(TG_ERR_SHAPE, "tg_decode_attn: d=%d (128 or 256)", d);
  }
  if (g < 1 || g > 8) return tgi::fail(TG_ERR_SHAPE, "tg_decode_attn: g=%d (1..8)", g);
  cudaError_t e = cudaFuncSetAttribute(*fn, cudaFuncAttributeMaxDynamicSharedMemorySize, *smem);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  return TG_OK;
}

}  // namespace

extern "C" int tg_query_ncta(int d, int g, int *N_CTA) {
  if (!N_CTA) return tgi::fail(TG_ERR_INVALID_ARG, "tg_query_ncta: NULL N_CTA");
  void *fn;
  int threads, smem;
  int rc = kernel_config(d, g, &fn, &threads, &smem);
  if (rc) return rc;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_query_ncta: %s", cudaGetErrorString(e));
  *N_CTA = per_sm * sms;
  return tgi::ok();
}

extern "C" int tg_decode_attn(tg_stream_t stream, const void *plan_host, const void *plan_dev, int layer,
                              const uint16_t *q, const uint16_t *pool, int64_t pool_pages,
                              const int64_t *pt_off, const int32_t *pt_ids, float scale,
                              void *workspace, int64_t workspace_bytes,
                              uint16_t *out, float *lse, int32_t *dev_status, int64_t *cta_time) {
  const char *fn_name = "tg_decode_attn";
  if (!plan_host || !plan_dev || !q || !pool || !pt_off || !pt_ids || !workspace || !out)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_decode_attn: NULL pointer argument");
  const tg_plan_header *hd;
  const tg_plan_layer *lt;
  int rc = check_decode_call(fn_name, plan_host, plan_dev, layer, q, pool, scale, &hd, &lt);
  if (rc) return rc;
  if (workspace_bytes < hd->workspace_bytes)
    return tgi::fail(TG_ERR_CAPACITY, "tg_decode_attn: workspace %lld < %lld bytes", (long long)workspace_bytes,
                     (long long)hd->workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_decode_attn: workspace must be 256-byte aligned");
  void *fn;
  int threads, smem;
  rc = kernel_config(hd->d, hd->H_q / hd->H, &fn, &threads, &smem);
  if (rc) return rc;
  CUtensorMap map;
  rc = make_pool_map(&map, pool, pool_pages, hd, fn_name);
  if (rc) return rc;
  DecodeArgs args = decode_args(hd, lt, plan_dev, static_cast<uint8_t *>(workspace), q, out, lse, pt_off, pt_ids,
                                pool_pages, scale, dev_status, cta_time);
  void *params[] = {&map, &args};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(hd->N_CTA);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, params);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_decode_attn: launch failed: %s", cudaGetErrorString(e));
  return tgi::ok();
}

// ---------------------------------------------------------------------------
// Allocation-free variant of tg_decode_attn.
//
// Some callers cannot allocate device memory when they call us: a serving
// process whose allocator reserved all GPU memory up front, or a plug-in that
// runs inside a host framework that owns the device heap, gets an error (or
// breaks the host's memory accounting) from cudaMalloc at request time.  This
// entry point takes its scratch (merge counters and split-KV partials) from
// the fixed array below instead of a caller workspace.
//
// The array lives in this library's module on every GPU that loads it, until
// the process exits.  Under CUDA's lazy module loading (the default) the
// module, and with it the array, is loaded on this entry point's first call on
// a device; a caller that reserves the GPU heap for its own allocator should
// make one call (or run with CUDA_MODULE_LOADING=EAGER) before reserving it.
// The array's device address belongs to a CUDA context, not to a device: it is
// looked up with cudaGetSymbolAddress on the first call in each context and
// cached under the context's unique id (cuCtxGetId), so a call after a device
// reset, or from another context on the same device, looks it up again.  Make
// the first call in a context before any stream capture.  Every call shares
// the array: the counters are cleared (cudaMemsetAsync) at the start of each
// call, and calls that overlap on the GPU (two streams, two host threads) race
// on it.
constexpr int64_t kStaticScratchBytes = 4 << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchSlot {
  unsigned long long ctx_id;  // cuCtxGetId of the context the address belongs to
  void *addr;
};
ScratchSlot g_scratch_slot[kMaxDevices] = {};

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry points (no link to libcuda)
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns &ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return f;
}

// the array's address in the current context (the runtime has made it current by now)
int static_scratch_address(void **out) {
  const char *fn_name = "tg_decode_attn_static_scratch";
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: %s", fn_name, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: device %d >= %d", fn_name, dev, kMaxDevices);
  const CtxFns &cf = ctx_fns();
  if (!cf.get_current || !cf.get_id) return tgi::fail(TG_ERR_CUDA, "%s: cuCtxGetCurrent/cuCtxGetId unavailable", fn_name);
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (cf.get_current(&ctx) != CUDA_SUCCESS || !ctx || cf.get_id(ctx, &id) != CUDA_SUCCESS)
    return tgi::fail(TG_ERR_CUDA, "%s: no current CUDA context", fn_name);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot &slot = g_scratch_slot[dev];
  if (!slot.addr || slot.ctx_id != id) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return tgi::fail(TG_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", fn_name, cudaGetErrorString(e));
    slot.ctx_id = id;
    slot.addr = p;
  }
  *out = slot.addr;
  return TG_OK;
}
}  // namespace

extern "C" int tg_decode_attn_static_scratch(tg_stream_t stream, const void *plan_host, const void *plan_dev,
                                             int layer, const uint16_t *q, const uint16_t *pool,
                                             int64_t pool_pages, const int64_t *pt_off, const int32_t *pt_ids,
                                             float scale, uint16_t *out, float *lse, int32_t *dev_status,
                                             int64_t *cta_time) {
  const char *fn_name = "tg_decode_attn_static_scratch";
  if (!plan_host || !plan_dev || !q || !pool || !pt_off || !pt_ids || !out)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_decode_attn_static_scratch: NULL pointer argument");
  // device faults (a copy wait that timed out, a bad page id) are reported only through the
  // caller's status word: the array's own word is cleared by the next call and read by nobody
  if (!dev_status)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_decode_attn_static_scratch: dev_status is required (device faults "
                                         "are reported only there)");
  const tg_plan_header *hd;
  const tg_plan_layer *lt;
  int rc = check_decode_call(fn_name, plan_host, plan_dev, layer, q, pool, scale, &hd, &lt);
  if (rc) return rc;
  if (hd->workspace_bytes > kStaticScratchBytes)
    return tgi::fail(TG_ERR_CAPACITY,
                     "tg_decode_attn_static_scratch: the plan needs %lld bytes of scratch, more than the fixed "
                     "%lld-byte array; use tg_decode_attn with a caller workspace",
                     (long long)hd->workspace_bytes, (long long)kStaticScratchBytes);
  void *fn;
  int threads, smem;
  rc = kernel_config(hd->d, hd->H_q / hd->H, &fn, &threads, &smem);
  if (rc) return rc;
  void *scratch = nullptr;
  rc = static_scratch_address(&scratch);
  if (rc) return rc;
  CUtensorMap map;
  rc = make_pool_map(&map, pool, pool_pages, hd, fn_name);
  if (rc) return rc;
  uint8_t *ws = static_cast<uint8_t *>(scratch);
  const tgi::WorkspaceLayout wl = tgi::workspace_layout(hd->batch, hd->H, hd->H_q / hd->H, hd->d, hd->max_slots);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the merge counters must start at zero
  cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)wl.ml, st);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_decode_attn_static_scratch: memset: %s", cudaGetErrorString(e));
  DecodeArgs args = decode_args(hd, lt, plan_dev, ws, q, out, lse, pt_off, pt_ids, pool_pages, scale, dev_status,
                                cta_time);
  void *params[] = {&map, &args};
  e = cudaLaunchKernel(fn, dim3(hd->N_CTA), dim3(threads), params, (size_t)smem, st);
  if (e != cudaSuccess)
    return tgi::fail(TG_ERR_CUDA, "tg_decode_attn_static_scratch: launch failed: %s", cudaGetErrorString(e));
  return tgi::ok();
}

extern "C" int tg_check_status(const int32_t *dev_status, int32_t *host_status) {
  if (!dev_status) return tgi::fail(TG_ERR_INVALID_ARG, "tg_check_status: NULL");
  int32_t v = 0;
  cudaError_t e = cudaMemcpy(&v, dev_status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_check_status: %s", cudaGetErrorString(e));
  if (host_status) *host_status = v;
  if (v & TG_STATUS_TIMEOUT) return tgi::fail(TG_ERR_TIMEOUT, "device status 0x%x: a copy wait timed out", v);
  if (v) return tgi::fail(TG_ERR_DEVICE, "device status 0x%x", v);
  return tgi::ok();
}
