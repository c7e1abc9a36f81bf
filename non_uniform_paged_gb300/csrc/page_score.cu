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
// into 16 slices of d/16, each summed left to right by one lane of a 16-lane
// half warp; the 16 lane sums are then added by xor-shuffles 8, 4, 2, 1, i.e.
// pairs (j, j+8), (j, j+4), (j, j+2), (j, j+1).  bf16 x bf16 products are exact
// in float32 and no multiply is fused into an add.
//
// One CTA per (request, KV head): scores of all pages go to shared memory as
// order-preserving keys, then an exact radix select finds the K-th largest
// and an ascending sweep lists the winners (ties to the lower page).
#include "block_select.cuh"
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

namespace {

using namespace tgk;

constexpr int kThreads = 512;
constexpr int kMaxPages = 16384;

struct ScoreArgs {
  const uint16_t *q, *minmax;
  int32_t *sel, *pt_ids, *status;
  int H, g, n_pages, K;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <int D, int GQ>
__global__ void __launch_bounds__(kThreads) page_score_topk_kernel(const ScoreArgs a) {
  constexpr int W = D / 16;      // elements per slice
  constexpr int WV = W / 8;      // 16-byte vectors per slice
  constexpr int NWARP = kThreads / 32;
  constexpr int kUnroll = D == 256 ? 2 : 4;  // pages per half warp in flight (register budget)
  extern __shared__ uint32_t keys[];  // [n_pages]
  __shared__ int hist[256];
  __shared__ int scan[33];
  __shared__ int sel_scratch[4];
  __shared__ int nan_flag;

  const int row = blockIdx.x, b = row / a.H, h = row % a.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, j = lane & 15;
  if (threadIdx.x == 0) nan_flag = 0;

  // this lane's slice of the g query heads (heads past g contribute nothing)
  uint32_t qv[GQ][W / 2];
#pragma unroll
  for (int i = 0; i < GQ; ++i) {
    const int qi = i < a.g ? i : 0;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.H * a.g + (size_t)h * a.g + qi) * D + j * W);
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const uint4 x = src[v];
      qv[i][4 * v] = x.x; qv[i][4 * v + 1] = x.y; qv[i][4 * v + 2] = x.z; qv[i][4 * v + 3] = x.w;
    }
  }
  __syncthreads();

  const uint16_t *mm_row = a.minmax + (size_t)row * a.n_pages * 2 * D;
  bool nan_seen = false;
  // the loop bound is the warp's base page so both halves iterate together (shuffles below)
  for (int base = warp * 2; base < a.n_pages; base += NWARP * 2 * kUnroll) {
    const int p0 = base + half;
    uint4 mnv[kUnroll][WV], mxv[kUnroll][WV];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int p = p0 + u * NWARP * 2;
      for (int v = 0; v < WV; ++v) mnv[u][v] = mxv[u][v] = make_uint4(0, 0, 0, 0);
      if (p < a.n_pages) {
        const uint4 *mn = reinterpret_cast<const uint4 *>(mm_row + (size_t)p * 2 * D + j * W);
        const uint4 *mx = reinterpret_cast<const uint4 *>(mm_row + (size_t)p * 2 * D + D + j * W);
#pragma unroll
        for (int v = 0; v < WV; ++v) {
          mnv[u][v] = __ldcs(mn + v);
          mxv[u][v] = __ldcs(mx + v);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int p = p0 + u * NWARP * 2;  // uniform within the half warp
      float best = -INFINITY;
#pragma unroll
      for (int i = 0; i < GQ; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int v = 0; v < WV; ++v) {
          const uint32_t mnw[4] = {mnv[u][v].x, mnv[u][v].y, mnv[u][v].z, mnv[u][v].w};
          const uint32_t mxw[4] = {mxv[u][v].x, mxv[u][v].y, mxv[u][v].z, mxv[u][v].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t qq = qv[i][4 * v + c];
            const float e_lo = fmaxf(__fmul_rn(bf16_lo(qq), bf16_lo(mnw[c])), __fmul_rn(bf16_lo(qq), bf16_lo(mxw[c])));
            acc = __fadd_rn(acc, e_lo);
            const float e_hi = fmaxf(__fmul_rn(bf16_hi(qq), bf16_hi(mnw[c])), __fmul_rn(bf16_hi(qq), bf16_hi(mxw[c])));
            acc = __fadd_rn(acc, e_hi);
          }
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
        if (i < a.g) {
          nan_seen |= is_nan(acc);
          best = i == 0 ? acc : fmaxf(best, acc);
        }
      }
      if (j == 0 && p < a.n_pages) keys[p] = float_key(best);
    }
  }
  if (nan_seen) nan_flag = 1;
  __syncthreads();
  if (nan_flag && threadIdx.x == 0) report(a.status, TG_STATUS_NONFINITE);

  uint32_t T;
  int need_eq;
  block_radix_select<kThreads>(a.n_pages, a.K, [&](int i) { return keys[i]; }, hist, sel_scratch, T, need_eq);

  int taken = 0, eq_seen = 0;
  for (int c0 = 0; c0 < a.n_pages && taken < a.K; c0 += kThreads) {
    const int p = c0 + threadIdx.x;
    const uint32_t key = p < a.n_pages ? keys[p] : 0u;
    const bool gt = p < a.n_pages && key > T, eq = p < a.n_pages && key == T;
    int eq_total, sel_total;
    const int eq_rank = eq_seen + block_excl_count<kThreads>(eq, scan, eq_total);
    const bool sel = gt || (eq && eq_rank < need_eq);
    const int k = taken + block_excl_count<kThreads>(sel, scan, sel_total);
    if (sel) {
      a.sel[(size_t)row * a.K + k] = p;
      if (a.pt_ids) a.pt_ids[(size_t)row * a.K + k] = row * a.n_pages + p;
    }
    taken += sel_total;
    eq_seen += eq_total;
  }
}

template <int D, int GQ>
cudaError_t launch_score(const ScoreArgs &a, int rows, cudaStream_t s) {
  auto fn = page_score_topk_kernel<D, GQ>;
  const int smem = a.n_pages * 4;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxPages * 4);
  if (e != cudaSuccess) return e;
  fn<<<rows, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_score_d(const ScoreArgs &a, int rows, cudaStream_t s) {
  if (a.g <= 1) return launch_score<D, 1>(a, rows, s);
  if (a.g <= 2) return launch_score<D, 2>(a, rows, s);
  if (a.g <= 4) return launch_score<D, 4>(a, rows, s);
  return launch_score<D, 8>(a, rows, s);
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

extern "C" int tg_page_score_topk(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                                  const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
                                  int32_t *dev_status) {
  if (batch < 0 || H <= 0 || g < 1 || g > 8) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_topk: bad batch/H/g");
  if (d != 128 && d != 256) return tgi::fail(TG_ERR_SHAPE, "tg_page_score_topk: d=%d (128 or 256)", d);
  if (n_pages < 1 || n_pages > kMaxPages || K < 1 || K > n_pages)
    return tgi::fail(TG_ERR_SHAPE, "tg_page_score_topk: need 1 <= K=%d <= n_pages=%d <= %d", K, n_pages, kMaxPages);
  if (batch == 0) return tgi::ok();
  if (!q || !minmax || !sel) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_topk: NULL q/minmax/sel");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(minmax)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_topk: q and minmax must be 16-byte aligned");
  if ((int64_t)batch * H * n_pages > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_page_score_topk: page ids overflow int32");
  ScoreArgs a{q, minmax, sel, pt_ids, dev_status, H, g, n_pages, K};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (d == 128) e = launch_score_d<128>(a, batch * H, s);
  else e = launch_score_d<256>(a, batch * H, s);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_page_score_topk: %s", cudaGetErrorString(e));
  return tgi::ok();
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
