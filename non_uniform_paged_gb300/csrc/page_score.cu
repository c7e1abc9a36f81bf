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

constexpr int kThreads = 256;
constexpr int kMaxPages = 16384;
constexpr int kChunkPages = 32;                      // pages per bulk copy
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // give up a copy wait after 2 s

template <int D>
struct ScoreCfg {
  static constexpr int NS = D == 256 ? 3 : 4;        // ring stages
  static constexpr int CHUNK = kChunkPages * 2 * D * 2;  // bytes per stage
  static int smem_bytes(int n_pages) { return NS * CHUNK + NS * 8 + n_pages * 4; }
};

struct ScoreArgs {
  const uint16_t *q, *minmax;
  int32_t *sel, *pt_ids, *status;
  int H, g, n_pages, K;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// One CTA per (request, KV head).  Thread 0 streams the row's MinMax vectors
// (contiguous, n_pages x 2 x d bf16) through an NS-stage shared-memory ring with
// 1-D bulk copies; every half warp scores pages out of shared memory.
template <int D, int GQ>
__global__ void __launch_bounds__(kThreads, 3) page_score_topk_kernel(const ScoreArgs a) {
  using CF = ScoreCfg<D>;
  constexpr int W = D / 16;  // elements per slice
  constexpr int WV = W / 8;  // 16-byte vectors per slice
  constexpr int NS = CF::NS, CHUNK = CF::CHUNK;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;                                           // [NS][CHUNK]
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + NS * CHUNK);  // [NS]
  uint32_t *keys = reinterpret_cast<uint32_t *>(bars + NS);        // [n_pages]
  __shared__ int hist[256];
  __shared__ int scan[33];
  __shared__ int sel_scratch[4];
  __shared__ int nan_flag;

  const int row = blockIdx.x, b = row / a.H, h = row % a.H;
  const int tid = threadIdx.x, lane = tid & 31;
  const int hw = tid >> 4, j = lane & 15;  // half warp 0..15, slice j
  if (tid == 0) {
    nan_flag = 0;
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
  }
  fence_barrier_init();
  __syncthreads();

  const uint8_t *src = reinterpret_cast<const uint8_t *>(a.minmax + (size_t)row * a.n_pages * 2 * D);
  const int nc = (a.n_pages + kChunkPages - 1) / kChunkPages;
  auto chunk_bytes = [&](int c) { return min(kChunkPages, a.n_pages - c * kChunkPages) * 2 * D * 2; };
  auto issue = [&](int c) {  // thread 0
    uint64_t *bar = &bars[c % NS];
    mbar_arrive_expect_tx(bar, (uint32_t)chunk_bytes(c));
    bulk_load(ring + (c % NS) * CHUNK, src + (size_t)c * CHUNK, (uint32_t)chunk_bytes(c), bar);
  };
  if (tid == 0)
    for (int c = 0; c < NS && c < nc; ++c) issue(c);

  // this lane's slice of the g query heads (heads past g contribute nothing)
  uint32_t qv[GQ][W / 2];
#pragma unroll
  for (int i = 0; i < GQ; ++i) {
    const int qi = i < a.g ? i : 0;
    const uint4 *qs = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.H * a.g + (size_t)h * a.g + qi) * D + j * W);
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const uint4 x = qs[v];
      qv[i][4 * v] = x.x; qv[i][4 * v + 1] = x.y; qv[i][4 * v + 2] = x.z; qv[i][4 * v + 3] = x.w;
    }
  }

  // q+ = max(q, 0) and q- = min(q, 0) of this lane's slice, as float32, when they fit in registers
  constexpr bool kSplitQ = GQ * W <= 32;
  float qp[kSplitQ ? GQ : 1][kSplitQ ? W : 1], qm[kSplitQ ? GQ : 1][kSplitQ ? W : 1];
  if constexpr (kSplitQ) {
#pragma unroll
    for (int i = 0; i < GQ; ++i)
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        const float lo = bf16_lo(qv[i][e / 2]), hi = bf16_hi(qv[i][e / 2]);
        qp[i][e] = fmaxf(lo, 0.f);
        qm[i][e] = fminf(lo, 0.f);
        qp[i][e + 1] = fmaxf(hi, 0.f);
        qm[i][e + 1] = fminf(hi, 0.f);
      }
  }

  bool nan_seen = false;
  int c = 0;
  bool failed = false;
  for (; c < nc; ++c) {
    const int s = c % NS;
    const bool ok = mbar_wait(&bars[s], (uint32_t)((c / NS) & 1), kWaitLimitNs);
    const int np = min(kChunkPages, a.n_pages - c * kChunkPages);
    const uint8_t *stage = ring + s * CHUNK;
    if constexpr (kSplitQ) {
      // this half warp scores pages hw and hw + 16 of the chunk together (two independent
      // sets of accumulator chains); pages past np read stale shared memory and are dropped
      const int pa = hw, pb = hw + 16;
      const uint4 *ra = reinterpret_cast<const uint4 *>(stage + pa * 4 * D + j * W * 2);
      const uint4 *rb = reinterpret_cast<const uint4 *>(stage + pb * 4 * D + j * W * 2);
      uint4 mna[WV], mxa[WV], mnb[WV], mxb[WV];
#pragma unroll
      for (int v = 0; v < WV; ++v) {
        mna[v] = ra[v];
        mxa[v] = ra[v + D / 8];  // the max row follows the min row: 2*D bytes = D/8 vectors
        mnb[v] = rb[v];
        mxb[v] = rb[v + D / 8];
      }
      // e_d = max(q_d mn_d, q_d mx_d) = q+_d mx_d + q-_d mn_d (mn <= mx, one product is 0):
      // two FMAs per element add exactly what mul-max-add adds, in the same order
      float acca[GQ], accb[GQ];
#pragma unroll
      for (int i = 0; i < GQ; ++i) acca[i] = accb[i] = 0.f;
#pragma unroll
      for (int v = 0; v < WV; ++v) {
        const uint32_t wna[4] = {mna[v].x, mna[v].y, mna[v].z, mna[v].w};
        const uint32_t wxa[4] = {mxa[v].x, mxa[v].y, mxa[v].z, mxa[v].w};
        const uint32_t wnb[4] = {mnb[v].x, mnb[v].y, mnb[v].z, mnb[v].w};
        const uint32_t wxb[4] = {mxb[v].x, mxb[v].y, mxb[v].z, mxb[v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int el = 8 * v + 2 * e;
          const float na0 = bf16_lo(wna[e]), na1 = bf16_hi(wna[e]), xa0 = bf16_lo(wxa[e]), xa1 = bf16_hi(wxa[e]);
          const float nb0 = bf16_lo(wnb[e]), nb1 = bf16_hi(wnb[e]), xb0 = bf16_lo(wxb[e]), xb1 = bf16_hi(wxb[e]);
#pragma unroll
          for (int i = 0; i < GQ; ++i) {
            acca[i] = fmaf(qp[i][el], xa0, acca[i]);
            accb[i] = fmaf(qp[i][el], xb0, accb[i]);
            acca[i] = fmaf(qm[i][el], na0, acca[i]);
            accb[i] = fmaf(qm[i][el], nb0, accb[i]);
            acca[i] = fmaf(qp[i][el + 1], xa1, acca[i]);
            accb[i] = fmaf(qp[i][el + 1], xb1, accb[i]);
            acca[i] = fmaf(qm[i][el + 1], na1, acca[i]);
            accb[i] = fmaf(qm[i][el + 1], nb1, accb[i]);
          }
        }
      }
      float besta = -INFINITY, bestb = -INFINITY;
#pragma unroll
      for (int i = 0; i < GQ; ++i) {
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
          acca[i] = __fadd_rn(acca[i], __shfl_xor_sync(0xffffffffu, acca[i], off));
          accb[i] = __fadd_rn(accb[i], __shfl_xor_sync(0xffffffffu, accb[i], off));
        }
        if (i < a.g) {
          besta = i == 0 ? acca[i] : fmaxf(besta, acca[i]);
          bestb = i == 0 ? accb[i] : fmaxf(bestb, accb[i]);
        }
      }
      if (j == 0 && ok) {
        if (pa < np) {
          nan_seen |= is_nan(besta);
          keys[c * kChunkPages + pa] = float_key(besta);
        }
        if (pb < np) {
          nan_seen |= is_nan(bestb);
          keys[c * kChunkPages + pb] = float_key(bestb);
        }
      }
    } else {
#pragma unroll
    for (int pl0 = 0; pl0 < kChunkPages; pl0 += 16) {  // both halves of a warp take 2 pages each
      const int pl = pl0 + hw;
      const bool valid = ok && pl < np;
      uint4 mnv[WV], mxv[WV];
#pragma unroll
      for (int v = 0; v < WV; ++v) {
        mnv[v] = valid ? reinterpret_cast<const uint4 *>(stage + pl * 4 * D + j * W * 2)[v] : make_uint4(0, 0, 0, 0);
        mxv[v] = valid ? reinterpret_cast<const uint4 *>(stage + pl * 4 * D + 2 * D + j * W * 2)[v] : make_uint4(0, 0, 0, 0);
      }
      float best = -INFINITY;
#pragma unroll
      for (int i = 0; i < GQ; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int v = 0; v < WV; ++v) {
          const uint32_t mnw[4] = {mnv[v].x, mnv[v].y, mnv[v].z, mnv[v].w};
          const uint32_t mxw[4] = {mxv[v].x, mxv[v].y, mxv[v].z, mxv[v].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t qq = qv[i][4 * v + e];
            const float e_lo = fmaxf(__fmul_rn(bf16_lo(qq), bf16_lo(mnw[e])), __fmul_rn(bf16_lo(qq), bf16_lo(mxw[e])));
            acc = __fadd_rn(acc, e_lo);
            const float e_hi = fmaxf(__fmul_rn(bf16_hi(qq), bf16_hi(mnw[e])), __fmul_rn(bf16_hi(qq), bf16_hi(mxw[e])));
            acc = __fadd_rn(acc, e_hi);
          }
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
        if (i < a.g) {
          nan_seen |= valid && is_nan(acc);
          best = i == 0 ? acc : fmaxf(best, acc);
        }
      }
      if (j == 0 && valid) keys[c * kChunkPages + pl] = float_key(best);
    }
    }
    // every thread is done with stage s; thread 0 refills it
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0 && c + NS < nc) {
      fence_proxy_async_smem();
      issue(c + NS);
    }
  }
  if (failed) {  // a copy wait gave up: report, drain our own copies in flight, leave
    if (tid == 0) {
      report(a.status, TG_STATUS_TIMEOUT);
      for (int t = c; t < nc && t < c + NS; ++t)
        if (!mbar_wait(&bars[t % NS], (uint32_t)((t / NS) & 1), kWaitLimitNs)) break;
    }
    return;
  }
  if (nan_seen) nan_flag = 1;
  __syncthreads();
  if (nan_flag && tid == 0) report(a.status, TG_STATUS_NONFINITE);

  uint32_t T;
  int need_eq;
  block_radix_select<kThreads>(a.n_pages, a.K, [&](int i) { return keys[i]; }, hist, sel_scratch, T, need_eq);

  int taken = 0, eq_seen = 0;
  for (int c0 = 0; c0 < a.n_pages && taken < a.K; c0 += kThreads) {
    const int p = c0 + tid;
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
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       ScoreCfg<D>::smem_bytes(kMaxPages));
  if (e != cudaSuccess) return e;
  fn<<<rows, kThreads, ScoreCfg<D>::smem_bytes(a.n_pages), s>>>(a);
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
