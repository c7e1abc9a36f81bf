// Token top-k retention and compaction into the ragged group pages.
//
// Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
// Multi-turn LLM Serving" (paper-review page), 3.1 Budget Reservation
// (I_{l,h} = Top(ceil(B_{l,h} N), s_{l,h}), done as each prefill chunk's KV is
// ready) and 3.2 Ragged Paging (each H_p-head group writes into its own pages
// of H_p x 2 x P x d elements).
//
// One 1024-thread CTA per SM; a row (request, KV head) gets C of them (C chosen so
// the grid fills the GPU, or, for up to 1024 rows, shares in proportion to the
// rows' work, rounded on the running sum).  CTA j of a row owns tokens
// [j N / C, (j+1) N / C) and talks to no other CTA:
//  1. exact top-n by an MSB-first radix select over order-preserving keys of
//     the float32 scores (every CTA of the row finds the same n-th largest key
//     T and how many keys equal to T to keep; the keys sit in shared memory when
//     the row fits, else in L2);
//  2. block-wide counts of the kept keys before its chunk give the chunk's
//     first output position;
//  3. one ascending sweep of its chunk, four positions per thread per round,
//     keeps key > T, plus the lowest-indexed keys equal to T, numbers them with
//     a block scan and copies their K and V rows (a fixed 16-byte column per
//     thread, two groups of rows alternating between load and store) to page
//     k/P, row k%P of the head's block inside its group page;
//  4. the row's last CTA zero-fills the rows of the head's last page past n,
//     so a decode kernel may read whole tiles.
#include "block_select.cuh"
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

#include <algorithm>

namespace {

using namespace tgk;

constexpr int kThreads = 1024;
constexpr int kRound = 4;  // positions per thread in one round of the kept-token sweep
constexpr int kSmemKeys = 49152;  // rows up to this length keep their keys in shared memory (192 KB)

struct CompactArgs {
  const int32_t *N;
  const float *scores;
  const uint16_t *K, *V;
  const int32_t *head_order, *ntok;
  const int64_t *pt_off;
  const int32_t *pt_ids;
  int64_t pool_pages;
  uint16_t *pool;
  int32_t *kept_idx;
  int32_t *status;
  int H, H_p, G, P, d, Nmax;
  int parts;  // CTAs per row (the even split)
  int prop;   // share the grid's CTAs among the rows in proportion to their retained tokens
  int rows;   // batch * H
};

constexpr int kPropRows = 1024;  // rows that the proportional split handles (one per thread)
constexpr int kMinPart = 2048;   // tokens per CTA at least
constexpr int kSweepDiv = 16;    // one swept position costs about 1/16 of one kept token's copy

// Proportional shares: every row gets one CTA; the others go to the rows in proportion to
// their work, retained tokens plus positions swept, rounded on the running sum (a row's CTAs
// each keep at least kMinPart tokens of its range).  Every
// CTA derives the same shares from ntok and writes its (row, part, parts) to out[0..2], or
// out[0] = -1 past the last share.
__device__ __forceinline__ void prop_share(const CompactArgs &a, int *hist, int *scan, int *out) {
  const int rows = a.rows, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // a row's work: its kept tokens' copies, plus the sweep over all its N positions (about
  // a sixteenth of a kept token's cost per position)
  int nr = 0, cap = 0;
  if (tid < rows) {
    const int Nr = max(0, a.N[tid / a.H]);
    nr = max(0, a.ntok[tid]) + Nr / kSweepDiv;
    cap = max(0, Nr / kMinPart - 1);
  }
  // inclusive prefix of the work over the rows (row order), and the total
  long long cum = nr;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, cum, o);
    if (lane >= o) cum += v;
  }
  long long *wsum = reinterpret_cast<long long *>(hist);  // 32 warp sums (256 bytes)
  if (lane == 31) wsum[warp] = cum;
  __syncthreads();
  long long tot = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) cum += wsum[w];
    tot += wsum[w];
  }
  // the extra CTAs in proportion to the work, rounded on the running sum: row r gets
  // floor(E C_{r+1} / tot) - floor(E C_r / tot), so every CTA of the grid has a share
  const long long extra_all = (long long)gridDim.x - rows;
  const long long hi = tot > 0 ? extra_all * cum / tot : 0ll, lo = tot > 0 ? extra_all * (cum - nr) / tot : 0ll;
  const int pr = tid < rows ? 1 + (int)min((long long)cap, hi - lo) : 0;
  // exclusive prefix of the shares: this CTA's row is the one whose range holds blockIdx.x
  int inc = pr;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) scan[warp] = inc;
  if (tid == 0) out[0] = -1;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += scan[w];
  const int first = before + inc - pr;
  if (tid < rows && (int)blockIdx.x >= first && (int)blockIdx.x < first + pr) {
    out[0] = tid;
    out[1] = (int)blockIdx.x - first;
    out[2] = pr;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) compact_topk_kernel(const CompactArgs a) {
  extern __shared__ uint32_t cache[];  // the row's keys when they fit, else the select's candidate list
  __shared__ int hist[256];
  __shared__ int scan[33];
  __shared__ int sel_scratch[4];
  __shared__ int tok_list[kRound * kThreads];
  __shared__ int rank_scratch[kRound * kThreads / 32 + 1];
  __shared__ int err_flag;

  int row = blockIdx.x / a.parts, part = blockIdx.x % a.parts, parts = a.parts;
  if (a.prop) {
    prop_share(a, hist, scan, sel_scratch);
    if (sel_scratch[0] < 0) return;  // past the last share
    row = sel_scratch[0];
    part = sel_scratch[1];
    parts = sel_scratch[2];
    __syncthreads();  // (hist, scan and sel_scratch are reused below)
  }
  const int b = row / a.H, h = row % a.H;
  const int Nb = a.N[b], n = a.ntok[row];
  if (threadIdx.x == 0) err_flag = 0;
  __syncthreads();
  if (Nb < 0 || Nb > a.Nmax || n < 0 || n > Nb) {
    if (threadIdx.x == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  // position of h in its group
  int pos = -1;
  for (int i = 0; i < a.H; ++i)
    if (a.head_order[i] == h) pos = i;
  if (pos < 0) {
    if (threadIdx.x == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int grp = pos / a.H_p, hpos = pos % a.H_p;
  const int64_t base = a.pt_off[b * a.G + grp];
  const int64_t npages = a.pt_off[b * a.G + grp + 1] - base;
  if ((int64_t)(n + a.P - 1) / a.P > npages) {
    if (threadIdx.x == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  if (n == 0) return;

  const float *srow = a.scores + (size_t)row * a.Nmax;
  const bool cached = a.Nmax <= kSmemKeys;  // the launch sized the cache for Nmax keys
  bool nan_seen = false;
  // the row's scores, eight loads in flight per thread: into the key cache when they fit,
  // else only checked for NaN
  for (int t0 = threadIdx.x; t0 < Nb; t0 += 8 * kThreads) {
    float f[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * kThreads;
      f[u] = t < Nb ? srow[t] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * kThreads;
      if (t < Nb) {
        nan_seen |= is_nan(f[u]);
        if (cached) cache[t] = float_key(f[u]);
      }
    }
  }
  if (nan_seen) err_flag = 1;
  __syncthreads();
  if (err_flag && threadIdx.x == 0 && part == 0) report(a.status, TG_STATUS_NONFINITE);
  auto key_of = [&](int t) -> uint32_t { return cached ? cache[t] : float_key(srow[t]); };

  uint32_t T;
  int need_eq, n_eq;
  // keys read from global memory: once the first digit is chosen, the unused key cache holds
  // the candidates left, and the remaining passes read only those
  block_select_kth<kThreads>(Nb, n, key_of, cached ? nullptr : cache, cached ? 0 : kSmemKeys, hist, sel_scratch, T,
                             need_eq, n_eq);

  const int d16 = a.d / 8;  // 16-byte chunks per row
  // copy layout: rpp rows per pass, chunk c8 / 8 of row r0 + j * rpp for this thread
  const int rpp = kThreads / d16, r0 = (int)threadIdx.x / d16;
  const int c8 = ((int)threadIdx.x % d16) * 8;
  const int pshift = (a.P & (a.P - 1)) == 0 ? __ffs(a.P) - 1 : -1;  // page of a slot by a shift when P is 2^k
  const size_t src_row0 = (size_t)row * a.Nmax;
  const int c_begin = (int)((int64_t)part * Nb / parts), c_end = (int)((int64_t)(part + 1) * Nb / parts);
  // keys kept before this chunk: all of them above T, and the first need_eq equal to T
  // (per-thread counts, four keys in flight, then one block sum)
  int gt_before = 0, eq_before = 0;
  {
    int gl = 0, el = 0;
    for (int c0 = 0; c0 < c_begin; c0 += 4 * kThreads) {
      uint32_t kk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = c0 + u * kThreads + threadIdx.x;
        kk[u] = t < c_begin ? key_of(t) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + u * kThreads + (int)threadIdx.x < c_begin) {
          gl += kk[u] > T;
          el += kk[u] == T;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gl += __shfl_xor_sync(0xffffffffu, gl, o);
      el += __shfl_xor_sync(0xffffffffu, el, o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
      scan[warp] = gl;
      hist[warp] = el;
    }
    __syncthreads();
    for (int w = 0; w < kThreads / 32; ++w) {
      gt_before += scan[w];
      eq_before += hist[w];
    }
    __syncthreads();
  }
  int taken = gt_before + min(eq_before, need_eq), eq_seen = eq_before;
  // rounds of kRound * kThreads positions, position c0 + u * kThreads + thread
  for (int c0 = c_begin; c0 < c_end && taken < n; c0 += kRound * kThreads) {
    bool gt[kRound], eq[kRound], sel[kRound];
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int t = c0 + u * kThreads + threadIdx.x;
      const uint32_t key = t < c_end ? key_of(t) : 0u;
      gt[u] = t < c_end && key > T;
      eq[u] = t < c_end && key == T;
    }
    int eq_rank[kRound], k_in[kRound], eq_total, sel_total;
    block_excl_count_multi<kThreads, kRound>(eq, rank_scratch, eq_rank, eq_total);
#pragma unroll
    for (int u = 0; u < kRound; ++u) sel[u] = gt[u] || (eq[u] && eq_seen + eq_rank[u] < need_eq);
    block_excl_count_multi<kThreads, kRound>(sel, rank_scratch, k_in, sel_total);
#pragma unroll
    for (int u = 0; u < kRound; ++u)
      if (sel[u]) {
        const int t = c0 + u * kThreads + threadIdx.x;
        tok_list[k_in[u]] = t;
        if (a.kept_idx) a.kept_idx[src_row0 + taken + k_in[u]] = t;
      }
    __syncthreads();
    // the round's kept rows: thread (r0, c) copies 16-byte chunk c of rows r0, r0 + rpp,
    // r0 + 2 rpp, ... of K and of V.  Two groups of two rows alternate, so one group's loads
    // are in flight while the other group is stored
    auto load2 = [&](int j0, uint4 (&kv)[2][2], int32_t (&page)[2]) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = r0 + (j0 + u) * rpp;
        page[u] = -2;
        if (r < sel_total) {
          const int k = taken + r;
          page[u] = a.pt_ids[base + (pshift >= 0 ? k >> pshift : k / a.P)];
          const size_t src = (src_row0 + tok_list[r]) * a.d + c8;
          kv[u][0] = *reinterpret_cast<const uint4 *>(a.K + src);
          kv[u][1] = *reinterpret_cast<const uint4 *>(a.V + src);
        }
      }
    };
    auto store2 = [&](int j0, const uint4 (&kv)[2][2], const int32_t (&page)[2]) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (page[u] == -2) continue;
        if (page[u] < 0 || (int64_t)page[u] >= a.pool_pages) {
          report(a.status, TG_STATUS_BAD_PAGE);
          continue;
        }
        const int k = taken + r0 + (j0 + u) * rpp;
        const int slot = pshift >= 0 ? k & (a.P - 1) : k % a.P;
        const size_t dst = (((size_t)page[u] * a.H_p + hpos) * 2 * a.P + slot) * a.d + c8;
        *reinterpret_cast<uint4 *>(a.pool + dst) = kv[u][0];
        *reinterpret_cast<uint4 *>(a.pool + dst + (size_t)a.P * a.d) = kv[u][1];
      }
    };
    if (r0 < rpp && r0 < sel_total) {
      const int J = (sel_total - r0 + rpp - 1) / rpp;  // this thread's rows
      uint4 ka[2][2], kb[2][2];
      int32_t pa[2], pb[2];
      load2(0, ka, pa);
      for (int j = 0;; j += 4) {
        load2(j + 2, kb, pb);
        store2(j, ka, pa);
        if (j + 4 >= J) {
          store2(j + 2, kb, pb);
          break;
        }
        load2(j + 4, ka, pa);
        store2(j + 2, kb, pb);
      }
    }
    taken += sel_total;
    eq_seen += eq_total;
    __syncthreads();
  }

  // zero the rows of the last page past n (K and V blocks)
  const int rem = n % a.P;
  if (rem && part == parts - 1) {
    const int32_t page = a.pt_ids[base + (n - 1) / a.P];
    if (page >= 0 && (int64_t)page < a.pool_pages) {
      const int rows = a.P - rem;
      for (int e = threadIdx.x; e < 2 * rows * d16; e += kThreads) {
        const int kv = e / (rows * d16), r = (e / d16) % rows, c = e % d16;
        const size_t dst = ((((size_t)page * a.H_p + hpos) * 2 + kv) * a.P + rem + r) * a.d + (size_t)c * 8;
        *reinterpret_cast<uint4 *>(a.pool + dst) = make_uint4(0, 0, 0, 0);
      }
    }
  }
}

}  // namespace

extern "C" int tg_compact_topk(tg_stream_t stream, int batch, int H, int H_p, int P, int d, int Nmax,
                               const int32_t *N, const float *scores, const uint16_t *K, const uint16_t *V,
                               const int32_t *head_order, const int32_t *ntok, const int64_t *pt_off,
                               const int32_t *pt_ids, int64_t pool_pages, uint16_t *pool, int32_t *kept_idx,
                               int32_t *dev_status) {
  if (batch < 0 || H <= 0 || H_p <= 0 || P <= 0 || d <= 0 || Nmax <= 0)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: sizes must be positive");
  if (H % H_p) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: H %% H_p != 0");
  if (P % 16 || d % 8 || d > 512) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: need P %% 16 == 0, d %% 8 == 0, d <= 512");
  if (batch == 0) return tgi::ok();
  if (!N || !scores || !K || !V || !head_order || !ntok || !pt_off || !pt_ids || !pool)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: NULL pointer argument");
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(pool)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: K, V and pool must be 16-byte aligned");
  CompactArgs a;
  a.N = N; a.scores = scores; a.K = K; a.V = V; a.head_order = head_order; a.ntok = ntok;
  a.pt_off = pt_off; a.pt_ids = pt_ids; a.pool_pages = pool_pages; a.pool = pool; a.kept_idx = kept_idx;
  a.status = dev_status; a.H = H; a.H_p = H_p; a.G = H / H_p; a.P = P; a.d = d; a.Nmax = Nmax;
  // the keys of a row when they fit, else the select's candidate list (kSmemKeys entries)
  const int smem = (Nmax <= kSmemKeys ? Nmax : kSmemKeys) * (int)sizeof(uint32_t);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(compact_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemKeys * 4);
  if (e == cudaSuccess) {
    // CTAs per row: about two waves of one resident 1024-thread CTA per SM when a row's keys
    // fit in shared memory (each CTA's select is then cheap), one wave when they are read
    // from L2 (every CTA of a row repeats the select); at most 16, and chunks of at least
    // 2048 tokens
    const int rows = batch * H;
    const int waves = Nmax <= kSmemKeys ? 2 : 1;
    int parts = (waves * sms + rows - 1) / rows;
    parts = std::max(1, std::min({parts, 16, (Nmax + 2047) / 2048}));
    a.parts = parts;
    a.rows = rows;
    a.prop = parts > 1 && rows <= kPropRows;
    // proportional shares take exactly the wanted waves (no partial wave at the end)
    const int64_t grid = a.prop ? std::max<int64_t>(rows, (int64_t)waves * sms) : (int64_t)rows * parts;
    if (grid > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: grid too large");
    compact_topk_kernel<<<(unsigned)grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_topk: %s", cudaGetErrorString(e));
  return tgi::ok();
}
