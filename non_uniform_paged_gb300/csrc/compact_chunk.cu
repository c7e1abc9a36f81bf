// Chunk-incremental retention and compaction, fused into chunked prefill.
//
// Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
// Multi-turn LLM Serving" (paper-review page), 3.1 Budget Reservation (the
// compression runs inside chunked prefill: as each chunk's KV is computed, the
// top-k selection I_{l,h} = Top(ceil(B_{l,h} N), s_{l,h}) is applied) and 4
// ("Compression Fusion into Prefill").
//
// A head's n = ceil(B N) slots are reserved when the request is admitted (N is
// the prompt length).  After each chunk the slots hold the best n tokens seen
// so far, by (score descending, token ascending); since a token's score is
// fixed once its chunk is computed, after the last chunk they hold exactly
// Top(n, s).  One CTA per (request, KV head) row and chunk:
//  * while the slots are not full, the chunk's tokens are appended in order;
//  * otherwise the current slots and the chunk's tokens are ranked together by
//    two radix selects (score key, then ~token among the keys equal to the
//    n-th score) -- a total order, so exactly n survive.  The slots whose token
//    dropped out are reused, the lowest freed slot by the lowest entering token,
//    and only the entering tokens' K/V rows are written into the pages.
// Slot k lives at page k / P, row k % P of the head's block in its group page,
// as in the one-shot compaction; only the order of tokens over the slots
// differs (attention does not depend on it).
#include "block_select.cuh"
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

namespace {

using namespace tgk;

constexpr int kThreads = 1024;
constexpr int kMaxChunk = 8192;        // tokens per chunk (entering-token list in shared memory)
constexpr int kSmemKeys = 45056;       // candidates whose score keys are cached in shared memory (176 KB)

struct ChunkArgs {
  const int32_t *N;
  const float *scores;                 // [batch][H][C]
  const uint16_t *K, *V;               // [batch][H][C][d]
  const int32_t *head_order, *ntok;
  const int64_t *pt_off;
  const int32_t *pt_ids;
  int64_t pool_pages;
  uint16_t *pool;
  int32_t *slot_tok;                   // [batch][H][nmax]
  uint32_t *slot_key;                  // [batch][H][nmax]
  int32_t *status;
  int H, H_p, G, P, d, C, nmax, chunk_start;
};

__global__ void __launch_bounds__(kThreads, 1) compact_chunk_kernel(const ChunkArgs a) {
  extern __shared__ uint32_t cache[];  // score keys of the candidates when they fit
  __shared__ int hist[256];
  __shared__ int scan[33];
  __shared__ int sel_scratch[4];
  __shared__ int incoming[kMaxChunk];  // entering chunk positions, ascending
  __shared__ int err_flag;

  const int row = blockIdx.x, b = row / a.H, h = row % a.H, tid = threadIdx.x;
  const int Nb = a.N[b], n = a.ntok[row];
  if (tid == 0) err_flag = 0;
  __syncthreads();
  if (Nb < 0 || n < 0 || n > Nb || n > a.nmax) {
    if (tid == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int len = max(0, min(a.C, Nb - a.chunk_start));
  if (n == 0 || len == 0) return;
  int pos = -1;
  for (int i = 0; i < a.H; ++i)
    if (a.head_order[i] == h) pos = i;
  if (pos < 0) {
    if (tid == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int grp = pos / a.H_p, hpos = pos % a.H_p;
  const int64_t base = a.pt_off[b * a.G + grp];
  const int64_t npages = a.pt_off[b * a.G + grp + 1] - base;
  if ((int64_t)(n + a.P - 1) / a.P > npages) {
    if (tid == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int filled = min(n, min(Nb, a.chunk_start));  // slots holding a token before this chunk
  int32_t *stok = a.slot_tok + (size_t)row * a.nmax;
  uint32_t *skey = a.slot_key + (size_t)row * a.nmax;
  const float *cs = a.scores + (size_t)row * a.C;
  const int d16 = a.d / 8;

  // the first chunk zeroes the rows of the head's last page past n (decode reads whole tiles)
  if (a.chunk_start == 0 && n % a.P) {
    const int rem = n % a.P, rows = a.P - rem;
    const int32_t page = a.pt_ids[base + (n - 1) / a.P];
    if (page >= 0 && (int64_t)page < a.pool_pages)
      for (int e = tid; e < 2 * rows * d16; e += kThreads) {
        const int kv = e / (rows * d16), r = (e / d16) % rows, c = e % d16;
        const size_t dst = ((((size_t)page * a.H_p + hpos) * 2 + kv) * a.P + rem + r) * a.d + (size_t)c * 8;
        *reinterpret_cast<uint4 *>(a.pool + dst) = make_uint4(0, 0, 0, 0);
      }
  }

  // candidates: i < filled is slot i (its token and key), i >= filled is chunk position i - filled
  const int m = filled + len;
  const bool cached = m <= kSmemKeys;
  bool nan_seen = false;
  if (cached)
    for (int i = tid; i < m; i += kThreads) {
      if (i < filled) {
        cache[i] = skey[i];
      } else {
        const float f = cs[i - filled];
        nan_seen |= is_nan(f);
        cache[i] = float_key(f);
      }
    }
  else
    for (int i = tid; i < len; i += kThreads) nan_seen |= is_nan(cs[i]);
  if (nan_seen) err_flag = 1;
  __syncthreads();
  if (err_flag && tid == 0) report(a.status, TG_STATUS_NONFINITE);
  auto hi_of = [&](int i) -> uint32_t {
    return cached ? cache[i] : (i < filled ? skey[i] : float_key(cs[i - filled]));
  };
  auto tok_of = [&](int i) -> int { return i < filled ? stok[i] : a.chunk_start + (i - filled); };

  // which chunk positions enter, and which slots they take
  int n_in = 0;
  uint32_t T_hi = 0u, T_lo = 0u;
  const bool append = m <= n;  // the slots are not full yet: every chunk token enters
  if (!append) {
    int need_hi;
    block_radix_select<kThreads>(m, n, hi_of, hist, sel_scratch, T_hi, need_hi);
    // among the keys equal to T_hi, the need_hi lowest tokens (largest ~token) survive
    int unused;
    block_radix_select<kThreads>(m, need_hi, [&](int i) { return hi_of(i) == T_hi ? ~(uint32_t)tok_of(i) : 0u; },
                                 hist, sel_scratch, T_lo, unused);
  }
  auto survives = [&](int i) {
    if (append) return true;
    const uint32_t hk = hi_of(i);
    return hk > T_hi || (hk == T_hi && ~(uint32_t)tok_of(i) >= T_lo);
  };
  for (int c0 = 0; c0 < len; c0 += kThreads) {  // entering chunk positions, ascending
    const int i = c0 + tid;
    const bool in = i < len && survives(filled + i);
    int total;
    const int r = n_in + block_excl_count<kThreads>(in, scan, total);
    if (in) incoming[r] = i;
    n_in += total;
  }
  __syncthreads();
  // freed slots in ascending order: dropped current slots, then the empty slots filled..n-1;
  // the r-th freed slot takes incoming[r]
  int freed = 0;
  for (int s0 = 0; s0 < n && freed < n_in; s0 += kThreads) {
    const int s = s0 + tid;
    const bool fr = s < n && (s >= filled || !survives(s));
    int total;
    const int r = freed + block_excl_count<kThreads>(fr, scan, total);
    int take = -1;
    if (fr && r < n_in) take = incoming[r];
    freed += total;
    __syncthreads();  // every thread has read the old slot state of this block of slots
    if (take >= 0) {
      stok[s] = a.chunk_start + take;
      skey[s] = float_key(cs[take]);
      incoming[r] = -1 - s;  // remember the slot for the copy below
    }
  }
  __syncthreads();
  // copy the entering tokens' K and V rows into their slots (16-byte vectors)
  for (int e = tid; e < n_in * d16; e += kThreads) {
    const int r = e / d16, c = e % d16;
    const int s = -1 - incoming[r];
    if (s < 0) continue;  // (cannot happen: every entering token found a slot)
    const int i = stok[s] - a.chunk_start;
    const int32_t page = a.pt_ids[base + s / a.P];
    if (page < 0 || (int64_t)page >= a.pool_pages) {
      report(a.status, TG_STATUS_BAD_PAGE);
      continue;
    }
    const size_t dst = ((((size_t)page * a.H_p + hpos) * 2) * a.P + (s % a.P)) * a.d + (size_t)c * 8;
    const size_t src = ((size_t)row * a.C + i) * a.d + (size_t)c * 8;
    *reinterpret_cast<uint4 *>(a.pool + dst) = *reinterpret_cast<const uint4 *>(a.K + src);
    *reinterpret_cast<uint4 *>(a.pool + dst + (size_t)a.P * a.d) = *reinterpret_cast<const uint4 *>(a.V + src);
  }
}

}  // namespace

extern "C" int tg_compact_chunk(tg_stream_t stream, int batch, int H, int H_p, int P, int d, int chunk_start, int C,
                                const int32_t *N, const float *scores, const uint16_t *K, const uint16_t *V,
                                const int32_t *head_order, const int32_t *ntok, const int64_t *pt_off,
                                const int32_t *pt_ids, int64_t pool_pages, uint16_t *pool, int32_t *slot_tok,
                                uint32_t *slot_key, int nmax, int32_t *dev_status) {
  if (batch < 0 || H <= 0 || H_p <= 0 || P <= 0 || d <= 0 || C <= 0 || nmax <= 0 || chunk_start < 0)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk: sizes must be positive");
  if (H % H_p) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: H %% H_p != 0");
  if (P % 16 || d % 8 || d > 512) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: need P %% 16 == 0, d %% 8 == 0, d <= 512");
  if (C > kMaxChunk) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: C=%d > %d", C, kMaxChunk);
  if (batch == 0) return tgi::ok();
  if (!N || !scores || !K || !V || !head_order || !ntok || !pt_off || !pt_ids || !pool || !slot_tok || !slot_key)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk: NULL pointer argument");
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(pool)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk: K, V and pool must be 16-byte aligned");
  ChunkArgs a;
  a.N = N; a.scores = scores; a.K = K; a.V = V; a.head_order = head_order; a.ntok = ntok;
  a.pt_off = pt_off; a.pt_ids = pt_ids; a.pool_pages = pool_pages; a.pool = pool;
  a.slot_tok = slot_tok; a.slot_key = slot_key; a.status = dev_status;
  a.H = H; a.H_p = H_p; a.G = H / H_p; a.P = P; a.d = d; a.C = C; a.nmax = nmax; a.chunk_start = chunk_start;
  const size_t smem = (size_t)kSmemKeys * 4;
  cudaError_t e = cudaFuncSetAttribute(compact_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    const int64_t rows = (int64_t)batch * H;
    if (rows > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: grid too large");
    compact_chunk_kernel<<<(unsigned)rows, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_chunk: %s", cudaGetErrorString(e));
  return tgi::ok();
}
