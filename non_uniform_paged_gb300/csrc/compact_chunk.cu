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
// Top(n, s).  Per (request, KV head) row and chunk, the row's first CTA:
//  * while the slots are not full, the chunk's tokens are appended in order;
//  * otherwise the current slots and the chunk's tokens are ranked together by
//    a radix select on the score key and, only when the n-th score is tied
//    across the cut, one on ~token among the keys equal to it -- a total
//    order, so exactly n survive.  The slots whose token dropped out are
//    reused, the lowest freed slot by the lowest entering token;
//  * only the entering tokens' K/V rows are written into the pages.  A row
//    whose slots are still filling shares that copy with three more CTAs.
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
constexpr int kSmemKeys = 40960;       // candidates whose score keys are cached in shared memory (160 KB)
constexpr int kCopyUnroll = 4;         // 16-byte K/V vectors each thread has in flight while copying
constexpr int kRowCtas = 4;            // CTAs per row: the first ranks; the others help copy a filling row

constexpr int kWarps = kThreads / 32;

// Key T of the k-th largest of `count` keys (1 <= k <= count), the number of keys equal to T that
// a top-k takes (need_eq = k - #{key > T}) and the number of keys equal to T (n_eq).  MSB-first
// radix select over 8-bit digits.  After the first pass the keys that share the chosen top digit
// are copied into `list` when at most `cap` of them do, and the remaining passes read only those
// (the first digit of real scores already narrows the candidates to a few percent).  `hist` is
// 256 ints and `scratch` 4 ints of shared memory.
template <typename GetKey>
__device__ void select_kth(int count, int k, GetKey get, uint32_t *list, int cap, int *hist, int *scratch,
                           uint32_t &T, int &need_eq, int &n_eq) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  int k_rem = k, n_list = -1, sel_count = count;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int cnt = n_list < 0 ? count : n_list;
    for (int base = 0; base < cnt; base += kThreads) {
      const int i = base + tid;
      uint32_t dg = 256u;  // no digit
      if (i < cnt) {
        const uint32_t key = n_list < 0 ? get(i) : list[i];
        if ((key & mask) == prefix) dg = (key >> shift) & 255u;
      }
      // lanes of a warp with the same digit add once
      const uint32_t peers = __match_any_sync(0xffffffffu, dg);
      if (dg < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[dg], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255-8l down to 248-8l; scan from the top digit down
      int local[8];
      int sum = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        local[t] = hist[255 - 8 * lane - t];
        sum += local[t];
      }
      int inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const int before = inc - sum;  // keys in digits above this lane's block
      if (before < k_rem && k_rem <= inc) {
        int above = before;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (above + local[t] >= k_rem) {
            scratch[0] = 255 - 8 * lane - t;
            scratch[1] = above;
            scratch[2] = local[t];
            break;
          }
          above += local[t];
        }
      }
      if (lane == 0) scratch[3] = 0;
    }
    __syncthreads();
    const uint32_t digit = (uint32_t)scratch[0];
    k_rem -= scratch[1];
    sel_count = scratch[2];
    prefix |= digit << shift;
    mask |= 255u << shift;
    if (n_list < 0 && shift > 0 && sel_count <= cap) {
      // copy the keys under the new prefix into the list (order does not matter for counts)
      for (int base = 0; base < count; base += kThreads) {
        const int i = base + tid;
        uint32_t key = 0;
        const bool keep = i < count && ((key = get(i)) & mask) == prefix;
        const uint32_t bal = __ballot_sync(0xffffffffu, keep);
        int at = 0;
        if (lane == 0 && bal) at = atomicAdd(&scratch[3], __popc(bal));
        at = __shfl_sync(0xffffffffu, at, 0);
        if (keep) list[at + __popc(bal & ((1u << lane) - 1u))] = key;
      }
      n_list = sel_count;
    }
    __syncthreads();
  }
  T = prefix;
  need_eq = k_rem;
  n_eq = sel_count;
}

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
  // the selects' key list, then: entering chunk positions (ascending) and the slot each takes
  __shared__ int work[2 * kMaxChunk];
  int *const incoming = work, *const slot_of = work + kMaxChunk;
  __shared__ int err_flag;

  // CTA part 0 of a row ranks and copies; parts 1.. copy their share of a row whose slots are
  // still filling (its chunk position i goes to slot filled + i, known without ranking), so
  // such a row's copy is not carried by one SM.  For the other rows they return at once.
  // (all rows' part 0 first, so every ranking CTA starts at once; the helpers fill the rest)
  const int n_rows = gridDim.x / kRowCtas;
  const int row = (int)(blockIdx.x % n_rows), part = (int)(blockIdx.x / n_rows);
  const int b = row / a.H, h = row % a.H, tid = threadIdx.x;
  const int Nb = a.N[b], n = a.ntok[row];
  if (tid == 0) err_flag = 0;
  __syncthreads();
  if (Nb < 0 || n < 0 || n > Nb || n > a.nmax) {
    if (tid == 0 && part == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int len = max(0, min(a.C, Nb - a.chunk_start));
  if (n == 0 || len == 0) return;
  int pos = -1;
  for (int i = 0; i < a.H; ++i)
    if (a.head_order[i] == h) pos = i;
  if (pos < 0) {
    if (tid == 0 && part == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int grp = pos / a.H_p, hpos = pos % a.H_p;
  const int64_t base = a.pt_off[b * a.G + grp];
  const int64_t npages = a.pt_off[b * a.G + grp + 1] - base;
  if ((int64_t)(n + a.P - 1) / a.P > npages) {
    if (tid == 0 && part == 0) report(a.status, TG_STATUS_BAD_INPUT);
    return;
  }
  const int filled = min(n, min(Nb, a.chunk_start));  // slots holding a token before this chunk
  int32_t *stok = a.slot_tok + (size_t)row * a.nmax;
  uint32_t *skey = a.slot_key + (size_t)row * a.nmax;
  const float *cs = a.scores + (size_t)row * a.C;
  const int d16 = a.d / 8;

  // candidates: i < filled is slot i (its token and key), i >= filled is chunk position i - filled
  const int m = filled + len;
  const bool append = m <= n;  // the slots are not full yet: every chunk token enters
  // this CTA's share of the chunk positions of a filling row
  const int share_lo = (int)((int64_t)part * len / kRowCtas), share_hi = (int)((int64_t)(part + 1) * len / kRowCtas);
  if (part > 0) {
    if (!append) return;
    const int nv = (share_hi - share_lo) * d16;
    for (int e0 = tid; e0 < nv; e0 += kCopyUnroll * kThreads) {
      uint4 kv[kCopyUnroll][2];
      int32_t page[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int e = e0 + u * kThreads;
        page[u] = -2;
        if (e < nv) {
          const int i = share_lo + e / d16, c = e % d16;
          page[u] = __ldcg(a.pt_ids + base + (filled + i) / a.P);
          const size_t src = ((size_t)row * a.C + i) * a.d + (size_t)c * 8;
          kv[u][0] = __ldcs(reinterpret_cast<const uint4 *>(a.K + src));
          kv[u][1] = __ldcs(reinterpret_cast<const uint4 *>(a.V + src));
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        if (page[u] == -2) continue;
        if (page[u] < 0 || (int64_t)page[u] >= a.pool_pages) {
          report(a.status, TG_STATUS_BAD_PAGE);
          continue;
        }
        const int e = e0 + u * kThreads, s = filled + share_lo + e / d16, c = e % d16;
        const size_t dst = ((((size_t)page[u] * a.H_p + hpos) * 2) * a.P + (s % a.P)) * a.d + (size_t)c * 8;
        *reinterpret_cast<uint4 *>(a.pool + dst) = kv[u][0];
        *reinterpret_cast<uint4 *>(a.pool + dst + (size_t)a.P * a.d) = kv[u][1];
      }
    }
    return;
  }

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

  const bool cached = !append && m <= kSmemKeys;
  bool nan_seen = false;
  if (cached) {
    // the slot keys: several independent loads in flight per thread
    for (int i0 = tid; i0 < filled; i0 += kCopyUnroll * kThreads) {
      uint32_t v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = i0 + u * kThreads;
        v[u] = i < filled ? __ldcg(skey + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (i0 + u * kThreads < filled) cache[i0 + u * kThreads] = v[u];
    }
  }
  for (int i = tid; i < len; i += kThreads) {
    const float f = cs[i];
    nan_seen |= is_nan(f);
    if (cached) cache[filled + i] = float_key(f);
  }
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
  if (!append) {
    uint32_t *const list = reinterpret_cast<uint32_t *>(work);
    int need_hi, n_eq;
    select_kth(m, n, hi_of, list, 2 * kMaxChunk, hist, sel_scratch, T_hi, need_hi, n_eq);
    // among the keys equal to T_hi, the need_hi lowest tokens (largest ~token) survive; with no
    // tie across the cut every one of them does, and T_lo = 0 keeps them all
    if (n_eq > need_hi) {
      int unused0, unused1;
      select_kth(m, need_hi, [&](int i) { return hi_of(i) == T_hi ? ~(uint32_t)tok_of(i) : 0u; }, list,
                 2 * kMaxChunk, hist, sel_scratch, T_lo, unused0, unused1);
    }
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
  // the r-th freed slot takes incoming[r].  Warp w scans the slots [w*seg, (w+1)*seg): it counts
  // its freed slots, a scan over the warps gives its first rank, and a second sweep assigns.  A
  // lane writes only its own slot, whose old state it has just read.
  if (append) {
    // every chunk position enters, in order, into the empty slots filled, filled + 1, ...
    for (int r = tid; r < n_in; r += kThreads) {
      stok[filled + r] = a.chunk_start + r;
      skey[filled + r] = float_key(cs[r]);
      slot_of[r] = filled + r;
    }
  } else if (n_in > 0) {
    const int lane = tid & 31, warp = tid >> 5;
    const int seg = (((n + kWarps - 1) / kWarps) + 31) & ~31;
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    auto is_freed = [&](int s) { return s < hi && (s >= filled || !survives(s)); };
    int cnt = 0;
    for (int s0 = lo; s0 < hi; s0 += 32) cnt += __popc(__ballot_sync(0xffffffffu, is_freed(s0 + lane)));
    if (lane == 0) scan[warp] = cnt;
    __syncthreads();
    if (warp == 0) {
      const int v = scan[lane];
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      scan[lane] = inc - v;
    }
    __syncthreads();
    int r0 = scan[warp];
    for (int s0 = lo; s0 < hi && r0 < n_in; s0 += 32) {
      const int s = s0 + lane;
      const bool fr = is_freed(s);
      const uint32_t bal = __ballot_sync(0xffffffffu, fr);
      const int r = r0 + __popc(bal & ((1u << lane) - 1u));
      if (fr && r < n_in) {
        const int take = incoming[r];
        stok[s] = a.chunk_start + take;
        skey[s] = cached ? cache[filled + take] : float_key(cs[take]);
        slot_of[r] = s;
      }
      r0 += __popc(bal);
    }
  }
  __syncthreads();
  // copy the entering tokens' K and V rows into their slots (16-byte vectors); the page id and
  // the K/V vectors of kCopyUnroll elements are loaded before any is stored
  // (every entering position found a slot: n_in <= freed); of a filling row, only this CTA's share
  const int n_vec = (append ? share_hi : min(n_in, n)) * d16;
  for (int e0 = tid; e0 < n_vec; e0 += kCopyUnroll * kThreads) {
    uint4 kv[kCopyUnroll][2];
    int32_t page[kCopyUnroll];
    int slot[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int e = e0 + u * kThreads;
      slot[u] = -1;
      if (e < n_vec) {
        const int r = e / d16, c = e % d16;
        slot[u] = slot_of[r];
        page[u] = __ldcg(a.pt_ids + base + slot[u] / a.P);
        const size_t src = ((size_t)row * a.C + incoming[r]) * a.d + (size_t)c * 8;
        kv[u][0] = __ldcs(reinterpret_cast<const uint4 *>(a.K + src));
        kv[u][1] = __ldcs(reinterpret_cast<const uint4 *>(a.V + src));
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      if (slot[u] < 0) continue;
      if (page[u] < 0 || (int64_t)page[u] >= a.pool_pages) {
        report(a.status, TG_STATUS_BAD_PAGE);
        continue;
      }
      const int c = (e0 + u * kThreads) % d16;
      const size_t dst = ((((size_t)page[u] * a.H_p + hpos) * 2) * a.P + (slot[u] % a.P)) * a.d + (size_t)c * 8;
      *reinterpret_cast<uint4 *>(a.pool + dst) = kv[u][0];
      *reinterpret_cast<uint4 *>(a.pool + dst + (size_t)a.P * a.d) = kv[u][1];
    }
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
    if (rows * kRowCtas > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: grid too large");
    compact_chunk_kernel<<<(unsigned)(rows * kRowCtas), kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_chunk: %s", cudaGetErrorString(e));
  return tgi::ok();
}
