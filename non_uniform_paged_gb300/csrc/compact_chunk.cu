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
//  * only the entering tokens' K/V rows are written into the pages, by a second
//    launch spread over the GPU: a row whose slots are still filling maps chunk
//    position i to slot filled + i, which needs no ranking, so those rows are
//    copied while the other rows rank; a ranking row leaves its (slot, chunk
//    position) list in the workspace for the copy.
// Slot k lives at page k / P, row k % P of the head's block in its group page,
// as in the one-shot compaction; only the order of tokens over the slots
// differs (attention does not depend on it).
#include "block_select.cuh"
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

#include <algorithm>

namespace {

using namespace tgk;

constexpr int kThreads = 1024;
constexpr int kMaxChunk = 8192;        // tokens per chunk (entering-token list in shared memory)
constexpr int kSmemKeys = 40960;       // candidates whose score keys are cached in shared memory (160 KB)
constexpr int kLoadUnroll = 12;        // slot keys each thread has in flight while loading
constexpr int kCopyThreads = 256;      // copy kernel: 8 warps per CTA
constexpr int kCopyTokens = 8;         // tokens a warp copies at once (their K/V vectors in flight)

constexpr int kWarps = kThreads / 32;

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
  int2 *elist;                         // [batch][H][C] (slot, chunk position) of each entering token
  int32_t *ecount;                     // [batch][H] entries of a ranking row
  int32_t *status;
  int H, H_p, G, P, d, C, nmax, chunk_start;
};

__global__ void __launch_bounds__(kThreads, 1) compact_chunk_kernel(const ChunkArgs a) {
  extern __shared__ uint32_t cache[];  // score keys of the candidates when they fit
  __shared__ int scan[33];
  __shared__ int sel_scratch[kWarps + 4];
  // the selects' key list, then the entering chunk positions (ascending)
  __shared__ int work[2 * kMaxChunk];
  int *const incoming = work;
  __shared__ int err_flag;

  // the copy launch that follows may be scheduled now: it copies the filling rows, then
  // waits for this grid before reading the entry lists
  griddep_launch_dependents();
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
  const int filled = min(n, min(Nb, a.chunk_start));  // slots holding a token before this chunk
  int32_t *stok = a.slot_tok + (size_t)row * a.nmax;
  uint32_t *skey = a.slot_key + (size_t)row * a.nmax;
  const float *cs = a.scores + (size_t)row * a.C;
  const int d16 = a.d / 8;

  // candidates: i < filled is slot i (its token and key), i >= filled is chunk position i - filled
  const int m = filled + len;
  const bool append = m <= n;  // the slots are not full yet: every chunk token enters

  const bool cached = !append && m <= kSmemKeys;
  bool nan_seen = false;
  if (cached) {
    // the slot keys: several independent loads in flight per thread
    for (int i0 = tid; i0 < filled; i0 += kLoadUnroll * kThreads) {
      uint32_t v[kLoadUnroll];
#pragma unroll
      for (int u = 0; u < kLoadUnroll; ++u) {
        const int i = i0 + u * kThreads;
        v[u] = i < filled ? __ldcg(skey + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kLoadUnroll; ++u)
        if (i0 + u * kThreads < filled) cache[i0 + u * kThreads] = v[u];
    }
  }
  // the chunk's scores, two per thread in flight
  for (int i0 = tid; i0 < len; i0 += 2 * kThreads) {
    float f[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) f[u] = i0 + u * kThreads < len ? cs[i0 + u * kThreads] : 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (i0 + u * kThreads < len) {
        nan_seen |= is_nan(f[u]);
        if (cached) cache[filled + i0 + u * kThreads] = float_key(f[u]);
      }
  }
  // the head's group page list (checked while the loads above are in flight; nothing has
  // been written yet)
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
    // the selects' key list, with the first digit's 4096 counters in the same memory; the later
    // digits' 1024 counters at the end of it
    uint32_t *const list = reinterpret_cast<uint32_t *>(work);
    int *const hist0 = work, *const hist1 = work + 2 * kMaxChunk - 1024;
    const int cap = 2 * kMaxChunk - 1024;
    int need_hi, n_eq;
    block_select_kth_wide<kThreads>(m, n, hi_of, list, cap, hist0, hist1, sel_scratch, T_hi, need_hi, n_eq);
    // among the keys equal to T_hi, the need_hi lowest tokens (largest ~token) survive; with no
    // tie across the cut every one of them does, and T_lo = 0 keeps them all
    if (n_eq > need_hi) {
      int unused0, unused1;
      block_select_kth_wide<kThreads>(
          m, need_hi, [&](int i) { return hi_of(i) == T_hi ? ~(uint32_t)tok_of(i) : 0u; }, list, cap, hist0, hist1,
          sel_scratch, T_lo, unused0, unused1);
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
    for (int r = tid; r < n_in; r += kThreads) {  // (copied by the copy launch from the row's bounds)
      stok[filled + r] = a.chunk_start + r;
      skey[filled + r] = float_key(cs[r]);
    }
  } else {
    if (tid == 0) a.ecount[row] = n_in;
  }
  if (!append && n_in > 0) {
    int2 *const elist = a.elist + (size_t)row * a.C;
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
        elist[r] = make_int2(s, take);
      }
      r0 += __popc(bal);
    }
  }
  __syncthreads();
}

// The checks compact_chunk_kernel makes on a row (it reports what fails them), and what the
// copy needs of the row: its slot range before this chunk, the chunk's length, its block.
struct CopyRow {
  bool ok, append;
  int filled, len, hpos;
  int64_t base;
};

__device__ CopyRow copy_row(const ChunkArgs &a, int row) {
  CopyRow r{};
  const int b = row / a.H, h = row % a.H;
  const int Nb = a.N[b], n = a.ntok[row];
  r.len = max(0, min(a.C, Nb - a.chunk_start));
  r.ok = Nb >= 0 && n > 0 && n <= Nb && n <= a.nmax && r.len > 0;
  int pos = -1;
  if (r.ok)
    for (int i = 0; i < a.H; ++i)
      if (a.head_order[i] == h) pos = i;
  r.ok = r.ok && pos >= 0;
  if (!r.ok) return r;
  const int grp = pos / a.H_p;
  r.hpos = pos % a.H_p;
  r.base = a.pt_off[b * a.G + grp];
  r.ok = (int64_t)(n + a.P - 1) / a.P <= a.pt_off[b * a.G + grp + 1] - r.base;
  r.filled = min(n, min(Nb, a.chunk_start));
  r.append = r.filled + r.len <= n;
  return r;
}

// The warp copies the K and V rows of up to 32 tokens, one per lane with `in` set: chunk
// position ci to slot `slot`, page `page`; kCopyTokens tokens' vectors in flight per lane.
__device__ __forceinline__ void copy_tokens(const ChunkArgs &a, int row, const CopyRow &r, bool in, int slot,
                                            int ci, int32_t page) {
  const int lane = threadIdx.x & 31;
  const int d16 = a.d / 8, nv = 2 * d16;  // 16-byte vectors of one token's K row then V row
  uint32_t mask = __ballot_sync(0xffffffffu, in);
  while (mask) {
    int src_l[kCopyTokens];
#pragma unroll
    for (int k = 0; k < kCopyTokens; ++k) {
      src_l[k] = mask ? __ffs(mask) - 1 : -1;
      if (mask) mask &= mask - 1;
    }
    for (int v0 = 0; v0 < nv; v0 += 32) {
      const int v = v0 + lane, kv = v / d16, c = v % d16;
      uint4 val[kCopyTokens];
      size_t dst[kCopyTokens];
      bool go[kCopyTokens];
#pragma unroll
      for (int k = 0; k < kCopyTokens; ++k) {
        const int l = src_l[k] < 0 ? 0 : src_l[k];
        const int32_t pg = __shfl_sync(0xffffffffu, page, l);
        const int pos = __shfl_sync(0xffffffffu, ci, l);
        const int sl = __shfl_sync(0xffffffffu, slot, l);
        go[k] = src_l[k] >= 0 && v < nv && pg >= 0 && (int64_t)pg < a.pool_pages;
        if (src_l[k] >= 0 && v < nv && !go[k]) report(a.status, TG_STATUS_BAD_PAGE);
        dst[k] = ((((size_t)pg * a.H_p + r.hpos) * 2 + kv) * a.P + sl % a.P) * a.d + (size_t)c * 8;
        if (go[k]) {
          const size_t src = ((size_t)row * a.C + pos) * a.d + (size_t)c * 8;
          val[k] = __ldcs(reinterpret_cast<const uint4 *>((kv ? a.V : a.K) + src));
        }
      }
#pragma unroll
      for (int k = 0; k < kCopyTokens; ++k)
        if (go[k]) *reinterpret_cast<uint4 *>(a.pool + dst[k]) = val[k];
    }
  }
}

// Copy of the entering tokens' K/V rows, in units of 32 chunk positions of one row, each warp
// taking a contiguous range of units (so its row, and the row's checks, rarely change):
//  1. rows whose slots are still filling: chunk position i to slot filled + i, before waiting
//     for the ranking kernel, so these copies overlap the other rows' ranking;
//  2. the ranking rows, from their (slot, chunk position) lists.
__global__ void __launch_bounds__(kCopyThreads) compact_copy_kernel(const ChunkArgs a, int rows) {
  constexpr int WPC = kCopyThreads / 32;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * WPC + (threadIdx.x >> 5), warps = (int64_t)gridDim.x * WPC;
  const int nblk = (a.C + 31) / 32;
  const int64_t units = (int64_t)rows * nblk;
  const int64_t u0 = warp0 * units / warps, u1 = (warp0 + 1) * units / warps;
  for (int phase = 0; phase < 2; ++phase) {
    if (phase == 1) griddep_wait();  // the ranking rows' lists come from the kernel just before
    int row_seen = -1;
    CopyRow r{};
    for (int64_t u = u0; u < u1; ++u) {
      const int row = (int)(u / nblk), blk = (int)(u % nblk);
      if (row != row_seen) {
        row_seen = row;
        r = copy_row(a, row);
      }
      if (!r.ok || r.append != (phase == 0)) continue;
      const int e = blk * 32 + lane;  // chunk position (phase 0) or list entry (phase 1)
      bool in;
      int slot = 0, ci = 0;
      if (phase == 0) {
        in = e < r.len;
        ci = e;
        slot = r.filled + e;
      } else {
        const int cnt = min(__ldcg(a.ecount + row), a.C);
        in = e < cnt;
        if (in) {
          const int2 en = __ldcg(a.elist + (size_t)row * a.C + e);
          slot = en.x;
          ci = en.y;
          in = slot >= 0 && slot < a.nmax && ci >= 0 && ci < r.len;
        }
      }
      if (!__any_sync(0xffffffffu, in)) continue;
      const int32_t page = in ? __ldcg(a.pt_ids + r.base + slot / a.P) : -1;
      copy_tokens(a, row, r, in, slot, ci, page);
    }
  }
}

}  // namespace

namespace {
// workspace: (slot, chunk position) entries [rows][C] | entry counts [rows]
struct ChunkWs {
  int64_t elist, ecount, total;
};
ChunkWs chunk_ws(int64_t rows, int C) {
  ChunkWs w;
  w.elist = 0;
  w.ecount = tgi::align_up(rows * C * (int64_t)sizeof(int2), 256);
  w.total = tgi::align_up(w.ecount + rows * 4, 256);
  return w;
}
}  // namespace

extern "C" int tg_compact_chunk_workspace(int batch, int H, int C, int64_t *workspace_bytes) {
  if (!workspace_bytes) return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk_workspace: NULL workspace_bytes");
  if (batch < 0 || H <= 0 || C <= 0)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk_workspace: batch=%d H=%d C=%d", batch, H, C);
  *workspace_bytes = chunk_ws((int64_t)batch * H, C).total;
  return tgi::ok();
}

extern "C" int tg_compact_chunk(tg_stream_t stream, int batch, int H, int H_p, int P, int d, int chunk_start, int C,
                                const int32_t *N, const float *scores, const uint16_t *K, const uint16_t *V,
                                const int32_t *head_order, const int32_t *ntok, const int64_t *pt_off,
                                const int32_t *pt_ids, int64_t pool_pages, uint16_t *pool, int32_t *slot_tok,
                                uint32_t *slot_key, int nmax, void *workspace, int64_t workspace_bytes,
                                int32_t *dev_status) {
  if (batch < 0 || H <= 0 || H_p <= 0 || P <= 0 || d <= 0 || C <= 0 || nmax <= 0 || chunk_start < 0)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk: sizes must be positive");
  if (H % H_p) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: H %% H_p != 0");
  if (P % 16 || d % 8 || d > 512) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: need P %% 16 == 0, d %% 8 == 0, d <= 512");
  if (C > kMaxChunk) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: C=%d > %d", C, kMaxChunk);
  if (batch == 0) return tgi::ok();
  if (!N || !scores || !K || !V || !head_order || !ntok || !pt_off || !pt_ids || !pool || !slot_tok || !slot_key ||
      !workspace)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk: NULL pointer argument");
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(pool) |
       reinterpret_cast<uintptr_t>(workspace)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_chunk: K, V, pool and workspace must be 16-byte aligned");
  const int64_t rows = (int64_t)batch * H;
  if (rows > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_chunk: grid too large");
  const ChunkWs wl = chunk_ws(rows, C);
  if (workspace_bytes < wl.total)
    return tgi::fail(TG_ERR_CAPACITY, "tg_compact_chunk: workspace %lld < %lld bytes", (long long)workspace_bytes,
                     (long long)wl.total);
  ChunkArgs a;
  a.N = N; a.scores = scores; a.K = K; a.V = V; a.head_order = head_order; a.ntok = ntok;
  a.pt_off = pt_off; a.pt_ids = pt_ids; a.pool_pages = pool_pages; a.pool = pool;
  a.slot_tok = slot_tok; a.slot_key = slot_key; a.status = dev_status;
  a.elist = reinterpret_cast<int2 *>(static_cast<uint8_t *>(workspace) + wl.elist);
  a.ecount = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + wl.ecount);
  a.H = H; a.H_p = H_p; a.G = H / H_p; a.P = P; a.d = d; a.C = C; a.nmax = nmax; a.chunk_start = chunk_start;
  const size_t smem = (size_t)kSmemKeys * 4;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaFuncSetAttribute(compact_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    compact_chunk_kernel<<<(unsigned)rows, kThreads, smem, st>>>(a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    // the copy over the whole GPU, started early (programmatic dependent launch)
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) {
      constexpr int WPC = kCopyThreads / 32;
      const int64_t units = rows * ((C + 31) / 32);
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>((units + WPC - 1) / WPC, (int64_t)sms * 8)));
      cfg.blockDim = dim3(kCopyThreads);
      cfg.dynamicSmemBytes = 0;
      cfg.stream = st;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, compact_copy_kernel, a, (int)rows);
    }
  }
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_chunk: %s", cudaGetErrorString(e));
  return tgi::ok();
}
