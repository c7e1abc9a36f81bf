// Token top-k retention and compaction into the ragged group pages.
//
// Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
// Multi-turn LLM Serving" (paper-review page), 3.1 Budget Reservation
// (I_{l,h} = Top(ceil(B_{l,h} N), s_{l,h}), done as each prefill chunk's KV is
// ready) and 3.2 Ragged Paging (each H_p-head group writes into its own pages
// of H_p x 2 x P x d elements).
//
// Two kernels per layer.  Positions of a row (request, KV head) are cut into blocks of
// kBlk = 1024.
//  select  one thread-block cluster of C CTAs per row.  CTA j brings its chunk of the row
//          (a range of whole blocks) into shared memory once, by bulk copies, turns the
//          float32 scores into order-preserving keys in place and checks them for NaN.  The
//          exact n-th largest key T of the whole row comes from an MSB-first radix select
//          with digits of 12, 10 and 10 bits: each CTA counts its own chunk's digits, and
//          after a cluster barrier every CTA adds up the cluster's counts through
//          distributed shared memory (first 256 sums of adjacent digits, then the digits
//          inside the chosen sum), so all of them take the same digit; the sums over the
//          lower ranks give each CTA the keys above T and equal to T before its chunk.
//          After the first digit each block keeps only its keys under that digit (moved to
//          its front), and the later passes read only those.  The cluster then writes T,
//          need_eq (the keys equal to T that a top-n takes: the lowest-indexed ones) and,
//          for every block, the keys > T and == T before it, to the workspace.  The row's
//          scores are read from memory once.
//  copy    1024-thread CTAs take shares of the rows' blocks, in proportion to the rows'
//          work (retained tokens plus positions swept).  A CTA reads the counts before its
//          first block from the workspace and sweeps its blocks in ascending order, four
//          positions per thread per round: it keeps key > T, plus keys equal to T while
//          fewer than need_eq of them came before, numbers them with a block scan and
//          copies their K and V rows (a fixed 16-byte column per thread, two groups of
//          rows alternating between load and store) to page k/P, row k%P of the head's
//          block inside its group page.  The row's last CTA zero-fills the rows of the
//          head's last page past n, so a decode kernel may read whole tiles.  It is a
//          programmatic dependent of select, which lets it launch as select's CTAs finish.
#include "block_select.cuh"
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

#include <algorithm>

namespace {

using namespace tgk;

constexpr int kBlk = 1024;  // positions per block of the prefix-count table

// ---------------------------------------------------------------- select --
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelKeys = 22528;  // keys of a chunk held in shared memory (88 KB, two CTAs per SM); the rest are re-read from L2
constexpr int kSelBlocks = kSelKeys / kBlk;  // blocks held in shared memory
constexpr int kPiece = 4096;                 // keys per bulk copy (16 KB)
constexpr int kPieces = (kSelKeys + kPiece - 1) / kPiece;
constexpr int kBits0 = 12, kBits1 = 10;      // digit widths: 12, 10, 10 bits from the top
constexpr int kBins0 = 1 << kBits0, kBins1 = 1 << kBits1;
constexpr int kMaxCluster = 8;
constexpr int kWsHead = 4;  // workspace row: T, need_eq, 2 unused, then (keys > T, keys == T) before each block
constexpr uint64_t kCopyWaitNs = 2000000000ull;  // give up a copy wait after 2 s
static_assert(kSelBlocks < 32 && kSelKeys % kBlk == 0 && kBins1 == 2 * kSelThreads, "select layout");

struct SelectArgs {
  const int32_t *N;
  const float *scores;
  const int32_t *ntok;
  int32_t *ws;
  int32_t *status;
  int64_t ws_row;  // ints per workspace row
  int H, Nmax, C;  // C: CTAs per cluster (one cluster per row)
  int vec;         // score rows start 16-byte aligned: chunks arrive by bulk copies
};

__global__ void __launch_bounds__(kSelThreads, 2) compact_select_kernel(const SelectArgs a) {
  extern __shared__ __align__(128) uint32_t keys[];  // the first kSelKeys keys of this CTA's chunk
  __shared__ __align__(16) int hist_a[kBins0];        // digit counts of passes 0 and 2
  __shared__ __align__(16) int hist_b[kBins1];        // of pass 1, later the per-block counts
  __shared__ int sup_buf[2][256];           // this CTA's super-digit counts, alternating between passes
  __shared__ int wtot[2][kSelWarps];
  __shared__ int pick[4];
  __shared__ int nc[kSelBlocks], gt0[kSelBlocks], coff[kSelBlocks + 1];  // candidates per cached block
  __shared__ __align__(8) uint64_t bars[kPieces];
  __shared__ int err;
  int(&bcnt)[2][kSelThreads] = *reinterpret_cast<int(*)[2][kSelThreads]>(hist_b);

  const int C = a.C, rank = (int)cluster_ctarank(), row = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Nb = a.N[row / a.H], n = a.ntok[row];
  // a row with nothing to select (the copy kernel reports bad sizes); every CTA of the
  // cluster reads the same values, so the whole cluster leaves before its first barrier
  if (Nb < 0 || Nb > a.Nmax || n <= 0 || n > Nb) return;
  const int nbr = (Nb + kBlk - 1) / kBlk;
  const int blk0 = (int)((int64_t)rank * nbr / C), blk1 = (int)((int64_t)(rank + 1) * nbr / C);
  const int p0 = blk0 * kBlk, cnt = max(0, min(blk1 * kBlk, Nb) - p0);
  const int cached = min(cnt, kSelKeys), ncb = (cached + kBlk - 1) / kBlk;
  const float *src = a.scores + (size_t)row * a.Nmax + p0;
  const int nbulk = a.vec ? (cached & ~3) : 0;  // keys that arrive by bulk copies
  const int npieces = (nbulk + kPiece - 1) / kPiece;

  if (tid == 0) {
    err = 0;
    for (int i = 0; i < npieces; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  for (int i = tid; i < kBins0; i += kSelThreads) hist_a[i] = 0;
  for (int i = tid; i < kBins1; i += kSelThreads) hist_b[i] = 0;
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < npieces; ++i) {
      const int k0 = i * kPiece, nk = min(kPiece, nbulk - k0);
      mbar_arrive_expect_tx(&bars[i], (uint32_t)nk * 4u);
      bulk_load(keys + k0, src + k0, (uint32_t)nk * 4u, &bars[i]);
    }

  // first digit (the top 12 bits: sign, exponent and three mantissa bits, which spread real
  // scores over many counters) of every key, counted while the chunk arrives; NaN checked
  constexpr int kShift0 = 32 - kBits0;
  bool nan_seen = false;
  // keys past the bulk copies: the cached tail, then the part of the chunk read from L2
  for (int i = nbulk + tid; i < cached; i += kSelThreads) {
    const uint32_t k = float_key(src[i]);
    nan_seen |= is_nan_key(k);
    keys[i] = k;
    atomicAdd(&hist_a[k >> kShift0], 1);
  }
  for (int base = cached; base < cnt; base += 4 * kSelThreads) {
    uint32_t kk[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * kSelThreads + tid;
      kk[u] = i < cnt ? float_key(src[i]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (base + u * kSelThreads + tid < cnt) {
        nan_seen |= is_nan_key(kk[u]);
        atomicAdd(&hist_a[kk[u] >> kShift0], 1);
      }
  }
  // the bulk-copied pieces, turned into keys in place as each one lands
  bool timed_out = false;
  for (int i = 0; i < npieces; ++i) {
    if (!mbar_wait(&bars[i], 0, kCopyWaitNs)) timed_out = true;
    const int g0 = i * kPiece / 4, ng = min(kPiece, nbulk - i * kPiece) / 4;
    uint4 *k4 = reinterpret_cast<uint4 *>(keys);
    for (int g = tid; g < ng; g += kSelThreads) {
      uint4 k = k4[g0 + g];
      k.x = float_key(__uint_as_float(k.x));
      k.y = float_key(__uint_as_float(k.y));
      k.z = float_key(__uint_as_float(k.z));
      k.w = float_key(__uint_as_float(k.w));
      nan_seen |= is_nan_key(k.x) | is_nan_key(k.y) | is_nan_key(k.z) | is_nan_key(k.w);
      k4[g0 + g] = k;
      atomicAdd(&hist_a[k.x >> kShift0], 1);
      atomicAdd(&hist_a[k.y >> kShift0], 1);
      atomicAdd(&hist_a[k.z >> kShift0], 1);
      atomicAdd(&hist_a[k.w >> kShift0], 1);
    }
  }
  if (nan_seen) atomicOr(&err, 1);
  if (timed_out) atomicOr(&err, 2);
  __syncthreads();
  if (tid == 0 && (err & 1)) report(a.status, TG_STATUS_NONFINITE);
  if (tid == 0 && (err & 2)) report(a.status, TG_STATUS_TIMEOUT);

  uint32_t prefix = 0, mask = 0;
  int k_rem = n, gt_lo = 0, eq_lo = 0;
  // One pass's digit over the cluster, in two steps that read only what every CTA wrote
  // before the cluster barrier: its 256 super-digit counts (sums of S = bins/256 adjacent
  // digits), and then, inside the chosen super-digit, its S digit counts.  Each step adds up
  // the counts over the cluster and over the lower ranks and scans from the top down for the
  // one that holds the k_rem-th key.
  auto reduce_pick = [&](int *h, int bins, int shift, int bits, int pass) {
    const int S = bins / 256;
    int *sup = sup_buf[pass & 1];  // (the other CTAs read the other buffer until the previous barrier)
    __syncthreads();               // this CTA's counts of the pass are complete
    if (tid < 256) {
      int t = 0;
      for (int i = 0; i < S; i += 4) {
        const int4 x = *reinterpret_cast<const int4 *>(&h[tid * S + i]);
        t += x.x + x.y + x.z + x.w;
      }
      sup[tid] = t;
    }
    cluster_arrive();  // also orders this CTA's own threads
    cluster_wait();
    int s = 0, l = 0;
    if (tid < 256) {
      const uint32_t addr = smem_addr(&sup[255 - tid]);
      int v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) v[r] = r == rank ? sup[255 - tid] : ld_cluster_s32(cluster_map(addr, (uint32_t)r));
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) {
          s += v[r];
          if (r < rank) l += v[r];
        }
    }
    int is = s, il = l;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, is, o), y = __shfl_up_sync(0xffffffffu, il, o);
      if (lane >= o) {
        is += x;
        il += y;
      }
    }
    if (tid < 256 && lane == 31) {
      wtot[0][warp] = is;
      wtot[1][warp] = il;
    }
    if (tid == 0) pick[0] = pick[1] = pick[2] = pick[3] = 0;  // (in range whatever the counts)
    __syncthreads();
    if (tid < 256) {
      int bs = 0, bl = 0;
      for (int w = 0; w < warp; ++w) {
        bs += wtot[0][w];
        bl += wtot[1][w];
      }
      const int above = bs + is - s;  // keys in the super-digits above this one
      if (above < k_rem && k_rem <= above + s) {
        pick[0] = 255 - tid;
        pick[1] = above;
        pick[2] = bl + il - l;  // the lower ranks' keys in the super-digits above
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane u (< S) holds digit sd*S + S-1-u of the chosen super-digit sd
      const int sd = pick[0], above0 = pick[1], above_l0 = pick[2];
      int s2 = 0, l2 = 0;
      if (lane < S) {
        const int dg = sd * S + S - 1 - lane;
        const uint32_t addr = smem_addr(&h[dg]);
        int v[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < C) v[r] = r == rank ? h[dg] : ld_cluster_s32(cluster_map(addr, (uint32_t)r));
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < C) {
            s2 += v[r];
            if (r < rank) l2 += v[r];
          }
      }
      int is2 = s2, il2 = l2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, is2, o), y = __shfl_up_sync(0xffffffffu, il2, o);
        if (lane >= o) {
          is2 += x;
          il2 += y;
        }
      }
      const int above = above0 + is2 - s2;
      __syncwarp();
      if (lane < S && above < k_rem && k_rem <= above + s2) {
        pick[0] = sd * S + S - 1 - lane;
        pick[1] = above;
        pick[2] = above_l0 + il2 - l2;
        pick[3] = l2;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)pick[0] << shift;
    mask |= ((1u << bits) - 1u) << shift;
    k_rem -= pick[1];
    gt_lo += pick[2];
    eq_lo = pick[3];
  };
  reduce_pick(hist_a, kBins0, kShift0, kBits0, 0);

  // Candidates: a warp takes one cached block, half a block at a time into registers (16
  // keys a lane), counts its keys above the chosen first digit (all of them > T) and writes
  // those with that digit to the front of the block, over keys already read (their order
  // inside the block does not matter to any count).
  const uint32_t d0 = prefix >> kShift0;
  for (int j = warp; j < ncb; j += kSelWarps) {
    const int q0 = j * kBlk, len = min(kBlk, cached - q0);
    int m = 0, g = 0;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int h0 = half * (kBlk / 2);
      uint32_t kv[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = h0 + 4 * (lane + 32 * u);
        if (i + 3 < len) {
          const uint4 x = *reinterpret_cast<const uint4 *>(&keys[q0 + i]);
          kv[4 * u] = x.x; kv[4 * u + 1] = x.y; kv[4 * u + 2] = x.z; kv[4 * u + 3] = x.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) kv[4 * u + e] = i + e < len ? keys[q0 + i + e] : 0u;
        }
      }
      int mh = 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const bool v = h0 + 4 * (lane + 32 * (u / 4)) + (u % 4) < len;
        mh += v && (kv[u] >> kShift0) == d0;
        g += v && (kv[u] >> kShift0) > d0;
      }
      int inc = mh;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += x;
      }
      __syncwarp();  // every lane holds its keys before any is overwritten
      int at = q0 + m + inc - mh;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const bool v = h0 + 4 * (lane + 32 * (u / 4)) + (u % 4) < len;
        if (v && (kv[u] >> kShift0) == d0) keys[at++] = kv[u];
      }
      m += __shfl_sync(0xffffffffu, inc, 31);
      __syncwarp();
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if (lane == 0) {
      nc[j] = m;
      gt0[j] = g;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // start of each block's candidates in one flat numbering
    const int v = lane < ncb ? nc[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    if (lane == 0) coff[0] = 0;
    if (lane < kSelBlocks) coff[lane + 1] = inc;
  }
  __syncthreads();
  const int ncand = coff[ncb];

  // digits 2 and 3 (10 bits each) over the candidates, and over the keys past the cache
  for (int p = 1; p < 3; ++p) {
    const int shift = kShift0 - kBits1 * p;
    int *h = p == 1 ? hist_b : hist_a;
    if (p == 2) {
      // (the other CTAs last read this buffer before they arrived at the previous barrier)
      for (int i = tid; i < kBins1; i += kSelThreads) h[i] = 0;
      __syncthreads();
    }
    int j = 0;
    for (int i = tid; i < ncand; i += kSelThreads) {
      while (coff[j + 1] <= i) ++j;
      const uint32_t k = keys[j * kBlk + i - coff[j]];
      if ((k & mask) == prefix) atomicAdd(&h[(k >> shift) & (kBins1 - 1)], 1);
    }
    for (int base = cached; base < cnt; base += 4 * kSelThreads) {
      uint32_t kk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * kSelThreads + tid;
        kk[u] = i < cnt ? float_key(src[i]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (base + u * kSelThreads + tid < cnt && (kk[u] & mask) == prefix)
          atomicAdd(&h[(kk[u] >> shift) & (kBins1 - 1)], 1);
    }
    reduce_pick(h, kBins1, shift, kBits1, p);
  }
  cluster_arrive_relaxed();  // done reading the other CTAs' histograms

  // per block of the chunk: keys > T and == T before it (a warp counts one block: a cached
  // block from its candidates and its count above the first digit, another from L2; groups of
  // kSelThreads blocks are scanned one after another).  The counts go where the pass-1
  // digits were, which no other CTA reads after the last barrier.
  const uint32_t T = prefix;
  int32_t *wrow = a.ws + (size_t)row * a.ws_row;
  if (rank == 0 && tid == 0) {
    wrow[0] = (int32_t)T;
    wrow[1] = k_rem;
  }
  const int nloc = blk1 - blk0;
  int carry_gt = gt_lo, carry_eq = eq_lo;
  for (int g0 = 0; g0 < nloc; g0 += kSelThreads) {
    const int ng = min(kSelThreads, nloc - g0);
    for (int jj = warp; jj < ng; jj += kSelWarps) {
      const int j = g0 + jj;
      int gt = 0, eq = 0;
      if (j < ncb) {
        for (int i = lane; i < nc[j]; i += 32) {
          const uint32_t k = keys[j * kBlk + i];
          gt += k > T;
          eq += k == T;
        }
      } else {
        const int q1 = min(j * kBlk + kBlk, cnt);
        for (int i = j * kBlk + lane; i < q1; i += 32) {
          const uint32_t k = float_key(src[i]);
          gt += k > T;
          eq += k == T;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
      }
      if (lane == 0) {
        bcnt[0][jj] = gt + (j < ncb ? gt0[j] : 0);
        bcnt[1][jj] = eq;
      }
    }
    __syncthreads();
    const int vg = tid < ng ? bcnt[0][tid] : 0, ve = tid < ng ? bcnt[1][tid] : 0;
    int ig = vg, ie = ve;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, ig, o), y = __shfl_up_sync(0xffffffffu, ie, o);
      if (lane >= o) {
        ig += x;
        ie += y;
      }
    }
    if (lane == 31) {
      wtot[0][warp] = ig;
      wtot[1][warp] = ie;
    }
    __syncthreads();
    int bg = 0, be = 0, tg = 0, te = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      if (w < warp) {
        bg += wtot[0][w];
        be += wtot[1][w];
      }
      tg += wtot[0][w];
      te += wtot[1][w];
    }
    if (tid < ng) {
      wrow[kWsHead + 2 * (blk0 + g0 + tid)] = carry_gt + bg + ig - vg;
      wrow[kWsHead + 2 * (blk0 + g0 + tid) + 1] = carry_eq + be + ie - ve;
    }
    carry_gt += tg;
    carry_eq += te;
    __syncthreads();
  }
  // after a copy wait that gave up, one thread waits (again bounded) for the copies still in
  // flight, so none lands in the shared memory of a CTA that has left (the CTA stays until
  // its last thread exits)
  if (tid == 0 && (err & 2))
    for (int i = 0; i < npieces; ++i) mbar_wait(&bars[i], 0, kCopyWaitNs);
  // the copy kernel may launch now (letting it take SMs earlier, while this kernel still
  // selects, measured 20-30% slower on long rows)
  griddep_launch_dependents();
  cluster_wait();  // no CTA leaves while another may still read its histograms
}

// ------------------------------------------------------------------ copy --
constexpr int kThreads = 1024;
constexpr int kRound = 4;       // positions per thread in one round of the kept-token sweep
constexpr int kPropRows = 1024;  // rows that the proportional split handles (one per thread)
constexpr int kMinBlocks = 2;   // blocks per CTA at least
constexpr int kSweepDiv = 16;   // one swept position costs about 1/16 of one kept token's copy

struct CompactArgs {
  const int32_t *N;
  const float *scores;
  const uint16_t *K, *V;
  const int32_t *head_order, *ntok;
  const int64_t *pt_off;
  const int32_t *pt_ids;
  const int32_t *ws;
  int64_t ws_row;
  int64_t pool_pages;
  uint16_t *pool;
  int32_t *kept_idx;
  int32_t *status;
  int H, H_p, G, P, d, Nmax;
  int parts;  // CTAs per row (the even split)
  int prop;   // share the grid's CTAs among the rows in proportion to their work
  int rows;   // batch * H
};

// Proportional shares: every row gets one CTA; the others go to the rows in proportion to
// their work, retained tokens plus positions swept, rounded on the running sum (a row's CTAs
// each sweep at least kMinBlocks blocks).  Every CTA derives the same shares from ntok and
// writes its (row, part, parts) to out[0..2], or out[0] = -1 past the last share.
__device__ __forceinline__ void prop_share(const CompactArgs &a, int *hist, int *scan, int *out) {
  const int rows = a.rows, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // a row's work: its kept tokens' copies, plus the sweep over all its N positions (about
  // a sixteenth of a kept token's cost per position)
  int nr = 0, cap = 0;
  if (tid < rows) {
    const int Nr = max(0, a.N[tid / a.H]);
    nr = max(0, a.ntok[tid]) + Nr / kSweepDiv;
    cap = max(0, (Nr + kBlk - 1) / kBlk / kMinBlocks - 1);
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

__global__ void __launch_bounds__(kThreads, 1) compact_copy_kernel(const CompactArgs a) {
  __shared__ int hist[64];
  __shared__ int scan[33];
  __shared__ int share[4];
  __shared__ int tok_list[kRound * kThreads];
  __shared__ int rank_scratch[kRound * kThreads / 32 + 1];

  int row = blockIdx.x / a.parts, part = blockIdx.x % a.parts, parts = a.parts;
  if (a.prop) {
    prop_share(a, hist, scan, share);
    if (share[0] < 0) return;  // past the last share
    row = share[0];
    part = share[1];
    parts = share[2];
  }
  const int b = row / a.H, h = row % a.H;
  const int Nb = a.N[b], n = a.ntok[row];
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

  const int nbr = (Nb + kBlk - 1) / kBlk;
  const int blk0 = (int)((int64_t)part * nbr / parts), blk1 = (int)((int64_t)(part + 1) * nbr / parts);
  const int c_begin = blk0 * kBlk, c_end = min(blk1 * kBlk, Nb);
  const float *srow = a.scores + (size_t)row * a.Nmax;
  const int d16 = a.d / 8;  // 16-byte chunks per row
  // copy layout: rpp rows per pass, chunk c8 / 8 of row r0 + j * rpp for this thread
  const int rpp = kThreads / d16, r0 = (int)threadIdx.x / d16;
  const int c8 = ((int)threadIdx.x % d16) * 8;
  const int pshift = (a.P & (a.P - 1)) == 0 ? __ffs(a.P) - 1 : -1;  // page of a slot by a shift when P is 2^k
  const size_t src_row0 = (size_t)row * a.Nmax;

  griddep_wait();  // T, need_eq and the block counts come from the select kernel
  const int32_t *wrow = a.ws + (size_t)row * a.ws_row;
  const uint32_t T = (uint32_t)wrow[0];
  const int need_eq = wrow[1];
  int taken = n, eq_seen = 0;
  if (c_begin < c_end) {
    eq_seen = wrow[kWsHead + 2 * blk0 + 1];
    taken = wrow[kWsHead + 2 * blk0] + min(eq_seen, need_eq);
  }
  // rounds of kRound * kThreads positions, position c0 + u * kThreads + thread
  for (int c0 = c_begin; c0 < c_end && taken < n; c0 += kRound * kThreads) {
    bool gt[kRound], eq[kRound], sel[kRound];
    float f[kRound];
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int t = c0 + u * kThreads + threadIdx.x;
      f[u] = t < c_end ? srow[t] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int t = c0 + u * kThreads + threadIdx.x;
      const uint32_t key = float_key(f[u]);
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

namespace {
int64_t compact_ws_ints_per_row(int Nmax) { return kWsHead + 2 * (((int64_t)Nmax + kBlk - 1) / kBlk); }
}  // namespace

extern "C" int tg_compact_topk_workspace(int batch, int H, int Nmax, int64_t *workspace_bytes) {
  if (!workspace_bytes) return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk_workspace: NULL output");
  if (batch < 0 || H <= 0 || Nmax <= 0)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk_workspace: sizes must be positive");
  *workspace_bytes = (int64_t)batch * H * compact_ws_ints_per_row(Nmax) * (int64_t)sizeof(int32_t);
  return tgi::ok();
}

extern "C" int tg_compact_topk(tg_stream_t stream, int batch, int H, int H_p, int P, int d, int Nmax,
                               const int32_t *N, const float *scores, const uint16_t *K, const uint16_t *V,
                               const int32_t *head_order, const int32_t *ntok, const int64_t *pt_off,
                               const int32_t *pt_ids, int64_t pool_pages, uint16_t *pool, int32_t *kept_idx,
                               void *workspace, int64_t workspace_bytes, int32_t *dev_status) {
  if (batch < 0 || H <= 0 || H_p <= 0 || P <= 0 || d <= 0 || Nmax <= 0)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: sizes must be positive");
  if (H % H_p) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: H %% H_p != 0");
  if (P % 16 || d % 8 || d > 512) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: need P %% 16 == 0, d %% 8 == 0, d <= 512");
  if (batch == 0) return tgi::ok();
  if (!N || !scores || !K || !V || !head_order || !ntok || !pt_off || !pt_ids || !pool || !workspace)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: NULL pointer argument");
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(pool)) & 15)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: K, V and pool must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 3)
    return tgi::fail(TG_ERR_INVALID_ARG, "tg_compact_topk: workspace must be 4-byte aligned");
  if ((int64_t)batch * H > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: batch * H too large");
  if (Nmax > INT32_MAX - kBlk) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: Nmax too large");
  const int rows = batch * H;
  const int64_t ws_row = compact_ws_ints_per_row(Nmax);
  if (workspace_bytes < (int64_t)rows * ws_row * (int64_t)sizeof(int32_t))
    return tgi::fail(TG_ERR_CAPACITY, "tg_compact_topk: workspace of %lld bytes, %lld needed",
                     (long long)workspace_bytes, (long long)((int64_t)rows * ws_row * 4));
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_topk: %s", cudaGetErrorString(e));
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int nblk = (Nmax + kBlk - 1) / kBlk;

  // select: C CTAs per row, one cluster each, and no CTA without a block of the longest row
  SelectArgs sa;
  sa.N = N; sa.scores = scores; sa.ntok = ntok; sa.ws = static_cast<int32_t *>(workspace); sa.status = dev_status;
  sa.ws_row = ws_row; sa.H = H; sa.Nmax = Nmax;
  sa.vec = (Nmax % 4 == 0) && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;
  {
    // one wave of two CTAs per SM, but at most 4 CTAs (the cluster's counts are read by every
    // CTA) unless more are needed for the chunks to fit
    const int fill = std::max(1, std::min(4, 2 * sms / rows));
    const int fit = (int)(((int64_t)nblk * kBlk + kSelKeys - 1) / kSelKeys);
    sa.C = std::max(1, std::min({std::max(fill, fit), kMaxCluster, nblk}));
  }
  if ((int64_t)rows * sa.C > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: grid too large");
  {
    const int smem = std::min(nblk * kBlk, kSelKeys) * (int)sizeof(uint32_t);
    e = cudaFuncSetAttribute(compact_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelKeys * 4);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(rows * sa.C));
      cfg.blockDim = dim3(kSelThreads);
      cfg.dynamicSmemBytes = (size_t)smem;
      cfg.stream = st;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = (unsigned)sa.C;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, compact_select_kernel, sa);
    }
  }
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_topk: select: %s", cudaGetErrorString(e));

  // copy: six waves of one resident 1024-thread CTA per SM, shared among the rows in
  // proportion to their work (or an even split of at most 16 CTAs per row past kPropRows
  // rows), each CTA at least kMinBlocks blocks.  A CTA has no fixed cost to speak of (the
  // select is done), so finer shares balance rows of very different length: two waves
  // measured 2.11 ms per layer of 256 rows of 4K-64K tokens, six 1.38 ms
  CompactArgs a;
  a.N = N; a.scores = scores; a.K = K; a.V = V; a.head_order = head_order; a.ntok = ntok;
  a.pt_off = pt_off; a.pt_ids = pt_ids; a.ws = sa.ws; a.ws_row = ws_row; a.pool_pages = pool_pages;
  a.pool = pool; a.kept_idx = kept_idx; a.status = dev_status;
  a.H = H; a.H_p = H_p; a.G = H / H_p; a.P = P; a.d = d; a.Nmax = Nmax;
  const int waves = 6;
  int parts = (waves * sms + rows - 1) / rows;
  parts = std::max(1, std::min({parts, 16, nblk / kMinBlocks}));
  a.parts = parts;
  a.rows = rows;
  a.prop = parts > 1 && rows <= kPropRows;
  // proportional shares take exactly the wanted waves (no partial wave at the end)
  const int64_t grid = a.prop ? std::max<int64_t>(rows, (int64_t)waves * sms) : (int64_t)rows * parts;
  if (grid > INT32_MAX) return tgi::fail(TG_ERR_SHAPE, "tg_compact_topk: grid too large");
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, compact_copy_kernel, a);
  }
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "tg_compact_topk: copy: %s", cudaGetErrorString(e));
  return tgi::ok();
}
