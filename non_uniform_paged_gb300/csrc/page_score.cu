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
//    half warp scores two pages at once, lane j owning slice j, with the two
//    pages' chains packed into f32x2 FMAs.  The 16 slice sums are combined by an
//    xor butterfly that also spreads the g heads over the lanes (every add is
//    one of the fixed pairs; a + b == b + a in float32).  Scores go to the
//    workspace as order-preserving keys.
//  * page_select_warp_kernel (rows of up to 1024 pages: one warp per (request,
//    KV head), keys in registers) or page_select_kernel (longer rows: one CTA,
//    keys in shared memory): an exact radix select of the K-th largest key, then
//    an ascending sweep (ties to the lower page).
#include "block_select.cuh"
#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

#include <algorithm>

namespace {

using namespace tgk;

constexpr int kMaxPages = 16384;                  // pages per (request, KV head) the select holds
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // give up a copy wait after 2 s
constexpr int kSelThreads = 256;

template <int D>
struct ScoreCfg {
  static constexpr int NW = 8;                   // warps per CTA
  static constexpr int PAGE = 4 * D;             // bytes of one page: min row, then max row (bf16)
  static constexpr int SP = D == 128 ? 8 : 4;    // pages per stage; a half warp scores SP/2 of them
  static constexpr int PPL = SP / 2;             // pages per lane (stage pages hw, hw+2, hw+4, ...)
  static constexpr int R = 4;                    // stages per warp
  static constexpr int STAGE = SP * PAGE;        // 4 KB
  static constexpr int RING = NW * R * STAGE;    // 128 KB
  static constexpr int SMEM = RING + NW * R * 8;
};

struct ScoreArgs {
  const uint16_t *q, *minmax;
  uint32_t *keys;      // [rows][n_pages] scores as keys (workspace)
  int32_t *row_cnt;    // [rows] pages scored so far (workspace, zero between calls)
  int32_t *sel, *pt_ids;
  int32_t *status;
  const int32_t *rows; // the (request, KV head) rows to score, in list order (NULL: all, in order)
  int64_t total_rows;  // batch * H: listed rows outside [0, total_rows) are reported and skipped
  int64_t units;       // listed rows * n_pages
  int g, n_pages, K;
  int fused;           // the warp that completes a row selects its top K (n_pages <= 1024)
  int let_next;        // let the next kernel start early (it waits before reading sel / pt_ids)
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint64_t pack2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &x, float &y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
// two independent IEEE fused multiply-adds, round to nearest: d.x = a.x b.x + d.x, d.y = a.y b.y + d.y
__device__ __forceinline__ void ffma2(uint64_t &d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__host__ __device__ constexpr int log2c(int n) { return n <= 1 ? 0 : 1 + log2c(n / 2); }

// Add the 16 slice sums of NV values over the 16 lanes of a half warp (lane j = slice j)
// in the fixed pair order: xor levels 8, 4, 2, 1 add the pairs (j, j^o).  While a lane
// holds more than one value, each level also halves what it keeps: it keeps one half of
// its values, sends the other half to its partner and adds the partner's copy of the half
// it kept (a + b == b + a in float32, so both lanes of a pair add the same two numbers).
// After min(4, log2 NV) such levels the lane holds NV >> LS values, value r being number
// base + r where base = sum over split levels k of (bit 8>>k of the lane) * NV >> (k+1).
template <int NV>
__device__ __forceinline__ void transpose_sum(float (&v)[NV], int lane) {
  constexpr int LS = log2c(NV) < 4 ? log2c(NV) : 4;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int o = 8 >> k;
    if (k < LS) {
      const int h = NV >> (k + 1);
      const bool up = lane & o;
      float recv[NV / 2 > 0 ? NV / 2 : 1];
#pragma unroll
      for (int t = 0; t < NV / 2; ++t)  // all shuffles of the level first, then the adds
        if (t < h) recv[t] = __shfl_xor_sync(0xffffffffu, up ? v[t] : v[t + h], o);
#pragma unroll
      for (int t = 0; t < NV / 2; ++t)
        if (t < h) v[t] = __fadd_rn(up ? v[t + h] : v[t], recv[t]);
    } else {
      float recv[NV >> LS];
#pragma unroll
      for (int t = 0; t < (NV >> LS); ++t) recv[t] = __shfl_xor_sync(0xffffffffu, v[t], o);
#pragma unroll
      for (int t = 0; t < (NV >> LS); ++t) v[t] = __fadd_rn(v[t], recv[t]);
    }
  }
}

// Top K of one (request, KV head) row of at most 32 x KPL pages, by one warp.  The row's keys
// sit in registers (lane l holds pages l, l+32, ...; missing pages hold key 0, which no
// candidate below reaches).  The K-th largest key T is built bit by bit from the top: a bit
// stays set when at least K keys are >= the prefix with it (a warp-wide count per bit; the
// bits on which all keys agree are taken as they are).  A ballot sweep then lists the winners
// in ascending page order: every key > T, and the lowest pages among the keys == T.
constexpr int kWarpKeysMax = 32;
constexpr int kRowQueue = 64;  // completed rows a score CTA queues for its warps to select

template <int KPL>
__device__ __noinline__ void warp_select_row(const uint32_t *rk, int n_pages, int K, int64_t row, int32_t *sel,
                                             int32_t *pt_ids) {
  const int lane = threadIdx.x & 31;
  uint32_t key[KPL];
  uint32_t k_and = 0xffffffffu, k_or = 0u;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const bool valid = 32 * i + lane < n_pages;
    key[i] = valid ? __ldcg(rk + 32 * i + lane) : 0u;
    k_and &= valid ? key[i] : 0xffffffffu;
    k_or |= key[i];
  }
  k_and = __reduce_and_sync(0xffffffffu, k_and);
  k_or = __reduce_or_sync(0xffffffffu, k_or);
  // number of keys >= c, for c >= 1 (missing pages hold 0): four independent partial counts
  auto count_ge = [&](uint32_t c) {
    int n[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < KPL; ++i) n[i & 3] += key[i] >= c;
    return (int)__reduce_add_sync(0xffffffffu, (unsigned)(n[0] + n[1] + n[2] + n[3]));
  };
  uint32_t T = k_and;  // all keys agree above the top differing bit (and T == k_and if they all agree)
  const uint32_t differ = k_and ^ k_or;
  if (differ) {
    const int top = 31 - __clz(differ);
    T = top == 31 ? 0u : T & ~((2u << top) - 1u);
#pragma unroll 1
    for (int bit = top; bit >= 0; --bit) {
      const uint32_t cand = T | (1u << bit);
      if (count_ge(cand) >= K) T = cand;
    }
  }
  const int need_eq = K - (T == 0xffffffffu ? 0 : count_ge(T + 1));  // keys equal to T to take
  const uint32_t lt = (1u << lane) - 1u;
  int taken = 0, eq_seen = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const bool eq = key[i] == T && 32 * i + lane < n_pages;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const bool take = key[i] > T || (eq && eq_seen + __popc(beq & lt) < need_eq);
    const uint32_t btake = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int pos = taken + __popc(btake & lt);
      const int p = 32 * i + lane;
      sel[(size_t)row * K + pos] = p;
      if (pt_ids) pt_ids[(size_t)row * K + pos] = (int32_t)(row * n_pages + p);
    }
    taken += __popc(btake);
    eq_seen += __popc(beq);
  }
}

// the KPL bucket for n_pages <= 32 * kWarpKeysMax
__device__ __forceinline__ void warp_select(const uint32_t *rk, int n_pages, int K, int64_t row, int32_t *sel,
                                            int32_t *pt_ids) {
  const int kpl = (n_pages + 31) / 32;
  if (kpl <= 4) warp_select_row<4>(rk, n_pages, K, row, sel, pt_ids);
  else if (kpl <= 8) warp_select_row<8>(rk, n_pages, K, row, sel, pt_ids);
  else if (kpl <= 16) warp_select_row<16>(rk, n_pages, K, row, sel, pt_ids);
  else if (kpl <= 24) warp_select_row<24>(rk, n_pages, K, row, sel, pt_ids);
  else warp_select_row<32>(rk, n_pages, K, row, sel, pt_ids);
}

template <int D, int GQ>
__global__ void __launch_bounds__(ScoreCfg<D>::NW * 32, 1) page_score_kernel(const ScoreArgs a) {
  using CF = ScoreCfg<D>;
  constexpr int NW = CF::NW, SP = CF::SP, PPL = CF::PPL, R = CF::R, PAGE = CF::PAGE, STAGE = CF::STAGE;
  constexpr int W = D / 16;   // elements per slice
  constexpr int WV = W / 8;   // 16-byte vectors per slice
  constexpr bool kPack = GQ * W <= 32;  // q+ and q- as duplicated f32x2 pairs fit in registers
  // values per lane after the slice sums: NV = PPL pages x GQ heads, value number slot * GQ + head
  constexpr int NV = PPL * GQ;
  constexpr int LS = log2c(NV) < 4 ? log2c(NV) : 4;  // split levels of transpose_sum
  constexpr int NR = NV >> LS;                       // values a lane holds afterwards
  static_assert(NR <= GQ && GQ % NR == 0, "a lane's values after the sum are heads of one page");
  // lane bits that index heads (split levels of weight < GQ) or that hold copies (levels past LS);
  // a lane with none of them set writes the page's key
  constexpr int kHeadLevels = log2c(GQ / NR);
  int wmask = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (k >= LS - kHeadLevels) wmask |= 8 >> k;
  static_assert(SP == 2 * PPL && PPL % 2 == 0, "pages are scored in f32x2 pairs");

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int64_t s_rows[kRowQueue];  // rows completed by this CTA's warps, to select
  __shared__ int s_nrows, s_more;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = lane >> 4, j = lane & 15;
  if (threadIdx.x == 0) {
    s_nrows = 0;
    s_more = 0;
  }
  __syncthreads();
  uint8_t *wring = smem + warp * R * STAGE;                                     // [R][STAGE]
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + CF::RING) + warp * R;   // [R]

  // with a separate select kernel next, it may be scheduled now (it waits for this grid
  // before reading keys); with the select fused in, the next kernel (a decode reading the
  // page lists before it waits) starts only when this grid is done
  if (!a.fused || a.let_next) griddep_launch_dependents();

  // this warp's units [u0, u1)
  const int64_t c0 = (int64_t)blockIdx.x * a.units / gridDim.x;
  const int64_t c1 = (int64_t)(blockIdx.x + 1) * a.units / gridDim.x;
  const int64_t u0 = c0 + warp * (c1 - c0) / NW, u1 = c0 + (warp + 1) * (c1 - c0) / NW;
  const int nst = (int)((u1 - u0 + SP - 1) / SP);
  if (lane < R) mbar_init(&wbar[lane], 1);
  fence_barrier_init();
  __syncwarp();
  const uint8_t *src = reinterpret_cast<const uint8_t *>(a.minmax);
  // row of list position lr (the rows of a listed call need not be adjacent in memory)
  auto row_id = [&](int64_t lr) -> int64_t {
    if (!a.rows) return lr;
    const int64_t r = __ldcg(a.rows + lr);
    return r >= 0 && r < a.total_rows ? r : -1;
  };
  auto issue = [&](int st) {  // lane 0: stage st of this warp, one bulk copy per row it touches
    const int64_t us = u0 + (int64_t)st * SP;
    const int cnt = (int)min((int64_t)SP, u1 - us);
    uint64_t *bar = &wbar[st % R];
    uint8_t *dst = wring + (st % R) * STAGE;
    mbar_arrive_expect_tx(bar, (uint32_t)(cnt * PAGE));
    if (!a.rows) {
      bulk_load(dst, src + us * PAGE, (uint32_t)(cnt * PAGE), bar);
      return;
    }
    for (int done = 0; done < cnt;) {
      const int64_t u = us + done, lr = u / a.n_pages, pg = u - lr * a.n_pages;
      const int seg = (int)min((int64_t)(cnt - done), a.n_pages - pg);
      int64_t r = row_id(lr);
      if (r < 0) {  // a listed row out of range: read row 0 instead, select nothing for it
        report(a.status, TG_STATUS_BAD_INPUT);
        r = 0;
      }
      bulk_load(dst + done * PAGE, src + (r * a.n_pages + pg) * PAGE, (uint32_t)(seg * PAGE), bar);
      done += seg;
    }
  };
  if (lane == 0)
    for (int st = 0; st < R && st < nst; ++st) issue(st);
  int issued = min(R, nst);

  // query slice of the current row: packed (q, q) pairs of q+ and q-, or raw bf16 words
  uint64_t qp2[kPack ? GQ : 1][kPack ? W : 1], qm2[kPack ? GQ : 1][kPack ? W : 1];
  uint32_t qv[kPack ? 1 : GQ][kPack ? 1 : W / 2];
  int64_t row = u0 / a.n_pages;
  int64_t row_lo = row * a.n_pages, row_hi = row_lo + a.n_pages;
  bool q_nan = false;  // a NaN in this lane's query slice (q+ and q- would hide it)
  auto load_q = [&]() {
    q_nan = false;
#pragma unroll
    for (int i = 0; i < GQ; ++i) {
      const int qi = i < a.g ? i : 0;  // heads past g repeat head 0: the max is unchanged
      const uint4 *qs = reinterpret_cast<const uint4 *>(a.q + ((size_t)max(row_id(row), (int64_t)0) * a.g + qi) * D + j * W);
#pragma unroll
      for (int v = 0; v < WV; ++v) {
        const uint4 x = __ldcg(qs + v);
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          q_nan |= i < a.g && (is_nan(bf16_lo(w4[e])) || is_nan(bf16_hi(w4[e])));
          if constexpr (kPack) {
            const float lo = bf16_lo(w4[e]), hi = bf16_hi(w4[e]);
            qp2[i][8 * v + 2 * e] = pack2(fmaxf(lo, 0.f), fmaxf(lo, 0.f));
            qm2[i][8 * v + 2 * e] = pack2(fminf(lo, 0.f), fminf(lo, 0.f));
            qp2[i][8 * v + 2 * e + 1] = pack2(fmaxf(hi, 0.f), fmaxf(hi, 0.f));
            qm2[i][8 * v + 2 * e + 1] = pack2(fminf(hi, 0.f), fminf(hi, 0.f));
          } else {
            qv[i][4 * v + e] = w4[e];
          }
        }
      }
    }
  };
  if (nst > 0) load_q();

  // page slot of this lane's values after transpose_sum (only meaningful for writers)
  int base = 0;
#pragma unroll
  for (int k = 0; k < LS; ++k)
    if (lane & (8 >> k)) base += NV >> (k + 1);
  const int my_slot = base / GQ;
  const bool writer = (lane & wmask) == 0;

  bool nan_seen = false, dead = false;
  int st = 0;
  for (; st < nst; ++st) {
    bool ok = mbar_wait(&wbar[st % R], (uint32_t)((st / R) & 1), kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) report(a.status, TG_STATUS_TIMEOUT);
      dead = true;
      break;
    }
    const uint8_t *stage = wring + (st % R) * STAGE;
    const int64_t us = u0 + (int64_t)st * SP;
    const int cnt = (int)min((int64_t)SP, u1 - us);
    // slot s of this lane is stage page hw + 2s; pages past cnt read stale shared memory
    // and are never written
    uint4 mn[PPL][WV], mx[PPL][WV];
#pragma unroll
    for (int sl = 0; sl < PPL; ++sl) {
      const uint4 *rp = reinterpret_cast<const uint4 *>(stage + (hw + 2 * sl) * PAGE + j * W * 2);
#pragma unroll
      for (int v = 0; v < WV; ++v) {
        mn[sl][v] = rp[v];
        mx[sl][v] = rp[v + D / 8];  // the max row follows the min row: 2*D bytes = D/8 vectors
      }
    }
    // score the stage pages in `mine` against the current row's query (all of them lie in it)
    auto score_pages = [&](const uint32_t mine) {
      float val[NV];  // slot * GQ + head
      if constexpr (kPack) {
        uint64_t acc[PPL / 2][GQ];  // (slot 2k, slot 2k+1) of head i
#pragma unroll
        for (int k = 0; k < PPL / 2; ++k)
#pragma unroll
          for (int i = 0; i < GQ; ++i) acc[k][i] = 0ull;
#pragma unroll
        for (int v = 0; v < WV; ++v) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int el = 8 * v + 2 * e;
            uint64_t x0[PPL / 2], n0[PPL / 2], x1[PPL / 2], n1[PPL / 2];
#pragma unroll
            for (int k = 0; k < PPL / 2; ++k) {
              const uint32_t wx0 = (&mx[2 * k][v].x)[e], wx1 = (&mx[2 * k + 1][v].x)[e];
              const uint32_t wn0 = (&mn[2 * k][v].x)[e], wn1 = (&mn[2 * k + 1][v].x)[e];
              x0[k] = pack2(bf16_lo(wx0), bf16_lo(wx1));
              n0[k] = pack2(bf16_lo(wn0), bf16_lo(wn1));
              x1[k] = pack2(bf16_hi(wx0), bf16_hi(wx1));
              n1[k] = pack2(bf16_hi(wn0), bf16_hi(wn1));
            }
            // four rounds over every (pair, head) chain: consecutive FMAs are independent
#pragma unroll
            for (int k = 0; k < PPL / 2; ++k)
#pragma unroll
              for (int i = 0; i < GQ; ++i) ffma2(acc[k][i], qp2[i][el], x0[k]);
#pragma unroll
            for (int k = 0; k < PPL / 2; ++k)
#pragma unroll
              for (int i = 0; i < GQ; ++i) ffma2(acc[k][i], qm2[i][el], n0[k]);
#pragma unroll
            for (int k = 0; k < PPL / 2; ++k)
#pragma unroll
              for (int i = 0; i < GQ; ++i) ffma2(acc[k][i], qp2[i][el + 1], x1[k]);
#pragma unroll
            for (int k = 0; k < PPL / 2; ++k)
#pragma unroll
              for (int i = 0; i < GQ; ++i) ffma2(acc[k][i], qm2[i][el + 1], n1[k]);
          }
        }
#pragma unroll
        for (int k = 0; k < PPL / 2; ++k)
#pragma unroll
          for (int i = 0; i < GQ; ++i) unpack2(acc[k][i], val[(2 * k) * GQ + i], val[(2 * k + 1) * GQ + i]);
      } else {
#pragma unroll
        for (int t = 0; t < NV; ++t) val[t] = 0.f;
#pragma unroll
        for (int v = 0; v < WV; ++v) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
#pragma unroll
            for (int sl = 0; sl < PPL; ++sl) {
              const uint32_t wn = (&mn[sl][v].x)[e], wx = (&mx[sl][v].x)[e];
#pragma unroll
              for (int i = 0; i < GQ; ++i) {
                const uint32_t qq = qv[i][4 * v + e];
                const float q0 = bf16_lo(qq), q1 = bf16_hi(qq);
                float &acc = val[sl * GQ + i];
                acc = __fadd_rn(acc, fmaxf(__fmul_rn(q0, bf16_lo(wn)), __fmul_rn(q0, bf16_lo(wx))));
                acc = __fadd_rn(acc, fmaxf(__fmul_rn(q1, bf16_hi(wn)), __fmul_rn(q1, bf16_hi(wx))));
              }
            }
          }
        }
      }
      transpose_sum<NV>(val, lane);
      // val[0 .. NR-1]: heads (base % GQ) .. of page slot my_slot; max over the page's heads
      float best = val[0];
      bool nan_here = is_nan(val[0]);
#pragma unroll
      for (int r = 1; r < NR; ++r) {
        best = fmaxf(best, val[r]);
        nan_here |= is_nan(val[r]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k >= LS - kHeadLevels && k < LS) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 8 >> k));
      const int po = hw + 2 * my_slot;  // stage page of this lane's values
      const bool own = (mine >> po) & 1u;
      nan_seen |= (own && nan_here) || (mine && q_nan);
      if (writer && own) a.keys[us + po] = float_key(best);
    };
    constexpr uint32_t kAll = (1u << SP) - 1u;
    if (cnt == SP && us >= row_lo && us + SP <= row_hi) {
      score_pages(kAll);  // the common case: a full stage inside the current row
    } else {
      uint32_t done = kAll & ~((1u << cnt) - 1u);
      while (done != kAll) {
        // one row at a time (a stage straddles a row end only rarely)
        const int first = __ffs(~done & kAll) - 1;
        if (us + first >= row_hi) {
          while (us + first >= row_hi) {
            ++row;
            row_lo = row_hi;
            row_hi += a.n_pages;
          }
          load_q();
        }
        const int lo = (int)max(row_lo - us, (int64_t)0), hi = (int)min(row_hi - us, (int64_t)SP);
        const uint32_t mine = ((1u << hi) - 1u) & ~((1u << lo) - 1u) & ~done;
        score_pages(mine);
        done |= mine;
      }
    }
    __syncwarp();
    if (issued < nst) {
      if (lane == 0) {
        fence_proxy_async_smem();  // our reads of this stage come before the refill
        issue(issued);
      }
      ++issued;
    }
  }
  if (dead && lane == 0) {  // drain this warp's copies still in flight
    for (int t = st; t < issued; ++t)
      if (!mbar_wait(&wbar[t % R], (uint32_t)((t / R) & 1), kWaitLimitNs)) break;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) report(a.status, TG_STATUS_NONFINITE);

  // ---- rows this warp scored: add their page counts.  A row whose count reaches n_pages
  // is complete (its keys are all in L2): the CTA queues it, and once all its warps are
  // done streaming, they share the queued selections, one row per warp at a time
  if (a.fused) {
    if (nst > 0 && !dead) {
      __threadfence();  // this lane's key stores before the count
      __syncwarp();
      const int64_t r_first = u0 / a.n_pages, r_last = (u1 - 1) / a.n_pages;
      for (int64_t r = r_first; r <= r_last; ++r) {
        const int64_t lo = max(u0, r * a.n_pages), hi = min(u1, (r + 1) * a.n_pages);
        if (lane == 0 && atomicAdd(&a.row_cnt[r], (int)(hi - lo)) + (int)(hi - lo) == a.n_pages) {
          const int at = atomicAdd(&s_nrows, 1);
          if (at < kRowQueue) s_rows[at] = r;
          else s_more = 1;  // more rows than the queue holds: the overflow is found below
        }
      }
    }
    __syncthreads();
    const int nq = min(s_nrows, kRowQueue);
    if (nq > 0) {
      __threadfence();   // the other CTAs' key stores, ordered by their counts
      griddep_wait();    // the previous kernel (a decode) may still read sel / pt_ids
      for (int i = warp; i < nq; i += NW) {
        const int64_t r = s_rows[i];
        const int64_t out = row_id(r);
        if (out >= 0) warp_select(a.keys + r * a.n_pages, a.n_pages, a.K, out, a.sel, a.pt_ids);
        if (lane == 0) a.row_cnt[r] = 0;
      }
    }
    if (s_more && nst > 0 && !dead) {  // rare: rescan this warp's rows for completed ones not queued
      const int64_t r_first = u0 / a.n_pages, r_last = (u1 - 1) / a.n_pages;
      for (int64_t r = r_first; r <= r_last; ++r) {
        int mine_row = 0;
        if (lane == 0 && atomicAdd(&a.row_cnt[r], 0) == a.n_pages) {
          mine_row = 1;
          for (int i = 0; i < nq; ++i) mine_row &= s_rows[i] != r;
          // claim it: only one warp of this CTA may select a row left out of the queue
          if (mine_row) mine_row = atomicCAS(&a.row_cnt[r], a.n_pages, -1) == a.n_pages;
        }
        if (__shfl_sync(0xffffffffu, mine_row, 0)) {
          __threadfence();
          griddep_wait();
          const int64_t out = row_id(r);
          if (out >= 0) warp_select(a.keys + r * a.n_pages, a.n_pages, a.K, out, a.sel, a.pt_ids);
          if (lane == 0) a.row_cnt[r] = 0;
        }
      }
    }
  }
  // complete only after the kernel before this one in the stream: the kernel that
  // follows may overwrite page lists that kernel reads
  griddep_wait();
}

// One CTA per (request, KV head): top-K of the row's keys, ascending, ties to the lower page.
__global__ void __launch_bounds__(kSelThreads) page_select_kernel(const uint32_t *keys, const int32_t *rows,
                                                                  int64_t total_rows, int n_pages, int K,
                                                                  int32_t *sel, int32_t *pt_ids) {
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
      if (pt_ids) pt_ids[(size_t)out_row * K + k] = (int32_t)(out_row * n_pages + p);
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
                          int K, int32_t *sel, int32_t *pt_ids, cudaStream_t s) {
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
  return cudaLaunchKernelEx(&cfg, page_select_kernel, keys, rows, total_rows, n_pages, K, sel, pt_ids);
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

extern "C" int tg_page_score_workspace(int batch, int H, int n_pages, int64_t *workspace_bytes) {
  if (!workspace_bytes) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_workspace: NULL workspace_bytes");
  if (batch < 0 || H <= 0 || n_pages < 1) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_workspace: bad sizes");
  // page keys, then one page counter per (request, KV head)
  *workspace_bytes = tgi::align_up((int64_t)batch * H * n_pages * 4, 256) + tgi::align_up((int64_t)batch * H * 4, 256);
  return tgi::ok();
}

namespace {
int score_topk(const char *fn, tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K, int n_rows,
               const int32_t *rows, const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
               void *workspace, int64_t workspace_bytes, uint32_t flags, int32_t *dev_status) {
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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = d == 128 ? launch_score_d<128>(a, s) : launch_score_d<256>(a, s);
  if (e == cudaSuccess && !a.fused) e = launch_select(a.keys, rows, a.total_rows, n_rows, n_pages, K, sel, pt_ids, s);
  if (e != cudaSuccess) return tgi::fail(TG_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return tgi::ok();
}
}  // namespace

extern "C" int tg_page_score_topk(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                                  const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
                                  void *workspace, int64_t workspace_bytes, uint32_t flags, int32_t *dev_status) {
  return score_topk("tg_page_score_topk", stream, batch, H, g, d, n_pages, K, batch * H, nullptr, q, minmax, sel,
                    pt_ids, workspace, workspace_bytes, flags, dev_status);
}

extern "C" int tg_page_score_topk_rows(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                                       int n_rows, const int32_t *rows, const uint16_t *q, const uint16_t *minmax,
                                       int32_t *sel, int32_t *pt_ids, void *workspace, int64_t workspace_bytes,
                                       uint32_t flags, int32_t *dev_status) {
  if (n_rows > 0 && !rows) return tgi::fail(TG_ERR_INVALID_ARG, "tg_page_score_topk_rows: NULL rows");
  return score_topk("tg_page_score_topk_rows", stream, batch, H, g, d, n_pages, K, n_rows, rows, q, minmax, sel,
                    pt_ids, workspace, workspace_bytes, flags, dev_status);
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
