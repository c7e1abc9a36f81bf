// Quest page-score body (scores over the flat page sequence, fused per-row top-K
// selection), shared by the score kernel and the fused sparse-layer kernel.  See
// page_score.cu for the design and the fixed float32 order.
#pragma once

#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>

namespace {

using namespace tgk;

// a row's selection is out: its sel / pt_ids stores (fenced by the warp before this call)
// become visible to a reader that sees the flag
__device__ __forceinline__ void publish_ready(int32_t *flag, int epoch) {
  __threadfence();
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(epoch) : "memory");
}

constexpr int kMaxPages = 16384;                  // pages per (request, KV head) the select holds
constexpr uint64_t kScoreWaitNs = 2000000000ull;  // give up a copy wait after 2 s
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
  static constexpr int QUEUE = 64 * 8 + 16;     // completed-row queue (kRowQueue rows) and its counts
  static constexpr int SMEM = RING + NW * R * 8 + QUEUE;
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
  const int64_t *dense_base;  // [rows] page id of a row's page 0 in pt_ids (NULL: row * n_pages)
  int32_t *row_ready;  // [rows] set to `epoch` once a row's selection is written (NULL: not kept)
  int epoch;
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
                                             int32_t *pt_ids, int64_t id_base) {
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
      if (pt_ids) pt_ids[(size_t)row * K + pos] = (int32_t)(id_base + p);
    }
    taken += __popc(btake);
    eq_seen += __popc(beq);
  }
}

// the KPL bucket for n_pages <= 32 * kWarpKeysMax
__device__ __forceinline__ void warp_select(const uint32_t *rk, int n_pages, int K, int64_t row, int32_t *sel,
                                            int32_t *pt_ids, int64_t id_base) {
  const int kpl = (n_pages + 31) / 32;
  if (kpl <= 4) warp_select_row<4>(rk, n_pages, K, row, sel, pt_ids, id_base);
  else if (kpl <= 8) warp_select_row<8>(rk, n_pages, K, row, sel, pt_ids, id_base);
  else if (kpl <= 16) warp_select_row<16>(rk, n_pages, K, row, sel, pt_ids, id_base);
  else if (kpl <= 24) warp_select_row<24>(rk, n_pages, K, row, sel, pt_ids, id_base);
  else warp_select_row<32>(rk, n_pages, K, row, sel, pt_ids, id_base);
}

// The scoring (and, with a.fused, the selection) done by one CTA; smem: ScoreCfg<D>::SMEM bytes
// of dynamic shared memory, 128-byte aligned.  The score kernel and the fused sparse-layer
// kernel both run it.
template <int D, int GQ>
__device__ __forceinline__ void score_body(const ScoreArgs &a, uint8_t *smem) {
  using CF = ScoreCfg<D>;
  constexpr int NW = CF::NW, SP = CF::SP, PPL = CF::PPL, R = CF::R, PAGE = CF::PAGE, STAGE = CF::STAGE;
  constexpr int W = D / 16;   // elements per slice
  constexpr int WV = W / 8;   // 16-byte vectors per slice
  constexpr bool kPack = GQ * W <= 32;  // q+ and q- of the slice fit in registers as f32x2 pairs
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

  static_assert(kRowQueue * 8 + 16 <= CF::QUEUE, "queue space");
  // rows completed by this CTA's warps, to select (after the mbarriers, in dynamic shared memory)
  int64_t *s_rows = reinterpret_cast<int64_t *>(smem + CF::RING + NW * R * 8);
  int &s_nrows = *reinterpret_cast<int *>(smem + CF::RING + NW * R * 8 + kRowQueue * 8);
  int &s_more = *reinterpret_cast<int *>(smem + CF::RING + NW * R * 8 + kRowQueue * 8 + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = lane >> 4, j = lane & 15;
  if (threadIdx.x == 0) {
    s_nrows = 0;
    s_more = 0;
  }
  __syncthreads();
  // warps past NW (a kernel launched with more threads, the fused sparse layer) stream nothing:
  // they take part in the barriers and in the row selections
  const bool streams = warp < NW;
  const int nwarps = (int)(blockDim.x >> 5);
  uint8_t *wring = smem + (streams ? warp : 0) * R * STAGE;                                 // [R][STAGE]
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + CF::RING) + (streams ? warp : 0) * R;  // [R]

  // with a separate select kernel next, it may be scheduled now (it waits for this grid
  // before reading keys); with the select fused in, the next kernel (a decode reading the
  // page lists before it waits) starts only when this grid is done
  if (!a.fused || a.let_next) griddep_launch_dependents();

  // this warp's units [u0, u1)
  const int64_t c0 = (int64_t)blockIdx.x * a.units / gridDim.x;
  const int64_t c1 = (int64_t)(blockIdx.x + 1) * a.units / gridDim.x;
  const int64_t u0 = streams ? c0 + warp * (c1 - c0) / NW : c1;
  const int64_t u1 = streams ? c0 + (warp + 1) * (c1 - c0) / NW : c1;
  const int nst = (int)((u1 - u0 + SP - 1) / SP);
  if (streams && lane < R) mbar_init(&wbar[lane], 1);
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

  // query slice of the current row: q+ and q- as f32x2 pairs of heads (2i, 2i+1) when g >= 2,
  // as (q, q) pairs for g = 1, or raw bf16 words
  constexpr bool kPair = kPack && GQ >= 2;  // q+ and q- of head pairs (2i, 2i+1) per f32x2
  constexpr int QA = kPair ? GQ / 2 : (kPack ? GQ : 1);
  uint64_t qp2[QA][kPack ? W : 1], qm2[QA][kPack ? W : 1];
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
          if constexpr (kPair) {
            const float lo = bf16_lo(w4[e]), hi = bf16_hi(w4[e]);
            const int el = 8 * v + 2 * e;
            auto put = [&](uint64_t &p, float f) {
              if ((i & 1) == 0) {
                p = pack2(f, 0.f);
              } else {
                float x, y;
                unpack2(p, x, y);
                p = pack2(x, f);
              }
            };
            put(qp2[i / 2][el], fmaxf(lo, 0.f));
            put(qm2[i / 2][el], fminf(lo, 0.f));
            put(qp2[i / 2][el + 1], fmaxf(hi, 0.f));
            put(qm2[i / 2][el + 1], fminf(hi, 0.f));
          } else if constexpr (kPack) {
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
    bool ok = mbar_wait(&wbar[st % R], (uint32_t)((st / R) & 1), kScoreWaitNs);
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
      if constexpr (kPair) {
        uint64_t acc[PPL][QA];  // (head 2i, head 2i+1) of slot k
#pragma unroll
        for (int k = 0; k < PPL; ++k)
#pragma unroll
          for (int i = 0; i < QA; ++i) acc[k][i] = 0ull;
#pragma unroll
        for (int v = 0; v < WV; ++v) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int el = 8 * v + 2 * e;
            uint64_t x0[PPL], n0[PPL], x1[PPL], n1[PPL];
#pragma unroll
            for (int k = 0; k < PPL; ++k) {
              const uint32_t wx = (&mx[k][v].x)[e], wn = (&mn[k][v].x)[e];
              x0[k] = pack2(bf16_lo(wx), bf16_lo(wx));
              n0[k] = pack2(bf16_lo(wn), bf16_lo(wn));
              x1[k] = pack2(bf16_hi(wx), bf16_hi(wx));
              n1[k] = pack2(bf16_hi(wn), bf16_hi(wn));
            }
#pragma unroll
            for (int k = 0; k < PPL; ++k)
#pragma unroll
              for (int i = 0; i < QA; ++i) ffma2(acc[k][i], qp2[i][el], x0[k]);
#pragma unroll
            for (int k = 0; k < PPL; ++k)
#pragma unroll
              for (int i = 0; i < QA; ++i) ffma2(acc[k][i], qm2[i][el], n0[k]);
#pragma unroll
            for (int k = 0; k < PPL; ++k)
#pragma unroll
              for (int i = 0; i < QA; ++i) ffma2(acc[k][i], qp2[i][el + 1], x1[k]);
#pragma unroll
            for (int k = 0; k < PPL; ++k)
#pragma unroll
              for (int i = 0; i < QA; ++i) ffma2(acc[k][i], qm2[i][el + 1], n1[k]);
          }
        }
#pragma unroll
        for (int k = 0; k < PPL; ++k)
#pragma unroll
          for (int i = 0; i < QA; ++i) unpack2(acc[k][i], val[k * GQ + 2 * i], val[k * GQ + 2 * i + 1]);
      } else if constexpr (kPack) {
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
      if (!mbar_wait(&wbar[t % R], (uint32_t)((t / R) & 1), kScoreWaitNs)) break;
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
      for (int i = warp; i < nq; i += nwarps) {
        const int64_t r = s_rows[i];
        const int64_t out = row_id(r);
        if (out >= 0) warp_select(a.keys + r * a.n_pages, a.n_pages, a.K, out, a.sel, a.pt_ids,
                                  a.dense_base ? a.dense_base[out] : out * a.n_pages);
        if (lane == 0) {
          a.row_cnt[r] = 0;
          if (a.row_ready && out >= 0) publish_ready(a.row_ready + out, a.epoch);
        }
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
          if (out >= 0) warp_select(a.keys + r * a.n_pages, a.n_pages, a.K, out, a.sel, a.pt_ids,
                                  a.dense_base ? a.dense_base[out] : out * a.n_pages);
          if (lane == 0) {
            a.row_cnt[r] = 0;
            if (a.row_ready && out >= 0) publish_ready(a.row_ready + out, a.epoch);
          }
        }
      }
    }
  }
  // complete only after the kernel before this one in the stream: the kernel that
  // follows may overwrite page lists that kernel reads
  griddep_wait();
}

}  // namespace
