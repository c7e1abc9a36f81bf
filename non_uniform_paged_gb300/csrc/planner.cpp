// Host-side planning of the ragged decode path: page tables (a1), the
// workload split map (a3) and the per-CTA decode plan (a4).
//
// Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
// Multi-turn LLM Serving" (paper-review page), sections 3.1-3.3.  The
// readings of the points that page leaves open are stated in include/tg.h
// next to each entry point.
#include "tg_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

namespace {
thread_local std::string g_error;
}

namespace tgi {
int fail(int code, const char *fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}
int ok() {
  g_error.clear();
  return TG_OK;
}
}  // namespace tgi

using tgi::fail;

extern "C" const char *tg_last_error_string(void) { return g_error.c_str(); }
extern "C" int tg_version(void) { return 100; }

namespace {

// ceil(B * N) for a float32 budget B in (0, 1], exactly: B = m * 2^-s with a
// 24-bit integer m, so B*N = m*N / 2^s is a ratio of integers (section 3.1,
// size of Top(ceil(B N), s)).  Clamped to [1, N]; 0 for an empty context.
int32_t retained_count(float B, int32_t N) {
  if (N <= 0) return 0;
  int e = 0;
  float fr = std::frexp(B, &e);  // B = fr * 2^e, fr in [0.5, 1)
  uint64_t m = (uint64_t)std::ldexp(fr, 24);
  int s = 24 - e;  // B = m / 2^s, s >= 23 because B <= 1
  unsigned __int128 num = (unsigned __int128)m * (uint64_t)N;
  int64_t n;
  if (s >= 120) {
    n = 1;  // m*N < 2^55 << 2^s: 0 < B*N < 1
  } else {
    unsigned __int128 q = num >> s;
    if ((q << s) != num) q += 1;
    n = (int64_t)q;
  }
  return (int32_t)std::max<int64_t>(1, std::min<int64_t>(N, n));
}

}  // namespace

extern "C" int tg_build_pages(int L, int batch, int H, int H_p, int P, float alpha,
                              const float *Bhat, const int32_t *N, int cluster,
                              int32_t *head_order, int32_t *ntok, int64_t *Phi,
                              int64_t *pt_off, int32_t *pt_ids, int64_t pt_cap,
                              int64_t *n_pages, int64_t *n_pages_monolithic) {
  if (L <= 0 || batch < 0 || H <= 0 || H_p <= 0 || P <= 0)
    return fail(TG_ERR_INVALID_ARG, "tg_build_pages: L=%d batch=%d H=%d H_p=%d P=%d must be positive",
                L, batch, H, H_p, P);
  if (H % H_p) return fail(TG_ERR_SHAPE, "tg_build_pages: H=%d is not a multiple of H_p=%d", H, H_p);
  if (P % 16) return fail(TG_ERR_SHAPE, "tg_build_pages: P=%d must be a multiple of 16", P);
  if (!Bhat || (batch > 0 && !N)) return fail(TG_ERR_INVALID_ARG, "tg_build_pages: NULL Bhat or N");
  if (!(std::isfinite(alpha) && alpha > 0.f))
    return fail(TG_ERR_NONFINITE, "tg_build_pages: alpha=%g must be finite and > 0", (double)alpha);
  const int G = H / H_p;
  std::vector<float> B((size_t)L * H);
  for (int i = 0; i < L * H; ++i) {
    if (!std::isfinite(Bhat[i]) || !(Bhat[i] > 0.f))
      return fail(TG_ERR_NONFINITE, "tg_build_pages: Bhat[%d]=%g must be finite and > 0", i, (double)Bhat[i]);
    float b = alpha * Bhat[i];  // one float32 rounding: B = fp32(alpha * B^)
    B[i] = b < 1.f ? b : 1.f;
  }
  for (int b = 0; b < batch; ++b)
    if (N[b] < 0) return fail(TG_ERR_INVALID_ARG, "tg_build_pages: N[%d]=%d is negative", b, N[b]);

  // group membership (section 3.2, budget-aware clustering)
  std::vector<int32_t> order((size_t)L * H);
  for (int l = 0; l < L; ++l) {
    int32_t *o = &order[(size_t)l * H];
    std::iota(o, o + H, 0);
    if (cluster) {
      const float *Bl = &B[(size_t)l * H];
      std::stable_sort(o, o + H, [Bl](int32_t a, int32_t c) { return Bl[a] > Bl[c]; });
    }
  }
  std::vector<int32_t> n((size_t)L * batch * H);
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < batch; ++b)
      for (int h = 0; h < H; ++h)
        n[((size_t)l * batch + b) * H + h] = retained_count(B[(size_t)l * H + h], N[b]);

  // pages per list (l, b, g), CSR offsets in (l, b, g) order
  const int64_t n_lists = (int64_t)L * batch * G;
  std::vector<int64_t> off(n_lists + 1, 0);
  int64_t mono = 0;
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < batch; ++b) {
      const int32_t *nb = &n[((size_t)l * batch + b) * H];
      int32_t all_max = 0;
      for (int g = 0; g < G; ++g) {
        int32_t mx = 0;
        for (int j = 0; j < H_p; ++j) mx = std::max(mx, nb[order[(size_t)l * H + g * H_p + j]]);
        all_max = std::max(all_max, mx);
        const int64_t list = ((int64_t)l * batch + b) * G + g;
        off[list + 1] = (mx + P - 1) / P;
      }
      mono += (all_max + P - 1) / P;
    }
  for (int64_t i = 0; i < n_lists; ++i) off[i + 1] += off[i];
  const int64_t total = off[n_lists];
  if (total > INT32_MAX) return fail(TG_ERR_CAPACITY, "tg_build_pages: %lld pages exceed int32 ids", (long long)total);

  if (n_pages) *n_pages = total;
  if (n_pages_monolithic) *n_pages_monolithic = mono;
  if (head_order) std::memcpy(head_order, order.data(), order.size() * sizeof(int32_t));
  if (ntok) std::memcpy(ntok, n.data(), n.size() * sizeof(int32_t));
  if (pt_off) std::memcpy(pt_off, off.data(), off.size() * sizeof(int64_t));
  if (Phi) {
    for (int l = 0; l < L; ++l)
      for (int g = 0; g < G; ++g) {
        int64_t s = 0;
        for (int b = 0; b < batch; ++b)
          for (int j = 0; j < H_p; ++j)
            s += n[((size_t)l * batch + b) * H + order[(size_t)l * H + g * H_p + j]];
        Phi[(size_t)l * G + g] = s;
      }
  }
  if (pt_ids) {
    if (pt_cap < total)
      return fail(TG_ERR_CAPACITY, "tg_build_pages: pt_cap=%lld < %lld pages", (long long)pt_cap, (long long)total);
    // ids in request-arrival order: (b, l, g, page)
    int32_t next = 0;
    for (int b = 0; b < batch; ++b)
      for (int l = 0; l < L; ++l)
        for (int g = 0; g < G; ++g) {
          const int64_t list = ((int64_t)l * batch + b) * G + g;
          for (int64_t p = off[list]; p < off[list + 1]; ++p) pt_ids[p] = next++;
        }
  }
  return tgi::ok();
}

namespace {
// One row of the split map (section 3.3, Algorithm 1): one CTA per group, then
// the rest by largest remainder, ties to the lower group.
void split_row(int G, int N_CTA, const int64_t *Phi, int32_t *S) {
  int64_t tot = 0;
  for (int i = 0; i < G; ++i) tot += Phi[i];
  std::vector<int64_t> w(Phi, Phi + G);
  if (tot == 0) {
    std::fill(w.begin(), w.end(), 1);
    tot = G;
  }
  const int64_t R = N_CTA - G;
  std::vector<int64_t> fl(G), rem(G);
  int64_t used = 0;
  for (int i = 0; i < G; ++i) {
    unsigned __int128 prod = (unsigned __int128)R * (uint64_t)w[i];
    fl[i] = (int64_t)(prod / (uint64_t)tot);
    rem[i] = (int64_t)(prod % (uint64_t)tot);
    used += fl[i];
  }
  std::vector<int> idx(G);
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int c) { return rem[a] > rem[c]; });
  for (int i = 0; i < G; ++i) S[i] = (int32_t)(1 + fl[i]);
  for (int64_t k = 0; k < R - used; ++k) S[idx[k]] += 1;
}
}  // namespace

extern "C" int tg_split_map(int L, int G, int N_CTA, const int64_t *Phi, int32_t *S) {
  if (L <= 0 || G <= 0 || !Phi || !S) return fail(TG_ERR_INVALID_ARG, "tg_split_map: bad L=%d G=%d or NULL", L, G);
  if (N_CTA < G) return fail(TG_ERR_SHAPE, "tg_split_map: N_CTA=%d < G=%d (every group needs a CTA)", N_CTA, G);
  for (int i = 0; i < L * G; ++i)
    if (Phi[i] < 0) return fail(TG_ERR_INVALID_ARG, "tg_split_map: Phi[%d]=%lld < 0", i, (long long)Phi[i]);
  for (int l = 0; l < L; ++l) split_row(G, N_CTA, Phi + (size_t)l * G, S + (size_t)l * G);
  return tgi::ok();
}

extern "C" int tg_plan_decode(int L, int batch, int H, int H_q, int H_p, int P, int d, int N_CTA,
                              const int32_t *S, const int32_t *head_order, const int32_t *ntok,
                              void *plan, int64_t plan_cap, int64_t *plan_bytes, int64_t *workspace_bytes) {
  if (L <= 0 || batch <= 0 || H <= 0 || H_q <= 0 || H_p <= 0 || P <= 0 || N_CTA <= 0)
    return fail(TG_ERR_INVALID_ARG, "tg_plan_decode: sizes must be positive");
  if (!S || !head_order || !ntok) return fail(TG_ERR_INVALID_ARG, "tg_plan_decode: NULL S/head_order/ntok");
  if (H % H_p || H_q % H) return fail(TG_ERR_SHAPE, "tg_plan_decode: H %% H_p or H_q %% H is not 0");
  if (P % 16) return fail(TG_ERR_SHAPE, "tg_plan_decode: P=%d must be a multiple of 16", P);
  const int g = H_q / H, G = H / H_p;
  if (g > 8) return fail(TG_ERR_SHAPE, "tg_plan_decode: g=%d > 8 query heads per KV head", g);
  if (d != 128 && d != 256) return fail(TG_ERR_SHAPE, "tg_plan_decode: d=%d (128 or 256)", d);

  std::vector<std::vector<tg_work_item>> items(L);
  std::vector<std::vector<int32_t>> cta_off(L);
  std::vector<int32_t> slots(L, 0);
  for (int l = 0; l < L; ++l) {
    const int32_t *Sl = S + (size_t)l * G;
    int64_t sum = 0;
    for (int i = 0; i < G; ++i) {
      if (Sl[i] < 1) return fail(TG_ERR_INVALID_ARG, "tg_plan_decode: S[%d][%d]=%d < 1", l, i, Sl[i]);
      sum += Sl[i];
    }
    if (sum != N_CTA)
      return fail(TG_ERR_SHAPE, "tg_plan_decode: row %d of S sums to %lld, not N_CTA=%d", l, (long long)sum, N_CTA);
    std::vector<int32_t> seen(H, 0);
    for (int i = 0; i < H; ++i) {
      int32_t h = head_order[(size_t)l * H + i];
      if (h < 0 || h >= H || seen[h]++) return fail(TG_ERR_INVALID_ARG, "tg_plan_decode: head_order[%d] is not a permutation", l);
    }
    std::vector<std::vector<tg_work_item>> per_cta(N_CTA);
    int cta_base = 0;
    int32_t next_slot = 0;
    for (int grp = 0; grp < G; ++grp) {
      const int Sg = Sl[grp];
      // the group's runs, laid end to end in (request, head-in-group) order
      struct Run { int b, h, j; int64_t start, n; };
      std::vector<Run> runs;
      int64_t W = 0;
      for (int b = 0; b < batch; ++b)
        for (int j = 0; j < H_p; ++j) {
          int h = head_order[(size_t)l * H + grp * H_p + j];
          int64_t nn = ntok[((size_t)l * batch + b) * H + h];
          if (nn < 0) return fail(TG_ERR_INVALID_ARG, "tg_plan_decode: negative ntok");
          runs.push_back({b, h, j, W, nn});
          W += nn;
        }
      std::vector<int64_t> bound(Sg + 1);
      for (int c = 0; c <= Sg; ++c) bound[c] = (int64_t)((unsigned __int128)c * (uint64_t)W / (uint64_t)Sg);
      for (const Run &r : runs) {
        tg_work_item it;
        std::memset(&it, 0, sizeof it);
        it.b = r.b; it.h = r.h; it.hpos = r.j; it.g = grp;
        if (r.n == 0) {
          it.t0 = it.t1 = 0; it.slot0 = -1; it.part = 0; it.nparts = 1;
          per_cta[cta_base].push_back(it);
          continue;
        }
        // CTA c holds units [bound[c], bound[c+1]); find the first one that holds r.start
        int c = (int)(std::upper_bound(bound.begin(), bound.end(), r.start) - bound.begin()) - 1;
        std::vector<std::pair<int, std::pair<int64_t, int64_t>>> pieces;
        for (; c < Sg && bound[c] < r.start + r.n; ++c) {
          int64_t lo = std::max(bound[c], r.start), hi = std::min(bound[c + 1], r.start + r.n);
          if (lo < hi) pieces.push_back({c, {lo - r.start, hi - r.start}});
        }
        const int np = (int)pieces.size();
        for (int k = 0; k < np; ++k) {
          it.t0 = (int32_t)pieces[k].second.first;
          it.t1 = (int32_t)pieces[k].second.second;
          it.nparts = np;
          it.part = k;
          it.slot0 = np > 1 ? next_slot : -1;
          per_cta[cta_base + pieces[k].first].push_back(it);
        }
        if (np > 1) next_slot += np;
      }
      cta_base += Sg;
    }
    cta_off[l].resize(N_CTA + 1);
    cta_off[l][0] = 0;
    for (int c = 0; c < N_CTA; ++c) {
      cta_off[l][c + 1] = cta_off[l][c] + (int32_t)per_cta[c].size();
      items[l].insert(items[l].end(), per_cta[c].begin(), per_cta[c].end());
    }
    slots[l] = next_slot;
  }

  // serialise: header | layer table | per layer (cta_off, items)
  int64_t pos = tgi::align_up(sizeof(tg_plan_header), 16);
  const int64_t layers_at = pos;
  pos = tgi::align_up(pos + (int64_t)L * sizeof(tg_plan_layer), 16);
  std::vector<tg_plan_layer> lt(L);
  int32_t max_slots = 0;
  for (int l = 0; l < L; ++l) {
    lt[l].cta_off = pos;
    pos = tgi::align_up(pos + (int64_t)(N_CTA + 1) * 4, 16);
    lt[l].lead = pos;
    pos = tgi::align_up(pos + (int64_t)N_CTA * sizeof(tg_work_item), 16);
    lt[l].items = pos;
    lt[l].n_items = (int32_t)items[l].size();
    lt[l].n_slots = slots[l];
    pos = tgi::align_up(pos + (int64_t)items[l].size() * sizeof(tg_work_item), 16);
    max_slots = std::max(max_slots, slots[l]);
  }
  const tgi::WorkspaceLayout ws = tgi::workspace_layout(batch, H, g, d, max_slots);
  if (plan_bytes) *plan_bytes = pos;
  if (workspace_bytes) *workspace_bytes = ws.total;
  if (!plan) return tgi::ok();
  if (plan_cap < pos) return fail(TG_ERR_CAPACITY, "tg_plan_decode: plan_cap=%lld < %lld", (long long)plan_cap, (long long)pos);
  uint8_t *base = static_cast<uint8_t *>(plan);
  std::memset(base, 0, pos);
  tg_plan_header hd;
  std::memset(&hd, 0, sizeof hd);
  hd.magic = TG_PLAN_MAGIC;
  hd.version = TG_PLAN_VERSION;
  hd.L = L; hd.batch = batch; hd.H = H; hd.H_q = H_q; hd.H_p = H_p; hd.P = P; hd.d = d; hd.G = G;
  hd.N_CTA = N_CTA;
  hd.max_slots = max_slots;
  hd.plan_bytes = pos;
  hd.workspace_bytes = ws.total;
  hd.layers = layers_at;
  std::memcpy(base, &hd, sizeof hd);
  std::memcpy(base + layers_at, lt.data(), L * sizeof(tg_plan_layer));
  for (int l = 0; l < L; ++l) {
    std::memcpy(base + lt[l].cta_off, cta_off[l].data(), (N_CTA + 1) * 4);
    if (!items[l].empty())
      std::memcpy(base + lt[l].items, items[l].data(), items[l].size() * sizeof(tg_work_item));
    // each CTA's first item with its item count and index, at a fixed place
    tg_work_item *lead = reinterpret_cast<tg_work_item *>(base + lt[l].lead);
    for (int c = 0; c < N_CTA; ++c) {
      const int32_t n = cta_off[l][c + 1] - cta_off[l][c];
      if (n > 0) lead[c] = items[l][cta_off[l][c]];
      lead[c].reserved[0] = n;
      lead[c].reserved[1] = cta_off[l][c];
      lead[c].reserved[2] = 0;
    }
  }
  return tgi::ok();
}

// ---------------------------------------------------------------------------
// Stability-aware rerank schedule ("FlexiCache ... (MLSys 2026)", paper-review
// page, "Core method / Tiered KV placement" and "Stability-aware rerank
// frequency"): an unstable head is re-scored every decode step; a stable head
// only every `period` steps, request b at the steps where (step + b * stagger)
// % period == 0.  Rows are (b, h) -> b * H + h, listed by b then h.
extern "C" int tg_rerank_rows(int L, int batch, int H, const uint8_t *unstable, int layer, int step, int period,
                              int stagger, int32_t *rows, int32_t *n_rows) {
  if (L <= 0 || batch < 0 || H <= 0 || period <= 0 || step < 0 || (stagger != 0 && stagger != 1))
    return fail(TG_ERR_INVALID_ARG, "tg_rerank_rows: bad L/batch/H/step/period/stagger");
  if (layer < 0 || layer >= L) return fail(TG_ERR_INVALID_ARG, "tg_rerank_rows: layer %d of %d", layer, L);
  if (!unstable || !n_rows || (!rows && batch > 0)) return fail(TG_ERR_INVALID_ARG, "tg_rerank_rows: NULL argument");
  int32_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const bool stable_due = ((int64_t)step + (int64_t)b * stagger) % period == 0;
    for (int h = 0; h < H; ++h)
      if (unstable[(size_t)layer * H + h] || stable_due) rows[n++] = b * H + h;
  }
  *n_rows = n;
  return tgi::ok();
}

extern "C" int tg_plan_set_flags(void *plan_host, uint32_t flags) {
  if (!plan_host) return fail(TG_ERR_INVALID_ARG, "tg_plan_set_flags: NULL plan");
  tg_plan_header *hd = static_cast<tg_plan_header *>(plan_host);
  if (hd->magic != TG_PLAN_MAGIC || hd->version != TG_PLAN_VERSION)
    return fail(TG_ERR_INVALID_ARG, "tg_plan_set_flags: not a tg_plan_decode buffer");
  if (flags & ~TG_PLAN_WAIT_TABLES) return fail(TG_ERR_INVALID_ARG, "tg_plan_set_flags: unknown flags 0x%x", flags);
  hd->flags = flags;
  return tgi::ok();
}
