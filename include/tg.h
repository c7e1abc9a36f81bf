/*
 * tg.h -- C ABI of the GB300 ragged paged decode-attention library.
 *
 * Decode attention over a head-wise non-uniform ("ragged") KV cache, after
 *   [Tangram] "Tangram: Unlocking Non-Uniform KV Cache Compression for
 *             Efficient Multi-turn LLM Serving" (paper-review page), section 3
 *             (3.1 Budget Reservation, 3.2 Ragged Paging, 3.3 AOT Load Balancing);
 * and Quest-style page scoring with per-KV-head top-K pages, after
 *   [FlexiCache] "FlexiCache: Leveraging Temporal Stability of Attention Heads
 *             for Efficient KV Cache Management (MLSys 2026)" (paper-review page),
 *             "Core method / Sparse decode" and "Assumption 2".
 *
 * Conventions
 *  - Every function returns TG_OK (0) or a negative TG_ERR_* code; the
 *    calling thread's tg_last_error_string() then says why.  No C++ exception
 *    crosses this boundary.
 *  - The caller owns every buffer.  "host" pointers are ordinary CPU memory,
 *    "device" pointers are CUDA device memory of the current device.  Nothing
 *    is allocated on the caller's behalf; sizes are queried first (size
 *    outputs, or NULL data outputs).
 *  - GPU entry points take a CUDA stream (cudaStream_t; NULL = legacy default
 *    stream), validate their arguments on the host and return synchronously,
 *    then run asynchronously on that stream.  Faults that only the device can
 *    see (a page id past the pool, a NaN score, a wait that gave up) set bits
 *    of the caller's int32 device status word (TG_STATUS_*), which
 *    tg_check_status() reads back.  No kernel traps.
 *  - GPU entry points only enqueue work on the caller's stream: no host
 *    synchronisation, no allocation.  They may be captured in a CUDA graph and
 *    replayed (bit-identical to eager calls); tg_sparse_layer's epoch needs the
 *    care its entry states.  tg_check_status() synchronises and is not captured.
 *    Independent callers on concurrent streams need their own workspaces and
 *    status words; the library keeps no other state between calls (except the
 *    fixed array of tg_decode_attn_static_scratch).
 *  - Tensors are dense row-major.  bf16 values travel as uint16_t bit patterns.
 *
 * Notation: L layers, batch requests, H KV heads, H_q query heads, g = H_q/H
 * (query head j reads KV head j/g), d head dim, P tokens per page, H_p heads
 * per page group, G = H/H_p groups, N_b context length of request b,
 * n_{l,b,h} = ceil(B_{l,h} * N_b) retained tokens of a head.
 */
#ifndef TG_H
#define TG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *tg_stream_t;   /* same type as cudaStream_t */

enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = -1, /* a NULL pointer, a non-positive size, a bad flag   */
  TG_ERR_SHAPE = -2,       /* sizes that do not fit together (H % H_p, d, g...) */
  TG_ERR_NONFINITE = -3,   /* NaN/Inf in a host input that must be finite       */
  TG_ERR_CAPACITY = -4,    /* an output buffer is too small                     */
  TG_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed                 */
  TG_ERR_TIMEOUT = -6,     /* reported by tg_check_status for TG_STATUS_TIMEOUT */
  TG_ERR_DEVICE = -7       /* reported by tg_check_status for other status bits */
};

/* Bits of the device status word. */
#define TG_STATUS_NONFINITE 0x1 /* a NaN score reached a top-k selection            */
#define TG_STATUS_BAD_PAGE 0x2  /* a page id outside [0, pool_pages)                */
#define TG_STATUS_TIMEOUT 0x4   /* a copy wait gave up (about 2 s); outputs invalid */
#define TG_STATUS_BAD_INPUT 0x8 /* a device-side size outside its limits            */

/* Reason for the last non-zero return on the calling thread ("" if none). */
const char *tg_last_error_string(void);

/* Library version: 10000 * major + 100 * minor + patch. */
int tg_version(void);

/* ------------------------------------------------------------------ a1 ---
 * tg_build_pages -- ragged page tables with budget-aware head clustering.
 *   [Tangram] 3.1: B = min(1, alpha * B^) with safety coefficient alpha;
 *   n = ceil(B * N_b), the size of Top(ceil(B N), s).  3.2: H_p-head groups,
 *   one page table per group, a page holds H_p x 2 x P x d elements, a group
 *   gets ceil(max_{h in group} n / P) pages; budget-aware clustering puts heads
 *   of similar retention in one group.  3.3: Phi = aggregate budget of a group.
 * Readings: B is float32; n is the exact ceiling of that float32 times N_b,
 *   clamped to [1, N_b] (0 when N_b = 0).  cluster != 0 sorts each layer's
 *   heads by (B descending, head ascending) and cuts the order into chunks of
 *   H_p; cluster == 0 keeps heads i*H_p .. i*H_p+H_p-1 in group i.  Page ids
 *   are numbered from 0 in (request, layer, group, page) order.
 * Inputs (host): Bhat float32 [L][H], each > 0 and finite; N int32 [batch],
 *   each >= 0; alpha > 0; H % H_p == 0; P % 16 == 0.
 * Outputs (host, each may be NULL):
 *   head_order int32 [L][H]  group i holds head_order[l][i*H_p + j], j < H_p
 *   ntok       int32 [L][batch][H]
 *   Phi        int64 [L][G]  sum of ntok over the requests and heads of a group
 *   pt_off     int64 [L*batch*G + 1]  CSR offsets; list (l, b, g) is index (l*batch + b)*G + g
 *   pt_ids     int32 [pt_cap]  page ids; TG_ERR_CAPACITY if pt_cap < *n_pages
 *   n_pages             total ragged pages
 *   n_pages_monolithic  pages (of H x 2 x P x d elements) one shared table would need
 * Pool layout implied: pool bf16 [n_pages][H_p][2][P][d]; retained token k of the
 *   head at group position j sits in page pt_ids[pt_off[list] + k/P], row k%P of
 *   block [j][0] (K) and [j][1] (V).
 */
int tg_build_pages(int L, int batch, int H, int H_p, int P, float alpha,
                   const float *Bhat, const int32_t *N, int cluster,
                   int32_t *head_order, int32_t *ntok, int64_t *Phi,
                   int64_t *pt_off, int32_t *pt_ids, int64_t pt_cap,
                   int64_t *n_pages, int64_t *n_pages_monolithic);

/* ------------------------------------------------------------------ a3 ---
 * tg_split_map -- the static Workload Split Map S in N^{L x G}.
 *   [Tangram] 3.3 (Algorithm 1): CTAs are given to each head group in
 *   proportion to its aggregate budget Phi_{l,i}; larger groups get more CTAs.
 * Reading: per layer row, every group gets 1 CTA, then R = N_CTA - G more by
 *   largest remainder of R*Phi_i/sum(Phi), ties to the lower group index; a
 *   row of zeros counts as equal Phi.  Each row sums to N_CTA.
 * Inputs (host): Phi int64 [L][G], each >= 0; N_CTA >= G.
 * Output (host): S int32 [L][G].
 */
int tg_split_map(int L, int G, int N_CTA, const int64_t *Phi, int32_t *S);

/* tg_query_ncta -- occupancy-derived N_CTA for tg_decode_attn on the current
 *   device: resident CTAs per SM of the kernel chosen for (d, g) times the SM
 *   count ([Tangram] 3.3, N_CTA from the CUDA max-occupancy query).
 *   d in {128, 256}, 1 <= g <= 8.  Output (host): *N_CTA. */
int tg_query_ncta(int d, int g, int *N_CTA);

/* ------------------------------------------------------------------ a4 ---
 * Decode plan: the split map turned into per-CTA work ([Tangram] 3.3: each
 * group's CTAs share its work evenly).  Inside group i of layer l the retained
 * tokens are laid end to end in (request, head-in-group, token) order, W =
 * Phi_{l,i} units; CTA j of the group's S_{l,i} CTAs takes units
 * [floor(j W / S), floor((j+1) W / S)).  Each piece of one head's run is one
 * tg_work_item.  A plan is a single self-describing byte buffer:
 *   tg_plan_header | tg_plan_layer[L] | per layer: int32 cta_off[N_CTA+1],
 *   tg_work_item lead[N_CTA], tg_work_item items[]
 * (every section 16-byte aligned; offsets are in bytes from the buffer start).
 * lead[c] is a copy of CTA c's first item (zeros when it has none) whose
 * reserved[0] holds the CTA's item count and reserved[1] the index of that first
 * item in items[]: a CTA finds its first item and its count at a fixed place, in
 * one load, without reading cta_off first. */
#define TG_PLAN_MAGIC 0x31504754u /* "TGP1" */
#define TG_PLAN_VERSION 3

/* Plan flag: each tg_decode_attn launch of this plan waits for the previous
 * kernel in the stream to complete before it reads q, pt_off or pt_ids (it
 * still starts early and reads the plan).  Set it when that kernel writes them
 * and lets the next kernel start early, as tg_page_score_topk does with
 * TG_SCORE_LET_NEXT_START. */
#define TG_PLAN_WAIT_TABLES 0x1u

typedef struct tg_plan_header {
  uint32_t magic;
  int32_t version;
  int32_t L, batch, H, H_q, H_p, P, d, G, N_CTA;
  int32_t max_slots;       /* most partial slots any layer uses */
  uint32_t flags;          /* TG_PLAN_* (tg_plan_set_flags); 0 from tg_plan_decode */
  int32_t reserved;
  int64_t plan_bytes;      /* size of the whole buffer */
  int64_t workspace_bytes; /* device workspace tg_decode_attn needs */
  int64_t layers;          /* byte offset of tg_plan_layer[L] */
} tg_plan_header;

typedef struct tg_plan_layer {
  int64_t cta_off; /* byte offset of int32 [N_CTA + 1]: items of CTA c are [cta_off[c], cta_off[c+1]) */
  int64_t lead;    /* byte offset of tg_work_item [N_CTA]: each CTA's first item, count and index */
  int64_t items;   /* byte offset of tg_work_item [n_items] */
  int32_t n_items;
  int32_t n_slots; /* partial slots of this layer */
} tg_plan_layer;

typedef struct tg_work_item {
  int32_t b, h;    /* request, KV head */
  int32_t hpos, g; /* position of h in its group, group index */
  int32_t t0, t1;  /* retained-token range [t0, t1) of (b, h); t0 == t1 only for an empty head */
  int32_t slot0;   /* first partial slot of the run of (b, h) (when nparts > 1) */
  int32_t part;    /* this CTA's piece of the run, 0 .. nparts-1 */
  int32_t nparts;  /* CTAs that share the run; 1 = this CTA finishes it alone */
  int32_t reserved[3]; /* 0 in items[]; in lead[]: item count, first item's index, 0 */
} tg_work_item;

/* tg_plan_decode -- build the plan for all L layers.
 * Inputs (host): S int32 [L][G] (tg_split_map), head_order int32 [L][H] and
 *   ntok int32 [L][batch][H] (tg_build_pages).  N_CTA = each row's sum.
 *   d in {128, 256}; g = H_q / H in [1, 8]; P % 16 == 0.
 * Outputs (host): plan (NULL to query the size) of plan_cap bytes;
 *   *plan_bytes; *workspace_bytes = device scratch tg_decode_attn needs.
 *   TG_ERR_CAPACITY if plan_cap < *plan_bytes. */
int tg_plan_decode(int L, int batch, int H, int H_q, int H_p, int P, int d, int N_CTA,
                   const int32_t *S, const int32_t *head_order, const int32_t *ntok,
                   void *plan, int64_t plan_cap, int64_t *plan_bytes, int64_t *workspace_bytes);

/* tg_plan_set_flags -- set the TG_PLAN_* flags of a plan (host buffer; the
 *   device copy needs no update: only the host launch reads them). */
int tg_plan_set_flags(void *plan_host, uint32_t flags);

/* ------------------------------------------------------------- a5 + a6 ---
 * tg_decode_attn -- split-KV flash decoding of one layer over the ragged pool,
 *   with the log-sum-exp merge fused in (the last CTA of a shared run merges).
 *   [Tangram] 3.3: one launch of N_CTA CTAs per layer under the static split
 *   map, no re-planning.  [FlexiCache] "Sparse decode": the same kernel runs
 *   over a per-head list of selected pages (H_p = 1 tables).
 *   For query head j = h*g + i of request b:
 *     out = sum_t softmax_t(scale * q . k_t) v_t over the retained tokens t of (b, h),
 *     lse = ln sum_t exp(scale * q . k_t)     (out = 0, lse = -inf for an empty head).
 *   bf16 inputs, float32 accumulation, bf16 output.
 * Arguments:
 *   plan_host / plan_dev  the same tg_plan_decode bytes in host and device memory
 *   layer                 which plan layer to run (0 <= layer < L)
 *   q     device bf16 [batch][H_q][d]
 *   pool  device bf16 [pool_pages][H_p][2][P][d]; 16-byte aligned.  Rows of a
 *         head's last page past its ntok must hold finite values
 *         (tg_compact_topk writes zeros there).
 *   pt_off device int64: the page-table offsets of THIS layer's lists,
 *         batch*G + 1 entries, list b*G + g; values index pt_ids
 *   pt_ids device int32 page ids
 *   scale  softmax scale (1/sqrt(d) for standard attention)
 *   workspace device, workspace_bytes >= the plan's; zero-filled before the
 *         first call.  The kernel returns its counters to zero, so one buffer
 *         serves every later call on the same stream; concurrent calls must
 *         use separate workspaces.  After a TG_STATUS_TIMEOUT, zero it again.
 *   out   device bf16 [batch][H_q][d];  lse device float32 [batch][H_q] (may be NULL)
 *   dev_status device int32, OR-ed with TG_STATUS_* (may be NULL)
 *   cta_time device int64 [2*N_CTA] (may be NULL): %globaltimer ns at each
 *         CTA's start and end, for CTA skew = max/mean of (end - start).
 * Launch: programmatic dependent launch.  The kernel lets the next kernel in
 *   the stream start as its CTAs finish, and it may itself start while the
 *   previous tg_decode_attn launch in the stream is finishing: before waiting
 *   for that launch it reads the plan, page tables, pool and q (never written
 *   by a decode launch); it waits before it touches the workspace, out or lse.
 *   Other kernels complete before it starts, unless they let it start early
 *   (tg_page_score_topk with TG_SCORE_LET_NEXT_START): the plan must then carry
 *   TG_PLAN_WAIT_TABLES, and the launch waits before it reads q and the tables.
 *   Such a launch lets the next kernel start only after that wait, when the
 *   kernel that wrote the tables is complete: a page-score call that follows
 *   it on the same score workspace cannot overlap the one before it. */
int tg_decode_attn(tg_stream_t stream, const void *plan_host, const void *plan_dev, int layer,
                   const uint16_t *q, const uint16_t *pool, int64_t pool_pages,
                   const int64_t *pt_off, const int32_t *pt_ids, float scale,
                   void *workspace, int64_t workspace_bytes,
                   uint16_t *out, float *lse, int32_t *dev_status, int64_t *cta_time);

/* ------------------------------------------------------------------ a2 ---
 * tg_compact_topk -- retain Top(n, s) of every head of one layer and write the
 *   retained K/V rows into the group pages.
 *   [Tangram] 3.1: I_{l,h} = Top(ceil(B_{l,h} N), s_{l,h}); 3.2: per-group pages.
 * Reading: ties go to the lower token index, -0.0 == +0.0; retained tokens
 *   are stored in ascending token order (token I[k] -> page k/P, row k%P).
 *   The rows of a head's last page past n are zero-filled.  A NaN score sets
 *   TG_STATUS_NONFINITE (the selection of that row is then unspecified).
 * Arguments (device unless stated):
 *   N int32 [batch] with N_b <= Nmax; scores float32 [batch][H][Nmax];
 *   K, V bf16 [batch][H][Nmax][d]; head_order int32 [H] and ntok int32 [batch][H]
 *   of this layer; pt_off int64 [batch*G + 1] of this layer's lists; pt_ids int32;
 *   pool bf16 [pool_pages][H_p][2][P][d] (output, 16-byte aligned);
 *   kept_idx int32 [batch][H][Nmax] (output, may be NULL): row (b, h) starts with
 *   the n retained token indices, ascending;
 *   workspace: scratch of at least tg_compact_topk_workspace(batch, H, Nmax) bytes,
 *   4-byte aligned, no initial contents needed (the call writes every entry it
 *   reads: each row's n-th largest key, and per block of 1024 positions the keys
 *   above it and equal to it before the block); concurrent calls need separate
 *   workspaces; TG_ERR_CAPACITY if it is smaller; dev_status may be NULL.
 *   Host sizes: d % 8 == 0, d <= 512, P % 16 == 0, Nmax >= 1.
 * Launches two kernels on `stream`: a select kernel of one thread-block cluster per
 *   row, and the copy kernel as its programmatic dependent. */
int tg_compact_topk(tg_stream_t stream, int batch, int H, int H_p, int P, int d, int Nmax,
                    const int32_t *N, const float *scores, const uint16_t *K, const uint16_t *V,
                    const int32_t *head_order, const int32_t *ntok, const int64_t *pt_off,
                    const int32_t *pt_ids, int64_t pool_pages, uint16_t *pool,
                    int32_t *kept_idx, void *workspace, int64_t workspace_bytes, int32_t *dev_status);

/* tg_compact_topk_workspace -- bytes of workspace tg_compact_topk needs:
 *   batch * H * (4 + 2 * ceil(Nmax / 1024)) * 4. */
int tg_compact_topk_workspace(int batch, int H, int Nmax, int64_t *workspace_bytes);

/* ------------------------------------------------------------------ f1 ---
 * tg_compact_chunk -- retention fused into chunked prefill: after each chunk of
 *   C tokens, every head's n = ntok[b][h] reserved slots hold the best n tokens
 *   seen so far (score descending, token ascending), so after the last chunk
 *   they hold exactly Top(n, s) (a token's score is fixed once its chunk is
 *   computed).  [Tangram] 3.1: compression runs inside chunked prefill; section 4
 *   "Compression Fusion into Prefill".
 *   Call it once per chunk, chunk_start = 0, C, 2C, ... (N[b] is the request's
 *   full prompt length; tokens past it are ignored).  While a head's slots are
 *   not full the chunk's tokens are appended; afterwards a slot whose token drops
 *   out is reused: the lowest freed slot takes the lowest entering token, and only
 *   entering tokens' K/V rows are written.  Slot k is page k/P, row k%P of the
 *   head's block (as tg_compact_topk), so tg_decode_attn reads the result
 *   unchanged; the tokens are in slot order, not ascending.
 * Arguments (device): scores float32 [batch][H][C], K, V bf16 [batch][H][C][d]
 *   (this chunk); head_order, ntok, pt_off, pt_ids, pool as tg_compact_topk;
 *   slot_tok int32 and slot_key uint32 [batch][H][nmax] (state, nmax >= every
 *   n; slot_tok[..][k] = the token in slot k).  C <= 8192; the first chunk also
 *   zeroes the rows of each head's last page past n.
 *   workspace: device scratch of at least tg_compact_chunk_workspace(batch, H, C)
 *   bytes, 16-byte aligned, no initial contents; one per stream (a call overwrites it).
 * Launch: a ranking kernel (one CTA per head) writes the slots and, for each head
 *   whose slots are full, its list of (slot, chunk position) entries; a copy kernel
 *   spread over the GPU (programmatic dependent launch) copies the entering K/V
 *   rows.  It copies the heads whose slots are still filling (chunk position i to
 *   slot filled + i) before it waits for the ranking kernel. */
int tg_compact_chunk(tg_stream_t stream, int batch, int H, int H_p, int P, int d, int chunk_start, int C,
                     const int32_t *N, const float *scores, const uint16_t *K, const uint16_t *V,
                     const int32_t *head_order, const int32_t *ntok, const int64_t *pt_off,
                     const int32_t *pt_ids, int64_t pool_pages, uint16_t *pool, int32_t *slot_tok,
                     uint32_t *slot_key, int nmax, void *workspace, int64_t workspace_bytes,
                     int32_t *dev_status);

/* tg_compact_chunk_workspace -- bytes of workspace tg_compact_chunk needs for
 *   batch * H heads and chunks of C tokens (host; TG_ERR_INVALID_ARG on bad sizes). */
int tg_compact_chunk_workspace(int batch, int H, int C, int64_t *workspace_bytes);

/* ------------------------------------------------------------------ a9 ---
 * tg_build_minmax -- per-page elementwise min and max of the keys (the MinMax
 *   cache of [FlexiCache] "Assumption 2"), exact in bf16.
 *   K device bf16 [batch][H][N][d]; minmax device bf16 [batch][H][ceil(N/P)][2][d]
 *   (row 0 = min, row 1 = max over the page's valid keys). */
int tg_build_minmax(tg_stream_t stream, int batch, int H, int N, int P, int d,
                    const uint16_t *K, uint16_t *minmax, int32_t *dev_status);

/* ------------------------------------------------------------------ a7 ---
 * tg_page_score_topk -- Quest page bound and per-KV-head top-K pages.
 *   [FlexiCache] "Core method / Sparse decode": every KV head attends only to
 *   its top-K pages, ranked by the min-max key bound of max q.k.
 *   score(b,h,p) = max over the g query heads j of sum_d max(q_jd mn_pd, q_jd mx_pd).
 * Reading: float32 arithmetic in one fixed order (d cut into 16 slices summed
 *   left to right, then partial sums added pairwise (j, j+8), (j, j+4), (j, j+2),
 *   (j, j+1)); ties to the lower page; output ascending.  A NaN sum in any
 *   query head sets TG_STATUS_NONFINITE (the selection is then unspecified).
 * Arguments (device): q bf16 [batch][H*g][d]; minmax bf16 [batch][H][n_pages][2][d];
 *   sel int32 [batch][H][K] (output, page indices 0..n_pages-1);
 *   pt_ids int32 [batch][H][K] (output, may be NULL): (b*H + h)*n_pages + sel,
 *   i.e. the ids of the selected pages in a dense pool [batch][H][n_pages] of
 *   H_p = 1 pages, ready as the page lists of tg_decode_attn;
 *   workspace: scratch of at least tg_page_score_workspace bytes (page scores and
 *   one page counter per (request, KV head)); zero-filled before the first call.
 *   Each call returns the counters to zero, so one workspace serves every later
 *   call on the same stream; concurrent calls need separate workspaces.  After a
 *   TG_STATUS_TIMEOUT, zero it again.  q, minmax and workspace 16-byte aligned.
 *   Host sizes: d in {128, 256}, 1 <= g <= 8, 1 <= K <= n_pages <= 16384.
 * Launch: the score kernel streams every page of the call, evenly split over
 *   one CTA per SM.  With n_pages <= 1024 the warp that scores the last page of
 *   a (request, KV head) selects its top K in the same kernel; longer rows are
 *   selected by a second kernel.  Programmatic dependent launch: the call may
 *   start while the previous kernel in the stream (a tg_decode_attn of the
 *   previous layer) finishes, reading q and minmax and writing only the
 *   workspace; it waits for that kernel before writing sel and pt_ids.
 *   flags: 0, or TG_SCORE_LET_NEXT_START to let the next kernel in the stream
 *   start before sel and pt_ids are complete; that kernel must then wait for
 *   this one before reading them, and let no later kernel start before that
 *   wait, since the next call on the same workspace writes it as soon as it
 *   starts (tg_decode_attn with a plan flagged TG_PLAN_WAIT_TABLES does both).
 *   Without the flag the next kernel starts only when sel and pt_ids are
 *   complete. */
#define TG_SCORE_LET_NEXT_START 0x1u
int tg_page_score_topk(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                       const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
                       void *workspace, int64_t workspace_bytes, uint32_t flags, int32_t *dev_status);

/* tg_page_score_topk_rows -- tg_page_score_topk restricted to a list of rows.
 *   [FlexiCache] "Stability-aware rerank frequency": only the heads due for a
 *   rerank are scored; every other row keeps its previous sel / pt_ids.
 *   rows: device int32 [n_rows], distinct row numbers b*H + h in [0, batch*H)
 *   (an entry outside that range sets TG_STATUS_BAD_INPUT and is skipped).
 *   n_rows = 0 launches nothing.  dense_base (device int64 [batch*H], may be NULL)
 *   gives each row's page-id base: pt_ids[r][k] = dense_base[r] + sel[r][k]
 *   (NULL: r*n_pages, as tg_page_score_topk).  Everything else as
 *   tg_page_score_topk, with sel / pt_ids still indexed by row (only the listed
 *   rows are written). */
int tg_page_score_topk_rows(tg_stream_t stream, int batch, int H, int g, int d, int n_pages, int K,
                            int n_rows, const int32_t *rows, const uint16_t *q, const uint16_t *minmax,
                            int32_t *sel, int32_t *pt_ids, const int64_t *dense_base, void *workspace,
                            int64_t workspace_bytes, uint32_t flags, int32_t *dev_status);

/* tg_rerank_rows -- the rows of one layer due for a rerank at a decode step (host).
 *   [FlexiCache] "Core method" (stable heads re-ranked every 16 steps, unstable
 *   heads every step; all-stable layers skip scoring).
 *   unstable uint8 [L][H] (1 = unstable).  Row b*H + h is listed when head h of
 *   the layer is unstable, or when (step + b*stagger) % period == 0 (stagger 0:
 *   every request's stable heads together, so an all-stable layer has no rows at
 *   15 of 16 steps; stagger 1: one request phase per step).  rows (host, capacity
 *   batch*H) in (b, h) order; *n_rows = the count (0: skip the layer). */
int tg_rerank_rows(int L, int batch, int H, const uint8_t *unstable, int layer, int step, int period,
                   int stagger, int32_t *rows, int32_t *n_rows);

/* tg_sparse_layer -- one sparse decode layer (a7 + a8) in one persistent kernel:
 *   Quest scores and top-K pages of the re-ranked (request, KV head) rows, then
 *   flash decoding over every row's selected pages.  [FlexiCache] "Core method /
 *   Sparse decode" and "Stability-aware rerank frequency".
 *   A cooperative launch of the plan's N_CTA CTAs (all resident): each scores its
 *   share of the re-ranked rows' pages, the warp completing a row selects it and
 *   raises the row's ready flag (in score_ws) to `epoch`; then each CTA waits for
 *   the re-ranked rows of its work items (at most wait_limit_ns each, 0 = about
 *   2 s; then TG_STATUS_TIMEOUT, and the rows it gave up on decode whatever page
 *   lists they hold) and decodes them.  Results are those of
 *   tg_page_score_topk_rows followed by tg_decode_attn, bit for bit.
 * Arguments: plan as tg_decode_attn, built for d = 128 and H_p = 1 page lists of
 *   K pages per (request, KV head) (pt_off = 0, K, 2K, ...); the plan's N_CTA must
 *   not exceed the CTAs that can be resident together (tg_query_ncta gives it).
 *   rows (device int32 [n_rows], b*H + h) and due (device uint8 [batch*H]): the
 *   rows re-ranked by this call and, for the decode phase, which rows to wait
 *   for (1) -- every listed row, and no other.  NULL rows: every row is
 *   re-ranked (due unused).  A row not re-ranked keeps the page list an earlier
 *   call wrote.  A row marked due that the list omits is never raised: its wait
 *   runs out (TG_STATUS_TIMEOUT) and its output is unspecified.
 *   q, minmax, sel, pt_ids, score_ws (tg_page_score_workspace bytes, zero-filled
 *   before the first call) as tg_page_score_topk, n_pages <= 1024; pt_ids doubles
 *   as the decode's page lists over pool (the dense cache [batch][H][n_pages] of
 *   H_p = 1 pages).  epoch >= 1 and above every earlier call's on the same score
 *   workspace (e.g. a call counter).  workspace, out, lse, dev_status as
 *   tg_decode_attn.  Launched without programmatic dependent launch.
 *   CUDA graphs: a captured call replays the epoch it was captured with, so
 *   zero score_ws ahead of it in the same graph (a captured memset) or replay
 *   two graphs captured with different epochs in turn. */
int tg_sparse_layer(tg_stream_t stream, const void *plan_host, const void *plan_dev, int n_pages, int K,
                    int n_rows, const int32_t *rows, const uint8_t *due, int64_t wait_limit_ns,
                    const uint16_t *q, const uint16_t *minmax, int32_t *sel, int32_t *pt_ids,
                    void *score_ws, int64_t score_ws_bytes, int epoch, const uint16_t *pool,
                    int64_t pool_pages, const int64_t *pt_off, float scale, void *workspace,
                    int64_t workspace_bytes, uint16_t *out, float *lse, int32_t *dev_status);

/* tg_page_score_workspace -- bytes of workspace tg_page_score_topk needs for
 *   batch x H rows of n_pages pages (host only). */
int tg_page_score_workspace(int batch, int H, int n_pages, int64_t *workspace_bytes);

/* tg_decode_attn_static_scratch -- tg_decode_attn without a caller workspace.
 *   The pages have no counterpart of this call: it exists for callers that
 *   cannot allocate device memory at call time (a serving process whose own
 *   allocator has reserved the GPU heap up front, a plug-in running inside a
 *   host framework that owns all device memory).  It computes exactly what
 *   tg_decode_attn computes and takes the same arguments except the workspace:
 *   its scratch is a fixed 4 MiB array inside this library, present on every
 *   GPU that loads the library until the process exits.  Nothing is
 *   allocated at call time (no cudaMalloc, no cudaFree, no allocating library
 *   call).
 *   - Plans whose workspace_bytes exceed 4 MiB are rejected with
 *     TG_ERR_CAPACITY (use tg_decode_attn with a workspace then).
 *   - dev_status is required (NULL is TG_ERR_INVALID_ARG): device faults are
 *     reported only there.
 *   - Under CUDA's lazy module loading (the default) the array is loaded with
 *     this library's module on the first call on a device.  A caller that
 *     reserves the GPU heap for its own allocator should make one call first
 *     (or run with CUDA_MODULE_LOADING=EAGER).
 *   - The array's address is looked up (cudaGetSymbolAddress) on the first
 *     call in each CUDA context and cached under the context's id, so a call
 *     after a device reset or from another context looks it up again; make
 *     the first call in a context before any stream capture.
 *   - Each call clears the array's merge counters on `stream` before the
 *     kernel.  All calls share the one array, so calls whose kernels may
 *     overlap on the GPU (different streams or host threads) race on it and
 *     must be serialised by the caller. */
int tg_decode_attn_static_scratch(tg_stream_t stream, const void *plan_host, const void *plan_dev, int layer,
                                  const uint16_t *q, const uint16_t *pool, int64_t pool_pages,
                                  const int64_t *pt_off, const int32_t *pt_ids, float scale,
                                  uint16_t *out, float *lse, int32_t *dev_status, int64_t *cta_time);

/* ------------------------------------------------------------------ f4 ---
 * tg_tier_promote -- tiered KV placement: fetch newly promoted pages of stable
 *   heads from host memory into GPU blocks freed in place, and build the decode
 *   lists.  [FlexiCache] "Core method / Tiered KV placement" (a stable head keeps
 *   only its top-K pages on the GPU, the rest in host memory; a rerank moves only
 *   the newly promoted pages), "Block Allocator" (blocks reclaimed and reassigned
 *   in place at rerank) and "KV transfer" (a kernel reads pinned host KV through
 *   unified addressing).
 * For each listed row r = b*H + h (device int32 rows[n_rows]):
 *   unstable[h] != 0 (device uint8 [H] of this layer): every page is on the GPU;
 *     pt_ids[r][k] = dense_base[r] + sel[r][k].
 *   stable: the row owns the K blocks slot_block[r][0..K) (device int32) of pool;
 *     slot_page[r][k] (device int32, in/out) is the page block k holds, -1 none.
 *     Blocks whose page is not in sel[r] are freed; the pages of sel[r] not held
 *     by any block are copied from host_kv into them, the lowest such page into
 *     the lowest freed slot; pages already held are not touched.  Then
 *     pt_ids[r][k] = the block holding sel[r][k].
 *   sel int32 [batch*H][K], each row ascending, distinct pages in [0, n_pages)
 *   (tg_page_score_topk's output).  host_kv: host memory [batch*H][n_pages][page_bytes],
 *   pinned (read through its device mapping), or pageable on a device that reads
 *   pageable memory (cudaDevAttrPageableMemoryAccess, e.g. Grace over NVLink-C2C);
 *   anything else is TG_ERR_INVALID_ARG.  pool [pool_pages][page_bytes];
 *   both 16-byte aligned, page_bytes a multiple of 16.  promoted (device int64,
 *   may be NULL) is increased by the number of pages copied.  grid_limit > 0
 *   caps the CTAs (one row at a time each), for a low-priority background copy.
 *   A bad row or block sets TG_STATUS_BAD_INPUT / TG_STATUS_BAD_PAGE.
 *   Sizes: 1 <= K <= n_pages, n_pages <= 16384, K <= 1024.
 * A layout that satisfies these rules (the one the Python TieredSparseDecoder
 *   builds): the pool holds the unstable rows' dense regions first, then the
 *   stable rows' blocks.  With u(r) the rank of row r among the unstable rows
 *   and s(r) its rank among the stable rows (both in row order), n_u and n_s
 *   their counts: dense_base[r] = u(r) * n_pages for an unstable row;
 *   slot_block[r][k] = n_u * n_pages + s(r) * K + k for a stable row (-1 for an
 *   unstable one); pool_pages = n_u * n_pages + n_s * K. */
int tg_tier_promote(tg_stream_t stream, int n_rows, const int32_t *rows, int grid_limit,
                    const uint8_t *unstable, int batch, int H, int n_pages, int K, const int32_t *sel,
                    int32_t *slot_page, const int32_t *slot_block, const int64_t *dense_base,
                    const void *host_kv, int page_bytes, void *pool, int64_t pool_pages,
                    int32_t *pt_ids, int64_t *promoted, int32_t *dev_status);

/* tg_tier_promote_background -- tg_tier_promote (same arguments, same results) for a
 *   copy that runs on a low-priority stream while decoding continues on another:
 *   [FlexiCache] "FlexiCache Scheduler" (a reloading request pauses, the rest of the
 *   batch decodes) and "KV transfer" (a low-priority background stream, a limited
 *   grid).  Its CTAs have 64 threads, at most 64 registers each and 16 KB of shared
 *   memory, so one stays resident beside a decode or page-score CTA on the same SM
 *   instead of holding the SM while it waits on the host link.  The caller orders
 *   it after the scores of the rows it promotes (an event), and the decode of those
 *   rows after it. */
int tg_tier_promote_background(tg_stream_t stream, int n_rows, const int32_t *rows, int grid_limit,
                               const uint8_t *unstable, int batch, int H, int n_pages, int K,
                               const int32_t *sel, int32_t *slot_page, const int32_t *slot_block,
                               const int64_t *dense_base, const void *host_kv, int page_bytes, void *pool,
                               int64_t pool_pages, int32_t *pt_ids, int64_t *promoted, int32_t *dev_status);

/* ------------------------------------------------------------------ f2 ---
 * Page allocator for budget reservation.  [Tangram] 3.1 Budget Reservation: a
 * request's compressed footprint is fixed when it is scheduled, so its pages
 * are allocated once, with no runtime page reclamation; 3.2 Ragged Paging: one
 * page table per (layer, request, head group).  Host only; the state lives in
 * caller memory (tg_alloc_state_bytes), one allocator per pool.
 *   tg_alloc_init: n_pages free pages, handed out lowest id first.
 *   tg_alloc_admit: pages_per_list int32 [n_lists] (e.g. the per-list page counts
 *     of tg_build_pages for one request); all-or-nothing: on success ids int32
 *     [*n_ids] gets the pages list after list (ids_cap >= their sum), else
 *     TG_ERR_CAPACITY and nothing is taken.  *n_ids is set either way.
 *   tg_alloc_release: returns pages; released pages are reused last-in first-
 *     out.  A page not allocated, or listed twice, is TG_ERR_INVALID_ARG and
 *     nothing is released.
 *   tg_alloc_query: free and allocated page counts.
 * To place a request of tg_build_pages' tables: pass its lists (l, b, g), at
 *   pt_off index (l*batch + b)*G + g, in (layer, group) order as pages_per_list
 *   (pt_off[i+1] - pt_off[i] each); the returned ids then fill those lists in the
 *   same order, list after list (the Python RaggedCache does exactly this). */
int tg_alloc_state_bytes(int64_t n_pages, int64_t *bytes);
int tg_alloc_init(void *state, int64_t state_cap, int64_t n_pages);
int tg_alloc_admit(void *state, int n_lists, const int32_t *pages_per_list, int32_t *ids, int64_t ids_cap,
                   int64_t *n_ids);
int tg_alloc_release(void *state, int64_t n, const int32_t *ids);
int tg_alloc_query(const void *state, int64_t *n_free, int64_t *n_live);

/* tg_check_status -- synchronously read a device status word (waits for the
 *   device).  Returns TG_OK when it is 0, TG_ERR_TIMEOUT when TG_STATUS_TIMEOUT
 *   is set, TG_ERR_DEVICE for any other bit; *host_status (may be NULL) gets
 *   the raw bits. */
int tg_check_status(const int32_t *dev_status, int32_t *host_status);

#ifdef __cplusplus
}
#endif
#endif /* TG_H */
