/* A plain C99 program that drives the library through include/tg.h alone, with no Python
 * and no PyTorch: it builds the ragged page tables, the split map and the decode plan of
 * one layer on the host and, given "gpu", retains each head's top tokens into the pool
 * (tg_compact_topk) and runs decode attention over them (tg_decode_attn) on the current
 * CUDA device, with memory from the CUDA runtime.
 *
 *   abi_consumer DIR [gpu]
 *   abi_consumer DIR sparse
 *
 * DIR holds the inputs as raw little-endian arrays and receives the outputs:
 *   dims        text: batch H H_q H_p P d Nmax N_CTA alpha cluster scale
 *   bhat.f32    [H]          per-head budgets B^ of the layer
 *   N.i32       [batch]      context lengths
 *   scores.f32  [batch][H][Nmax]            (gpu)
 *   K.u16 V.u16 [batch][H][Nmax][d] bf16    (gpu)
 *   q.u16       [batch][H_q][d] bf16        (gpu)
 * host outputs: head_order.i32 [H], ntok.i32 [batch][H], Phi.i64 [G], pt_off.i64
 *   [batch*G+1], pt_ids.i32 [n_pages], S.i32 [G], items.i32 [n_items][7] = (cta, b, h,
 *   t0, t1, part, nparts) in plan order
 * gpu outputs: kept.i32 [batch][H][Nmax], out.u16 [batch][H_q][d], lse.f32 [batch][H_q],
 *   status.i32 [1]
 * "sparse" runs the page-selection path instead, over a dense cache of H_p = 1 pages:
 *   sdims       text: batch H H_q d N P K N_CTA scale   (N % P == 0)
 *   K.u16 V.u16 [batch][H][N][d] bf16;  q.u16 [batch][H_q][d] bf16
 * It builds the MinMax cache (tg_build_minmax), selects each KV head's top K pages
 * (tg_page_score_topk) and decodes over them (tg_decode_attn with a plan of K pages per
 * head); outputs sel.i32 [batch][H][K], out.u16, lse.f32, status.i32.
 * Exit status 0 on success; otherwise the failing call and tg_last_error_string(). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tg.h"

static char g_dir[4096];

static void die(const char *what, const char *why) {
  fprintf(stderr, "abi_consumer: %s: %s\n", what, why);
  exit(1);
}

#define TG(call)                                       \
  do {                                                 \
    if ((call) != TG_OK) die(#call, tg_last_error_string()); \
  } while (0)

#define CU(call)                                               \
  do {                                                         \
    cudaError_t e_ = (call);                                   \
    if (e_ != cudaSuccess) die(#call, cudaGetErrorString(e_)); \
  } while (0)

static const char *path(const char *name) {
  static char p[4200];
  snprintf(p, sizeof p, "%s/%s", g_dir, name);
  return p;
}

static void *read_file(const char *name, size_t bytes) {
  FILE *f = fopen(path(name), "rb");
  void *buf = malloc(bytes ? bytes : 1);
  if (!f || !buf) die("open", name);
  if (bytes && fread(buf, 1, bytes, f) != bytes) die("short read", name);
  fclose(f);
  return buf;
}

static void write_file(const char *name, const void *buf, size_t bytes) {
  FILE *f = fopen(path(name), "wb");
  if (!f) die("create", name);
  if (bytes && fwrite(buf, 1, bytes, f) != bytes) die("short write", name);
  fclose(f);
}

static void *to_device(const void *host, size_t bytes) {
  void *d = NULL;
  CU(cudaMalloc(&d, bytes ? bytes : 16));
  if (bytes) CU(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
  return d;
}

/* The page-selection path of one layer (see the header comment). */
static int run_sparse(void) {
  int batch, H, H_q, d, N, P, K, N_CTA, b, h, p, n_pages;
  float scale;
  FILE *f = fopen(path("sdims"), "r");
  if (!f) die("open", "sdims");
  if (fscanf(f, "%d %d %d %d %d %d %d %d %f", &batch, &H, &H_q, &d, &N, &P, &K, &N_CTA, &scale) != 9)
    die("parse", "sdims");
  fclose(f);
  if (batch <= 0 || H <= 0 || H_q % H || P <= 0 || N % P || K <= 0 || K > N / P) die("sdims", "sizes out of range");
  n_pages = N / P;
  {
    const size_t n_kv = (size_t)batch * H * N * d, n_q = (size_t)batch * H_q * d, rows = (size_t)batch * H;
    const size_t page_elems = (size_t)2 * P * d;  /* one H_p = 1 page: K rows then V rows */
    const int64_t pool_pages = (int64_t)rows * n_pages;
    uint16_t *Kh = (uint16_t *)read_file("K.u16", sizeof(uint16_t) * n_kv);
    uint16_t *Vh = (uint16_t *)read_file("V.u16", sizeof(uint16_t) * n_kv);
    uint16_t *qh = (uint16_t *)read_file("q.u16", sizeof(uint16_t) * n_q);
    uint16_t *pool = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)pool_pages * page_elems);
    int32_t *ntok = (int32_t *)malloc(sizeof(int32_t) * rows), *order = (int32_t *)malloc(sizeof(int32_t) * H);
    int64_t *Phi = (int64_t *)calloc((size_t)H, sizeof(int64_t)), *pt_off = (int64_t *)malloc(sizeof(int64_t) * (rows + 1));
    int32_t *S = (int32_t *)malloc(sizeof(int32_t) * H), *sel = (int32_t *)malloc(sizeof(int32_t) * rows * K);
    uint16_t *out = (uint16_t *)malloc(sizeof(uint16_t) * n_q);
    float *lse = (float *)malloc(sizeof(float) * (size_t)batch * H_q);
    int64_t plan_bytes = 0, work_bytes = 0, ws_bytes = 0;
    int32_t status = 0;
    uint8_t *plan;
    void *d_K, *d_q, *d_pool, *d_off, *d_plan, *d_mm = NULL, *d_ws = NULL, *d_sel = NULL, *d_ids = NULL;
    void *d_work = NULL, *d_out = NULL, *d_lse = NULL, *d_status = NULL;
    if (!pool || !ntok || !order || !Phi || !pt_off || !S || !sel || !out || !lse) die("malloc", "sparse arrays");
    /* the dense cache [batch][H][n_pages][2][P][d] from K and V [batch][H][N][d] */
    for (b = 0; b < batch; ++b)
      for (h = 0; h < H; ++h)
        for (p = 0; p < n_pages; ++p) {
          const size_t row = (size_t)b * H + h, src = (row * N + (size_t)p * P) * d;
          uint16_t *dst = pool + (row * n_pages + p) * page_elems;
          memcpy(dst, Kh + src, sizeof(uint16_t) * P * d);
          memcpy(dst + (size_t)P * d, Vh + src, sizeof(uint16_t) * P * d);
        }
    /* host plan: every KV head attends K whole pages; H_p = 1, so group g is head g */
    for (h = 0; h < H; ++h) order[h] = h;
    for (b = 0; b < batch; ++b)
      for (h = 0; h < H; ++h) {
        ntok[b * H + h] = K * P;
        Phi[h] += K * P;
      }
    TG(tg_split_map(1, H, N_CTA, Phi, S));
    TG(tg_plan_decode(1, batch, H, H_q, 1, P, d, N_CTA, S, order, ntok, NULL, 0, &plan_bytes, &work_bytes));
    plan = (uint8_t *)malloc((size_t)plan_bytes);
    if (!plan) die("malloc", "plan");
    TG(tg_plan_decode(1, batch, H, H_q, 1, P, d, N_CTA, S, order, ntok, plan, plan_bytes, &plan_bytes, &work_bytes));
    /* list b*H + h (G = H groups of one head) holds that head's K selected pages */
    for (b = 0; b <= (int)rows; ++b) pt_off[b] = (int64_t)b * K;

    /* device: MinMax cache, page scores and top-K (page ids into the dense pool), decode */
    d_K = to_device(Kh, sizeof(uint16_t) * n_kv);
    d_q = to_device(qh, sizeof(uint16_t) * n_q);
    d_pool = to_device(pool, sizeof(uint16_t) * (size_t)pool_pages * page_elems);
    d_off = to_device(pt_off, sizeof(int64_t) * (rows + 1));
    d_plan = to_device(plan, (size_t)plan_bytes);
    CU(cudaMalloc(&d_mm, sizeof(uint16_t) * rows * n_pages * 2 * d));
    TG(tg_page_score_workspace(batch, H, n_pages, &ws_bytes));
    CU(cudaMalloc(&d_ws, (size_t)ws_bytes));
    CU(cudaMemset(d_ws, 0, (size_t)ws_bytes));
    CU(cudaMalloc(&d_sel, sizeof(int32_t) * rows * K));
    CU(cudaMalloc(&d_ids, sizeof(int32_t) * rows * K));
    CU(cudaMalloc(&d_work, (size_t)(work_bytes ? work_bytes : 16)));
    CU(cudaMemset(d_work, 0, (size_t)(work_bytes ? work_bytes : 16)));
    CU(cudaMalloc(&d_out, sizeof(uint16_t) * n_q));
    CU(cudaMalloc(&d_lse, sizeof(float) * (size_t)batch * H_q));
    CU(cudaMalloc(&d_status, sizeof(int32_t)));
    CU(cudaMemset(d_status, 0, sizeof(int32_t)));
    TG(tg_build_minmax(NULL, batch, H, N, P, d, (const uint16_t *)d_K, (uint16_t *)d_mm, (int32_t *)d_status));
    TG(tg_page_score_topk(NULL, batch, H, H_q / H, d, n_pages, K, (const uint16_t *)d_q, (const uint16_t *)d_mm,
                          (int32_t *)d_sel, (int32_t *)d_ids, d_ws, ws_bytes, 0, (int32_t *)d_status));
    TG(tg_decode_attn(NULL, plan, d_plan, 0, (const uint16_t *)d_q, (const uint16_t *)d_pool, pool_pages,
                      (const int64_t *)d_off, (const int32_t *)d_ids, scale, d_work, work_bytes, (uint16_t *)d_out,
                      (float *)d_lse, (int32_t *)d_status, NULL));
    CU(cudaDeviceSynchronize());
    if (tg_check_status((const int32_t *)d_status, &status) != TG_OK && status == 0)
      die("tg_check_status", tg_last_error_string());
    CU(cudaMemcpy(sel, d_sel, sizeof(int32_t) * rows * K, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(out, d_out, sizeof(uint16_t) * n_q, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(lse, d_lse, sizeof(float) * (size_t)batch * H_q, cudaMemcpyDeviceToHost));
    write_file("sel.i32", sel, sizeof(int32_t) * rows * K);
    write_file("out.u16", out, sizeof(uint16_t) * n_q);
    write_file("lse.f32", lse, sizeof(float) * (size_t)batch * H_q);
    write_file("status.i32", &status, sizeof status);

    cudaFree(d_K); cudaFree(d_q); cudaFree(d_pool); cudaFree(d_off); cudaFree(d_plan); cudaFree(d_mm);
    cudaFree(d_ws); cudaFree(d_sel); cudaFree(d_ids); cudaFree(d_work); cudaFree(d_out); cudaFree(d_lse);
    cudaFree(d_status);
    free(Kh); free(Vh); free(qh); free(pool); free(ntok); free(order); free(Phi); free(pt_off); free(S);
    free(sel); free(out); free(lse); free(plan);
    return 0;
  }
}

int main(int argc, char **argv) {
  int batch, H, H_q, H_p, P, d, Nmax, N_CTA, cluster;
  float alpha, scale;
  int G, c, i;
  int gpu = argc > 2 && strcmp(argv[2], "gpu") == 0;
  FILE *f;
  float *bhat;
  int32_t *N, *head_order, *ntok, *pt_ids, *S, *items_out;
  int64_t *Phi, *pt_off, n_pages = 0, n_mono = 0, plan_bytes = 0, work_bytes = 0;
  uint8_t *plan;
  const tg_plan_header *hdr;
  const tg_plan_layer *lay;
  const int32_t *cta_off;
  const tg_work_item *items;

  if (argc < 2) die("usage", "abi_consumer DIR [gpu | sparse]");
  snprintf(g_dir, sizeof g_dir, "%s", argv[1]);
  if (argc > 2 && strcmp(argv[2], "sparse") == 0) return run_sparse();
  f = fopen(path("dims"), "r");
  if (!f) die("open", "dims");
  if (fscanf(f, "%d %d %d %d %d %d %d %d %f %d %f", &batch, &H, &H_q, &H_p, &P, &d, &Nmax, &N_CTA, &alpha,
             &cluster, &scale) != 11)
    die("parse", "dims");
  fclose(f);
  if (batch <= 0 || H <= 0 || H_p <= 0 || H % H_p || Nmax <= 0) die("dims", "sizes out of range");
  G = H / H_p;

  /* ---- host: page tables (a query for the size first), split map, plan */
  bhat = (float *)read_file("bhat.f32", sizeof(float) * (size_t)H);
  N = (int32_t *)read_file("N.i32", sizeof(int32_t) * (size_t)batch);
  head_order = (int32_t *)malloc(sizeof(int32_t) * (size_t)H);
  ntok = (int32_t *)malloc(sizeof(int32_t) * (size_t)batch * H);
  Phi = (int64_t *)malloc(sizeof(int64_t) * (size_t)G);
  pt_off = (int64_t *)malloc(sizeof(int64_t) * ((size_t)batch * G + 1));
  S = (int32_t *)malloc(sizeof(int32_t) * (size_t)G);
  if (!head_order || !ntok || !Phi || !pt_off || !S) die("malloc", "host arrays");
  TG(tg_build_pages(1, batch, H, H_p, P, alpha, bhat, N, cluster, head_order, ntok, Phi, pt_off, NULL, 0,
                    &n_pages, &n_mono));
  pt_ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_pages ? n_pages : 1));
  if (!pt_ids) die("malloc", "pt_ids");
  TG(tg_build_pages(1, batch, H, H_p, P, alpha, bhat, N, cluster, head_order, ntok, Phi, pt_off, pt_ids, n_pages,
                    &n_pages, &n_mono));
  TG(tg_split_map(1, G, N_CTA, Phi, S));
  TG(tg_plan_decode(1, batch, H, H_q, H_p, P, d, N_CTA, S, head_order, ntok, NULL, 0, &plan_bytes, &work_bytes));
  plan = (uint8_t *)malloc((size_t)plan_bytes);
  if (!plan) die("malloc", "plan");
  TG(tg_plan_decode(1, batch, H, H_q, H_p, P, d, N_CTA, S, head_order, ntok, plan, plan_bytes, &plan_bytes,
                    &work_bytes));

  /* read the plan through the header's self-description */
  hdr = (const tg_plan_header *)plan;
  if (hdr->magic != TG_PLAN_MAGIC || hdr->version != TG_PLAN_VERSION || hdr->N_CTA != N_CTA)
    die("plan", "unexpected header");
  lay = (const tg_plan_layer *)(plan + hdr->layers);
  cta_off = (const int32_t *)(plan + lay->cta_off);
  items = (const tg_work_item *)(plan + lay->items);
  items_out = (int32_t *)malloc(sizeof(int32_t) * 7 * (size_t)(lay->n_items ? lay->n_items : 1));
  if (!items_out) die("malloc", "items");
  for (c = 0; c < N_CTA; ++c)
    for (i = cta_off[c]; i < cta_off[c + 1]; ++i) {
      int32_t *o = items_out + 7 * (size_t)i;
      o[0] = c;
      o[1] = items[i].b;
      o[2] = items[i].h;
      o[3] = items[i].t0;
      o[4] = items[i].t1;
      o[5] = items[i].part;
      o[6] = items[i].nparts;
    }
  write_file("head_order.i32", head_order, sizeof(int32_t) * (size_t)H);
  write_file("ntok.i32", ntok, sizeof(int32_t) * (size_t)batch * H);
  write_file("Phi.i64", Phi, sizeof(int64_t) * (size_t)G);
  write_file("pt_off.i64", pt_off, sizeof(int64_t) * ((size_t)batch * G + 1));
  write_file("pt_ids.i32", pt_ids, sizeof(int32_t) * (size_t)n_pages);
  write_file("S.i32", S, sizeof(int32_t) * (size_t)G);
  write_file("items.i32", items_out, sizeof(int32_t) * 7 * (size_t)lay->n_items);

  if (gpu) {
    /* ---- device: retention into the pool, then decode attention of the layer */
    const size_t n_sc = (size_t)batch * H * Nmax, n_kv = n_sc * (size_t)d, n_q = (size_t)batch * H_q * d;
    const size_t pool_bytes = (size_t)(n_pages ? n_pages : 1) * H_p * 2 * P * d * sizeof(uint16_t);
    float *scores = (float *)read_file("scores.f32", sizeof(float) * n_sc);
    uint16_t *K = (uint16_t *)read_file("K.u16", sizeof(uint16_t) * n_kv);
    uint16_t *V = (uint16_t *)read_file("V.u16", sizeof(uint16_t) * n_kv);
    uint16_t *q = (uint16_t *)read_file("q.u16", sizeof(uint16_t) * n_q);
    uint16_t *out = (uint16_t *)malloc(sizeof(uint16_t) * n_q);
    float *lse = (float *)malloc(sizeof(float) * (size_t)batch * H_q);
    int32_t *kept = (int32_t *)malloc(sizeof(int32_t) * n_sc);
    int32_t status = 0;
    int64_t ws_bytes = 0;
    void *d_N, *d_sc, *d_K, *d_V, *d_q, *d_order, *d_ntok, *d_off, *d_ids, *d_plan;
    void *d_pool = NULL, *d_kept = NULL, *d_ws = NULL, *d_work = NULL, *d_out = NULL, *d_lse = NULL;
    void *d_status = NULL;
    if (!out || !lse || !kept) die("malloc", "outputs");

    d_N = to_device(N, sizeof(int32_t) * (size_t)batch);
    d_sc = to_device(scores, sizeof(float) * n_sc);
    d_K = to_device(K, sizeof(uint16_t) * n_kv);
    d_V = to_device(V, sizeof(uint16_t) * n_kv);
    d_q = to_device(q, sizeof(uint16_t) * n_q);
    d_order = to_device(head_order, sizeof(int32_t) * (size_t)H);
    d_ntok = to_device(ntok, sizeof(int32_t) * (size_t)batch * H);
    d_off = to_device(pt_off, sizeof(int64_t) * ((size_t)batch * G + 1));
    d_ids = to_device(pt_ids, sizeof(int32_t) * (size_t)(n_pages ? n_pages : 1));
    d_plan = to_device(plan, (size_t)plan_bytes);
    CU(cudaMalloc(&d_pool, pool_bytes));
    CU(cudaMalloc(&d_kept, sizeof(int32_t) * n_sc));
    CU(cudaMemset(d_kept, 0xff, sizeof(int32_t) * n_sc));
    TG(tg_compact_topk_workspace(batch, H, Nmax, &ws_bytes));
    CU(cudaMalloc(&d_ws, (size_t)ws_bytes));
    CU(cudaMalloc(&d_work, (size_t)(work_bytes ? work_bytes : 16)));
    CU(cudaMemset(d_work, 0, (size_t)(work_bytes ? work_bytes : 16)));
    CU(cudaMalloc(&d_out, sizeof(uint16_t) * n_q));
    CU(cudaMalloc(&d_lse, sizeof(float) * (size_t)batch * H_q));
    CU(cudaMalloc(&d_status, sizeof(int32_t)));
    CU(cudaMemset(d_status, 0, sizeof(int32_t)));

    TG(tg_compact_topk(NULL, batch, H, H_p, P, d, Nmax, (const int32_t *)d_N, (const float *)d_sc,
                       (const uint16_t *)d_K, (const uint16_t *)d_V, (const int32_t *)d_order,
                       (const int32_t *)d_ntok, (const int64_t *)d_off, (const int32_t *)d_ids, n_pages,
                       (uint16_t *)d_pool, (int32_t *)d_kept, d_ws, ws_bytes, (int32_t *)d_status));
    TG(tg_decode_attn(NULL, plan, d_plan, 0, (const uint16_t *)d_q, (const uint16_t *)d_pool, n_pages,
                      (const int64_t *)d_off, (const int32_t *)d_ids, scale, d_work, work_bytes,
                      (uint16_t *)d_out, (float *)d_lse, (int32_t *)d_status, NULL));
    CU(cudaDeviceSynchronize());
    if (tg_check_status((const int32_t *)d_status, &status) != TG_OK && status == 0)
      die("tg_check_status", tg_last_error_string());
    CU(cudaMemcpy(out, d_out, sizeof(uint16_t) * n_q, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(lse, d_lse, sizeof(float) * (size_t)batch * H_q, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(kept, d_kept, sizeof(int32_t) * n_sc, cudaMemcpyDeviceToHost));
    write_file("kept.i32", kept, sizeof(int32_t) * n_sc);
    write_file("out.u16", out, sizeof(uint16_t) * n_q);
    write_file("lse.f32", lse, sizeof(float) * (size_t)batch * H_q);
    write_file("status.i32", &status, sizeof status);

    cudaFree(d_N); cudaFree(d_sc); cudaFree(d_K); cudaFree(d_V); cudaFree(d_q); cudaFree(d_order);
    cudaFree(d_ntok); cudaFree(d_off); cudaFree(d_ids); cudaFree(d_plan); cudaFree(d_pool); cudaFree(d_kept);
    cudaFree(d_ws); cudaFree(d_work); cudaFree(d_out); cudaFree(d_lse); cudaFree(d_status);
    free(scores); free(K); free(V); free(q); free(out); free(lse); free(kept);
  }
  free(bhat); free(N); free(head_order); free(ntok); free(Phi); free(pt_off); free(pt_ids); free(S);
  free(plan); free(items_out);
  return 0;
}
