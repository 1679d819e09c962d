/*
 * iso_oracle.c -- plain float64 CPU oracle for the invariant GEMM, RMSNorm,
 * selected-token logprob and MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA library, and never calls it.
 *
 * Every quantity is computed from its plain definition in double precision.
 * The leaf / tree / chunk decomposition that the numerical contract fixes is
 * written out as explicit loops, so the reader can check it against the
 * pages by eye:
 *
 *   - GEMM as contiguous K-leaves combined by a fixed binary tree:
 *     [IsoExec blog, "Parallelism-invariant kernels"]; the same tree for
 *     every tensor-parallel size: [RL-Kernel blog, §6 table, row 06].
 *   - one FP32->BF16 conversion after accumulation:
 *     [RL-Kernel blog, §2 "Four Common Trigger Points"; §7 "GEMM"].
 *   - LSE with max shift and the two-block merge
 *     m = max(m1,m2), s = s1*e^(m1-m) + s2*e^(m2-m):
 *     [RL-Kernel blog, §4 "Focus: ... LogSumExp", "Causal Chain: How Block
 *     Merge Order Alters LSE"]; fixed vocab-tile merge order: [RL-Kernel
 *     blog, §7 "LogP"].
 *   - selected-token logprob = log-softmax over the vocabulary gathered at
 *     the chosen token: [RL-Kernel blog, §1 table; §4 "Right Linear LogP
 *     box"]; delta_t: [VeXact paper, §2 Eq. (1)]; mismatch diagnostics
 *     (K1, K3, truncated importance weights, sequence rejection): [VeXact
 *     paper, §4.1, §4.2 Eq. (6)-(7), Appendix A.4].
 *   - RMSNorm reduction over the hidden dimension: [RL-Kernel blog, §4
 *     table]; batch-invariant RMSNorm: [VeXact paper, §3.1].
 *   - MoE: deterministic top-k routing, packed gate/up -> SwiGLU -> down as
 *     separate stages, combine in fixed routing order over 8 fp32 leaves:
 *     [IsoExec blog, "Unified model", "Unified execution contract"
 *     composition example (moe.combine), "Parallelism-invariant kernels"];
 *     [RL-Kernel blog, §6 table row 04; §7 "FFN"].
 *
 * Where the pages leave a step open the oracle takes these readings:
 *   - tree: balanced binary tree over leaves in index order, leaf count a
 *     power of two; the left operand of every add is the lower index.
 *   - inside a leaf: ascending k.  In double every bf16*bf16 product is exact
 *     and the running sum is within ~K*2^-53 relative of the exact value.
 *   - vocab tiles of 128 columns, chunks of a fixed number of tiles; tiles
 *     folded left-to-right inside a chunk with the two-block merge; chunks
 *     combined by a balanced pairwise tree, an odd last node carried up.
 *   - RMSNorm: y = bf16(x * (1/sqrt(mean(x^2) + eps)) * gamma).
 *   - routing: top-k by (logit descending, expert id ascending); gates are
 *     the softmax of the k selected logits (equal to renormalising the full
 *     softmax); slot order = router output order.
 *   - expert rounding points: gate/up root -> bf16, silu(g)*u -> bf16, down
 *     root -> bf16, weighted slot tree -> bf16.
 *
 * Compile with -ffp-contract=off so no multiply-add is fused behind the
 * reader's back.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> double                                                          */
/* ------------------------------------------------------------------------ */

double iso_oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), directly from double. */
uint16_t iso_oracle_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  double f = frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  double q;
  if (e - 1 >= -126) {
    /* normal: 8 significant bits */
    q = ldexp(rint(ldexp(f, 8)), e - 8);
  } else {
    /* subnormal: fixed quantum 2^-133 */
    q = ldexp(rint(ldexp(a, 133)), -133);
  }
  if (q >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float fq = (float)q; /* exact: q has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &fq, sizeof u);
  return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void iso_oracle_round_bf16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = iso_oracle_double_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* a tiny parallel-for over rows                                            */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(void* ctx, int64_t row, double* scratch);

typedef struct {
  row_fn fn;
  void* ctx;
  int64_t nrows;
  int nthreads;
  int tid;
  size_t scratch_doubles;
} par_job;

static void* par_worker(void* p) {
  par_job* j = (par_job*)p;
  double* scratch = NULL;
  if (j->scratch_doubles) scratch = (double*)malloc(j->scratch_doubles * sizeof(double));
  for (int64_t r = j->tid; r < j->nrows; r += j->nthreads) j->fn(j->ctx, r, scratch);
  free(scratch);
  return NULL;
}

static void parallel_rows(row_fn fn, void* ctx, int64_t nrows, int nthreads, size_t scratch_doubles) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nrows < nthreads) nthreads = (int)(nrows > 0 ? nrows : 1);
  pthread_t th[256];
  par_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].nrows = nrows;
    jobs[t].nthreads = nthreads;
    jobs[t].tid = t;
    jobs[t].scratch_doubles = scratch_doubles;
  }
  if (nthreads == 1) {
    par_worker(&jobs[0]);
    return;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, par_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* Balanced binary tree over n vectors of length len, in place.             */
/* Level by level: (0,1),(2,3),... then (0,2),(4,6),...; left = lower index.*/
/* n must be a power of two.  Result in v[0].                               */
/* ------------------------------------------------------------------------ */

static void tree_reduce(double* v, int n, int64_t len) {
  for (int w = 1; w < n; w *= 2)
    for (int p = 0; p + w < n; p += 2 * w) {
      double* left = v + (int64_t)p * len;
      const double* right = v + (int64_t)(p + w) * len;
      for (int64_t j = 0; j < len; ++j) left[j] = left[j] + right[j];
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM: leaf partials and the fixed tree                                   */
/* [IsoExec blog, "Parallelism-invariant kernels"]                          */
/*                                                                          */
/* A: M x K bf16 row-major (lda), B: K x N bf16 row-major (ldb).            */
/* Leaf l covers k in [l*K/L, (l+1)*K/L).  The function returns the root of */
/* the subtree over leaves [leaf_lo, leaf_hi) (an aligned power-of-two      */
/* block of the L leaves; [0, L) is the whole tree) as doubles, unrounded.  */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* A;
  int64_t lda;
  const uint16_t* B;
  int64_t ldb;
  int N, K, L, leaf_lo, leaf_hi;
  double* root;
  int64_t ldr;
} gemm_ctx;

static void gemm_leaf_partials(const uint16_t* arow, const uint16_t* B, int64_t ldb, int N, int K,
                               int L, int leaf_lo, int leaf_hi, double* P) {
  int kl = K / L;
  int nl = leaf_hi - leaf_lo;
  memset(P, 0, sizeof(double) * (size_t)nl * (size_t)N);
  for (int l = leaf_lo; l < leaf_hi; ++l) {
    double* p = P + (int64_t)(l - leaf_lo) * N;
    for (int k = l * kl; k < (l + 1) * kl; ++k) { /* ascending k */
      double a = iso_oracle_bf16_to_double(arow[k]);
      if (a == 0.0) continue; /* adds of exact zero products change nothing */
      const uint16_t* brow = B + (int64_t)k * ldb;
      for (int j = 0; j < N; ++j) p[j] = p[j] + a * iso_oracle_bf16_to_double(brow[j]);
    }
  }
}

static void gemm_row(void* c, int64_t i, double* P) {
  gemm_ctx* g = (gemm_ctx*)c;
  int nl = g->leaf_hi - g->leaf_lo;
  gemm_leaf_partials(g->A + i * g->lda, g->B, g->ldb, g->N, g->K, g->L, g->leaf_lo, g->leaf_hi, P);
  tree_reduce(P, nl, g->N);
  memcpy(g->root + i * g->ldr, P, sizeof(double) * (size_t)g->N);
}

static int is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int iso_oracle_gemm_root(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int M, int N,
                         int K, int L, int leaf_lo, int leaf_hi, double* root, int64_t ldr,
                         int nthreads) {
  if (!is_pow2(L) || K % L != 0 || leaf_lo < 0 || leaf_hi > L || leaf_hi <= leaf_lo) return -1;
  if (!is_pow2(leaf_hi - leaf_lo) || leaf_lo % (leaf_hi - leaf_lo) != 0) return -1;
  gemm_ctx g = {A, lda, B, ldb, N, K, L, leaf_lo, leaf_hi, root, ldr};
  parallel_rows(gemm_row, &g, M, nthreads, (size_t)(leaf_hi - leaf_lo) * (size_t)N);
  return 0;
}

/* The rank-local view: rank r of R owns leaves [r*L/R, (r+1)*L/R) of the   */
/* global tree; its A_r / B_r are the K/R-wide slices.  The subtree over a  */
/* rank's own L/R leaves is the balanced tree over them.                    */
int iso_oracle_gemm_leaf_partial(const uint16_t* A_r, int64_t lda, const uint16_t* B_r, int64_t ldb,
                                 int M, int N, int K_local, int L, int R, double* S_r, int64_t lds,
                                 int nthreads) {
  if (!is_pow2(R) || L % R != 0) return -1;
  return iso_oracle_gemm_root(A_r, lda, B_r, ldb, M, N, K_local, L / R, 0, L / R, S_r, lds, nthreads);
}

/* The top log2(R) levels of the tree over R subtree roots S[r][M][lds].    */
int iso_oracle_tree_combine(const double* S, int R, int64_t rank_stride, int M, int N, int64_t lds,
                            double* root, int64_t ldr) {
  if (!is_pow2(R)) return -1;
  double* v = (double*)malloc(sizeof(double) * (size_t)R * (size_t)N);
  for (int64_t i = 0; i < M; ++i) {
    for (int r = 0; r < R; ++r) memcpy(v + (int64_t)r * N, S + r * rank_stride + i * lds, sizeof(double) * (size_t)N);
    tree_reduce(v, R, N);
    memcpy(root + i * ldr, v, sizeof(double) * (size_t)N);
  }
  free(v);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm: y = bf16(x * (1/sqrt(mean(x^2) + eps)) * gamma)                  */
/* [RL-Kernel blog, §4 table "RMSNorm / hidden dimension"]                  */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* x;
  const uint16_t* gamma;
  double eps;
  int H;
  uint16_t* y;
  double* y_exact;
} rms_ctx;

static void rms_row(void* c, int64_t t, double* unused) {
  (void)unused;
  rms_ctx* g = (rms_ctx*)c;
  const uint16_t* xr = g->x + t * g->H;
  double ss = 0.0;
  for (int i = 0; i < g->H; ++i) {
    double v = iso_oracle_bf16_to_double(xr[i]);
    ss = ss + v * v;
  }
  double ms = ss / (double)g->H;
  double r = 1.0 / sqrt(ms + g->eps);
  for (int i = 0; i < g->H; ++i) {
    double v = iso_oracle_bf16_to_double(xr[i]) * r * iso_oracle_bf16_to_double(g->gamma[i]);
    if (g->y_exact) g->y_exact[t * g->H + i] = v;
    if (g->y) g->y[t * g->H + i] = iso_oracle_double_to_bf16(v);
  }
}

int iso_oracle_rmsnorm(const uint16_t* x, const uint16_t* gamma, double eps, int T, int H, uint16_t* y,
                       double* y_exact, int nthreads) {
  if (H <= 0 || T < 0) return -1;
  rms_ctx g = {x, gamma, eps, H, y, y_exact};
  parallel_rows(rms_row, &g, T, nthreads, 0);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* LSE statistics and the two-block merge                                   */
/* [RL-Kernel blog, §4 "Causal Chain: How Block Merge Order Alters LSE"]    */
/* An empty block is (m, s) = (-inf, 0); it is the identity of the merge.   */
/* ------------------------------------------------------------------------ */

typedef struct {
  double m, s;
} lse_stat;

static lse_stat lse_merge(lse_stat a, lse_stat b) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  lse_stat r;
  r.m = a.m > b.m ? a.m : b.m;
  r.s = a.s * exp(a.m - r.m) + b.s * exp(b.m - r.m);
  return r;
}

void iso_oracle_lse_merge(double m1, double s1, double m2, double s2, double* m, double* s) {
  lse_stat a = {m1, s1}, b = {m2, s2};
  lse_stat r = lse_merge(a, b);
  *m = r.m;
  *s = r.s;
}

/* Statistics of one block of scores: m = max, s = sum_i exp(x_i - m), i ascending. */
static lse_stat lse_block(const double* z, int n) {
  lse_stat r = {-INFINITY, 0.0};
  if (n <= 0) return r;
  double m = z[0];
  for (int i = 1; i < n; ++i)
    if (z[i] > m) m = z[i];
  double s = 0.0;
  for (int i = 0; i < n; ++i) s = s + exp(z[i] - m);
  r.m = m;
  r.s = s;
  return r;
}

/* ------------------------------------------------------------------------ */
/* Selected-token logprob                                                   */
/* z[t, v] = tree root of h[t,:] . W[:, v]  (fp64 here, never rounded)      */
/* tile stats per tile_cols columns; chunk = chunk_tiles tiles folded left  */
/* to right; chunks combined by a balanced pairwise tree (odd node carried);*/
/* lse = m + log s; out = z[t, id_t] - lse.                                 */
/* [RL-Kernel blog, §4 "Focus", "Causal Chain"; §6 table row 05;            */
/*  §7 "LogP"]; [VeXact paper, §2 Eq. (1)]                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* h;
  const uint16_t* W;
  const int32_t* ids;
  int H, V, L, tile_cols, chunk_tiles;
  double* out;
  double* lse_chunked;
  double* lse_direct;
  double* z_sel;
  double* chunk_m; /* optional [T][C] */
  double* chunk_s;
} lp_ctx;

static int lp_num_chunks(int V, int tile_cols, int chunk_tiles) {
  int tiles = (V + tile_cols - 1) / tile_cols;
  return (tiles + chunk_tiles - 1) / chunk_tiles;
}

int iso_oracle_logprob_num_chunks(int V, int tile_cols, int chunk_tiles) {
  return lp_num_chunks(V, tile_cols, chunk_tiles);
}

static void lp_row(void* c, int64_t t, double* scratch) {
  lp_ctx* g = (lp_ctx*)c;
  int V = g->V;
  double* z = scratch;             /* [V]      */
  double* P = scratch + V;         /* [L][V]   */
  gemm_leaf_partials(g->h + t * g->H, g->W, V, V, g->H, g->L, 0, g->L, P);
  tree_reduce(P, g->L, V);
  memcpy(z, P, sizeof(double) * (size_t)V);

  int C = lp_num_chunks(V, g->tile_cols, g->chunk_tiles);
  lse_stat* cs = (lse_stat*)(P + V); /* reuse tail of P: C entries (L >= 1, so room exists) */
  for (int ci = 0; ci < C; ++ci) {
    lse_stat acc = {-INFINITY, 0.0};
    for (int tt = 0; tt < g->chunk_tiles; ++tt) {
      int col0 = (ci * g->chunk_tiles + tt) * g->tile_cols;
      if (col0 >= V) break;
      int n = V - col0 < g->tile_cols ? V - col0 : g->tile_cols;
      acc = lse_merge(acc, lse_block(z + col0, n)); /* left fold, ascending tiles */
    }
    cs[ci] = acc;
    if (g->chunk_m) g->chunk_m[t * C + ci] = acc.m;
    if (g->chunk_s) g->chunk_s[t * C + ci] = acc.s;
  }
  /* balanced pairwise tree over chunks, odd last node carried up */
  int n = C;
  while (n > 1) {
    int k = 0;
    for (int p = 0; p + 1 < n; p += 2) cs[k++] = lse_merge(cs[p], cs[p + 1]);
    if (n & 1) cs[k++] = cs[n - 1];
    n = k;
  }
  double lse = cs[0].m + log(cs[0].s);
  lse_stat all = lse_block(z, V);
  double lse_direct = all.m + log(all.s);
  int id = g->ids[t];
  double zs = (id >= 0 && id < V) ? z[id] : NAN;
  if (g->out) g->out[t] = zs - lse;
  if (g->lse_chunked) g->lse_chunked[t] = lse;
  if (g->lse_direct) g->lse_direct[t] = lse_direct;
  if (g->z_sel) g->z_sel[t] = zs;
}

int iso_oracle_selected_logprob(const uint16_t* h, const uint16_t* W, const int32_t* ids, int T, int H,
                                int V, int L, int tile_cols, int chunk_tiles, double* out,
                                double* lse_chunked, double* lse_direct, double* z_sel,
                                double* chunk_m, double* chunk_s, int nthreads) {
  if (!is_pow2(L) || H % L != 0 || V <= 0 || tile_cols <= 0 || chunk_tiles <= 0) return -1;
  lp_ctx g = {h, W, ids, H, V, L, tile_cols, chunk_tiles, out, lse_chunked, lse_direct, z_sel, chunk_m, chunk_s};
  int C = lp_num_chunks(V, tile_cols, chunk_tiles);
  size_t need = (size_t)V * (size_t)(L + 1) + 2 * (size_t)C + 2;
  parallel_rows(lp_row, &g, T, nthreads, need);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* MoE routing: top-k by (logit desc, id asc); gates = softmax of the k     */
/* selected logits.  [IsoExec blog, "Unified model": deterministic routing] */
/* ------------------------------------------------------------------------ */

int iso_oracle_moe_route(const float* logits, int T, int E, int k, int32_t* ids, double* w) {
  if (k <= 0 || k > E) return -1;
  char* taken = (char*)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower id on ties */
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    double m = (double)l[ids[t * k]];
    double s = 0.0;
    for (int j = 0; j < k; ++j) s = s + exp((double)l[ids[t * k + j]] - m);
    for (int j = 0; j < k; ++j) w[t * k + j] = exp((double)l[ids[t * k + j]] - m) / s;
  }
  free(taken);
  return 0;
}

/* Stable counting sort of the (token, slot) pairs by expert, keeping only  */
/* experts with mask[e] != 0 (mask NULL = all).  perm lists pair indices    */
/* t*k + j; offsets[e]..offsets[e+1] is expert e's range.  Returns count.   */
int iso_oracle_moe_permute(const int32_t* ids, int T, int E, int k, const uint8_t* mask, int32_t* perm,
                           int32_t* offsets) {
  int64_t P = (int64_t)T * k;
  int32_t* cnt = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int64_t p = 0; p < P; ++p) {
    int e = ids[p];
    if (e < 0 || e >= E) {
      free(cnt);
      return -1;
    }
    if (!mask || mask[e]) cnt[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + cnt[e];
  memset(cnt, 0, sizeof(int32_t) * (size_t)E);
  for (int64_t p = 0; p < P; ++p) {
    int e = ids[p];
    if (mask && !mask[e]) continue;
    perm[offsets[e] + cnt[e]++] = (int32_t)p;
  }
  int total = offsets[E];
  free(cnt);
  return total;
}

/* ------------------------------------------------------------------------ */
/* MoE expert layer for one token (all k slots):                            */
/*   G = tree(x . W1_e) (K = H leaves); g = bf16(G[:F]), u = bf16(G[F:]);   */
/*   h = bf16(silu(g) * u); y = bf16(tree(h . W2_e)) (K = F leaves);        */
/*   out = bf16(tree over slots j of w_j * y_j).                            */
/* [IsoExec blog, "Unified execution contract" (moe.combine, leaves 8,      */
/*  fp32 leaves), "Parallelism-invariant kernels" (fixed routing order)];   */
/* [RL-Kernel blog, §6 table row 04 (packed gate/up, SwiGLU, down, separate */
/*  stages)]                                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* x;
  const int32_t* ids;
  const double* w;
  const uint16_t* W1;
  const uint16_t* W2;
  int E, k, H, F, L;
  uint16_t* y_slots; /* optional [T][k][H] */
  uint16_t* out;     /* [T][H] */
  double* out_exact; /* optional [T][H] */
} moe_ctx;

static void moe_row(void* c, int64_t t, double* scratch) {
  moe_ctx* g = (moe_ctx*)c;
  int H = g->H, F = g->F, L = g->L, k = g->k;
  double* P1 = scratch;                        /* [L][2F] */
  double* P2 = P1 + (size_t)L * 2 * F;         /* [L][H]  */
  uint16_t* hb = (uint16_t*)(P2 + (size_t)L * H); /* [F] bf16 */
  double* ys = (double*)(hb + F + 8);          /* [k][H] weighted slots (aligned enough) */
  ys = (double*)(((uintptr_t)ys + 7) & ~(uintptr_t)7);
  for (int j = 0; j < k; ++j) {
    int e = g->ids[t * k + j];
    const uint16_t* W1e = g->W1 + (int64_t)e * H * 2 * F;
    const uint16_t* W2e = g->W2 + (int64_t)e * F * H;
    gemm_leaf_partials(g->x + t * H, W1e, 2 * F, 2 * F, H, L, 0, L, P1);
    tree_reduce(P1, L, 2 * F);
    for (int c2 = 0; c2 < F; ++c2) {
      double gv = iso_oracle_bf16_to_double(iso_oracle_double_to_bf16(P1[c2]));
      double uv = iso_oracle_bf16_to_double(iso_oracle_double_to_bf16(P1[F + c2]));
      double silu = gv / (1.0 + exp(-gv));
      hb[c2] = iso_oracle_double_to_bf16(silu * uv);
    }
    gemm_leaf_partials(hb, W2e, H, H, F, L, 0, L, P2);
    tree_reduce(P2, L, H);
    double wj = g->w[t * k + j];
    for (int c2 = 0; c2 < H; ++c2) {
      uint16_t yb = iso_oracle_double_to_bf16(P2[c2]);
      if (g->y_slots) g->y_slots[(t * k + j) * (int64_t)H + c2] = yb;
      ys[(int64_t)j * H + c2] = wj * iso_oracle_bf16_to_double(yb);
    }
  }
  /* slot tree: k must be a power of two */
  tree_reduce(ys, k, H);
  for (int c2 = 0; c2 < H; ++c2) {
    if (g->out_exact) g->out_exact[t * H + c2] = ys[c2];
    g->out[t * H + c2] = iso_oracle_double_to_bf16(ys[c2]);
  }
}

int iso_oracle_moe_layer(const uint16_t* x, const int32_t* ids, const double* w, const uint16_t* W1,
                         const uint16_t* W2, int T, int E, int k, int H, int F, int L, uint16_t* y_slots,
                         uint16_t* out, double* out_exact, int nthreads) {
  if (!is_pow2(L) || !is_pow2(k) || H % L != 0 || F % L != 0) return -1;
  moe_ctx g = {x, ids, w, W1, W2, E, k, H, F, L, y_slots, out, out_exact};
  size_t need = (size_t)L * 2 * F + (size_t)L * H + (size_t)F / 4 + 8 + (size_t)k * H + 16;
  parallel_rows(moe_row, &g, T, nthreads, need);
  return 0;
}

/* Weighted slot combine alone, from given bf16 slot outputs. */
int iso_oracle_moe_combine(const uint16_t* y_slots, const double* w, int T, int k, int H, uint16_t* out,
                           double* out_exact) {
  if (!is_pow2(k)) return -1;
  double* ys = (double*)malloc(sizeof(double) * (size_t)k * (size_t)H);
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j)
      for (int c = 0; c < H; ++c)
        ys[(int64_t)j * H + c] = w[t * k + j] * iso_oracle_bf16_to_double(y_slots[(t * k + j) * (int64_t)H + c]);
    tree_reduce(ys, k, H);
    for (int c = 0; c < H; ++c) {
      if (out_exact) out_exact[t * H + c] = ys[c];
      out[t * H + c] = iso_oracle_double_to_bf16(ys[c]);
    }
  }
  free(ys);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Token-level mismatch delta_t = log pi_train - log pi_rollout             */
/* [VeXact paper, §2 Eq. (1)]                                               */
/* ------------------------------------------------------------------------ */

void iso_oracle_delta(const double* logp_train, const double* logp_rollout, int64_t n, double* delta) {
  for (int64_t i = 0; i < n; ++i) delta[i] = logp_train[i] - logp_rollout[i];
}

/* ------------------------------------------------------------------------ */
/* Mismatch diagnostics over packed sequences of (train, rollout) logprobs  */
/* [VeXact paper, §2 Eq. (1): delta_t; §4.1 "KL estimators are not          */
/*  sufficient indicators": K1(r) = -log r, K3(r) = (r - 1) - log r;        */
/*  §4.2 Eq. (6): truncated importance weight min(r_corr, tau_tok),         */
/*  Eq. (7): sequence rejection 1[S_seq <= tau_seq] with                    */
/*  S_seq = sum_t K(q_t), q_t = r_corr,t = pi_train / pi_rollout;           */
/*  Appendix A.4: tau_tok = 2, tau_seq = 0.001]                             */
/* Sequence b holds tokens [offsets[b], offsets[b+1]).  Everything is       */
/* computed in double, summed in ascending token order.  Since r_corr is    */
/* pi_train / pi_rollout, log r_corr is delta_t itself: K1 = -delta_t and   */
/* K3 = (r_corr - 1) - delta_t.                                             */
/* ------------------------------------------------------------------------ */

int iso_oracle_mismatch(const float* logp_train, const float* logp_rollout, const int32_t* offsets, int B,
                        double tau_tok, double tau_seq, double* delta, double* tis_weight, double* seq_k1,
                        double* seq_k3, uint8_t* accept_k1, uint8_t* accept_k3, double* seq_max_abs_delta,
                        int32_t* seq_mismatches) {
  if (B < 0 || !offsets) return -1;
  for (int b = 0; b < B; ++b) {
    if (offsets[b + 1] < offsets[b]) return -2;
    double s1 = 0.0, s3 = 0.0, mx = 0.0;
    int32_t nmis = 0;
    for (int32_t t = offsets[b]; t < offsets[b + 1]; ++t) {
      const double d = (double)logp_train[t] - (double)logp_rollout[t]; /* Eq. (1) */
      const double r = exp(d);                                           /* r_corr */
      /* log r_corr = log pi_train - log pi_rollout = delta_t exactly */
      const double k1 = -d;
      const double k3 = (r - 1.0) - d;
      delta[t] = d;
      tis_weight[t] = r < tau_tok ? r : tau_tok; /* min(r_corr, tau_tok) */
      s1 += k1;
      s3 += k3;
      if (fabs(d) > mx) mx = fabs(d);
      if (logp_train[t] != logp_rollout[t]) ++nmis;
    }
    seq_k1[b] = s1;
    seq_k3[b] = s3;
    accept_k1[b] = s1 <= tau_seq ? 1 : 0;
    accept_k3[b] = s3 <= tau_seq ? 1 : 0;
    seq_max_abs_delta[b] = mx;
    seq_mismatches[b] = nmis;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Causal attention over packed variable-length sequences                    */
/* [RL-Kernel blog, §4 "Focus: The Shared Dependency of Attention and Linear */
/*  LogP on LogSumExp": softmax over the visible keys, LSE statistic;        */
/*  §6 table row 03 and §7 "Attention": no KV split, fixed chunking; VeXact  */
/*  paper, §3.1: KV splitting disabled]                                      */
/* Q [Tq x Hq x d], K and V [Tk x Hkv x d] bf16; query head h reads KV head  */
/* h / (Hq / Hkv).  Sequence b owns query rows [q_start[b], q_start[b+1])    */
/* and keys [k_start[b], k_start[b+1]); its query row r sits at position     */
/* p = pos0[b] + (r - q_start[b]) and sees the keys k_start[b] .. k_start[b] */
/* + p.  The plain definition in double: s_j = scale * (q . k_j),            */
/* m = max_j s_j, l = sum_j exp(s_j - m), out = sum_j exp(s_j - m) v_j / l,  */
/* lse = m + log(l).                                                         */
/* ------------------------------------------------------------------------ */

int iso_oracle_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* q_start,
                         const int32_t* k_start, const int32_t* pos0, int B, int Hq, int Hkv, int d, double scale,
                         double* out_exact, uint16_t* out, double* lse) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
  const int group = Hq / Hkv;
  double* s = NULL;
  int cap = 0;
  for (int b = 0; b < B; ++b) {
    for (int32_t r = q_start[b]; r < q_start[b + 1]; ++r) {
      const int32_t p = pos0[b] + (r - q_start[b]);
      const int32_t nvis = p + 1;
      if (p < 0 || k_start[b] + nvis > k_start[b + 1]) {
        free(s);
        return -2;
      }
      if (nvis > cap) {
        free(s);
        cap = nvis;
        s = (double*)malloc(sizeof(double) * (size_t)cap);
        if (!s) return -3;
      }
      for (int h = 0; h < Hq; ++h) {
        const int g = h / group;
        const uint16_t* q = Q + ((int64_t)r * Hq + h) * d;
        double m = -INFINITY;
        for (int32_t j = 0; j < nvis; ++j) {
          const uint16_t* k = K + ((int64_t)(k_start[b] + j) * Hkv + g) * d;
          double dot = 0.0;
          for (int e = 0; e < d; ++e) dot += iso_oracle_bf16_to_double(q[e]) * iso_oracle_bf16_to_double(k[e]);
          s[j] = scale * dot;
          if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int32_t j = 0; j < nvis; ++j) l += exp(s[j] - m);
        double* o = out_exact + ((int64_t)r * Hq + h) * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        for (int32_t j = 0; j < nvis; ++j) {
          const double w = exp(s[j] - m) / l;
          const uint16_t* v = V + ((int64_t)(k_start[b] + j) * Hkv + g) * d;
          for (int e = 0; e < d; ++e) o[e] += w * iso_oracle_bf16_to_double(v[e]);
        }
        for (int e = 0; e < d; ++e) out[((int64_t)r * Hq + h) * d + e] = iso_oracle_double_to_bf16(o[e]);
        lse[(int64_t)r * Hq + h] = m + log(l);
      }
    }
  }
  free(s);
  return 0;
}
