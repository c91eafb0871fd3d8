/*
 * pisa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the PISA pyramid Top-K block-selection
 * stage, written from the method's description so that the CUDA path can be
 * checked against it.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline / reference legs may load this library.  The CUDA
 * product path never calls it, links it or shares code with it.
 *
 * Sources (page title, section):
 *   [P2] "Block Sparse Attention with Log-Linear Complexity"
 *        §3.1 Fine to coarse: building the pyramid         -> level sizes, means
 *        §3.2 Coarse to fine: narrowing the Top-K          -> the walk, <=K rule
 *        "Scoring: LogSumExp, and why not the mean"        -> the LSE block score
 *        §4.1 An inconsistency the paper discloses         -> GQA head sum
 *   [P1] "PISA cuts block-sparse attention selection to O(N log N) with pyramid
 *        Top-K ..." (news summary)                         -> the same walk, the
 *        latency-benchmark shape (C=64, g=2, K=8, d=64).
 *
 * Readings where the pages are silent:
 *   - logits are scaled by 1/sqrt(d);
 *   - a ragged node is the mean over the tokens actually present;
 *   - causal: a node is eligible for query t iff its first token is <= t; a
 *     child that starts after t is left out of its parent's LSE (at the leaf
 *     level the children are raw keys, so keys after t are masked);
 *   - the LSE score is un-normalised (no "- log g");
 *   - ties in the Top-K go to the lower node index;
 *   - query head h belongs to KV group h / (Hq/Hkv) (contiguous groups);
 *   - the output lists the selected leaves in ascending order, padded with -1;
 *   - the score reported for a selected leaf is its exact raw-key LSE summed
 *     over the group's heads (computed whether or not the leaf level was
 *     scored); padded slots get -inf.
 *
 * Everything is computed in double precision from the exact fp32 values of the
 * bf16 inputs, with max-subtracted exponent sums, in the pages' order: no
 * blocking, no fusion, no reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_LEVELS 64

typedef struct {
  int L;                               /* number of levels that hold nodes (1..L) */
  int64_t M[ORACLE_MAX_LEVELS + 1];    /* M[l] = nodes at level l; M[0] = tokens   */
  int64_t off[ORACLE_MAX_LEVELS + 1];  /* offset of level l in the node array      */
  int64_t total;                       /* sum of M[1..L]                            */
  int64_t width[ORACLE_MAX_LEVELS + 1];/* tokens spanned by a full node of level l */
} oracle_levels;

/* [P2 §3.1] level 0 = raw keys (M_0 = N), level 1 = leaves (M_1 = ceil(N/C)),
 * above that every g adjacent blocks merge (M_l = ceil(M_{l-1}/g)) up to one root. */
static int levels_init(oracle_levels* lv, int64_t n, int C, int g) {
  memset(lv, 0, sizeof(*lv));
  if (n <= 0 || C <= 0 || g < 2) return -1;
  lv->M[0] = n;
  lv->width[0] = 1;
  lv->M[1] = (n + C - 1) / C;
  lv->width[1] = C;
  lv->off[1] = 0;
  int l = 1;
  while (lv->M[l] > 1) {
    if (l >= ORACLE_MAX_LEVELS) return -1;
    lv->M[l + 1] = (lv->M[l] + g - 1) / g;
    lv->width[l + 1] = lv->width[l] * g;
    lv->off[l + 1] = lv->off[l] + lv->M[l];
    ++l;
  }
  lv->L = l;
  lv->total = lv->off[l] + lv->M[l];
  return 0;
}

int pisa_oracle_num_levels(int64_t n, int C, int g) {
  oracle_levels lv;
  if (levels_init(&lv, n, C, g)) return -1;
  return lv.L;
}

int64_t pisa_oracle_level_size(int64_t n, int C, int g, int level) {
  oracle_levels lv;
  if (levels_init(&lv, n, C, g)) return -1;
  if (level < 0 || level > lv.L) return 0;
  return lv.M[level];
}

int64_t pisa_oracle_total_nodes(int64_t n, int C, int g) {
  oracle_levels lv;
  if (levels_init(&lv, n, C, g)) return -1;
  return lv.total;
}

/* First token of node i at level l (level 0 = raw key i). */
static int64_t node_start(const oracle_levels* lv, int l, int64_t i) { return i * lv->width[l]; }

/* One past the last token of node i at level l, clipped to the sequence. */
static int64_t node_end(const oracle_levels* lv, int l, int64_t i) {
  int64_t e = (i + 1) * lv->width[l];
  return e < lv->M[0] ? e : lv->M[0];
}

/* keys: [B][n_cap][Hkv][d] fp32 holding bf16 values; element (b, r, kv, j). */
static double key_at(const float* keys, int64_t n_cap, int Hkv, int d, int b, int64_t r, int kv, int j) {
  return (double)keys[(((int64_t)b * n_cap + r) * Hkv + kv) * d + j];
}

/* [P2 §3.1] every summary is the mean of all original keys in its block; for a
 * ragged block (the sequence's tail) the mean is over the tokens present.
 * Direct route: average the raw keys of the span.  out: [total][d] for (b, kv). */
static void build_direct(const float* keys, int64_t n_cap, int Hkv, int d, int b, int kv,
                         const oracle_levels* lv, double* out) {
  for (int l = 1; l <= lv->L; ++l) {
    for (int64_t i = 0; i < lv->M[l]; ++i) {
      double* row = out + (lv->off[l] + i) * d;
      int64_t s = node_start(lv, l, i), e = node_end(lv, l, i);
      for (int j = 0; j < d; ++j) row[j] = 0.0;
      for (int64_t r = s; r < e; ++r)
        for (int j = 0; j < d; ++j) row[j] += key_at(keys, n_cap, Hkv, d, b, r, kv, j);
      for (int j = 0; j < d; ++j) row[j] /= (double)(e - s);
    }
  }
}

/* Recursive route of [P2 §3.1]: a summary is the mean of its children's
 * summaries, weighted by how many tokens each child holds (equal weights when
 * the children are full).  Used only to check that both routes agree. */
static void build_recursive(const float* keys, int64_t n_cap, int Hkv, int d, int b, int kv,
                            int g, const oracle_levels* lv, double* out) {
  for (int64_t i = 0; i < lv->M[1]; ++i) {
    double* row = out + (lv->off[1] + i) * d;
    int64_t s = node_start(lv, 1, i), e = node_end(lv, 1, i);
    for (int j = 0; j < d; ++j) row[j] = 0.0;
    for (int64_t r = s; r < e; ++r)
      for (int j = 0; j < d; ++j) row[j] += key_at(keys, n_cap, Hkv, d, b, r, kv, j);
    for (int j = 0; j < d; ++j) row[j] /= (double)(e - s);
  }
  for (int l = 2; l <= lv->L; ++l) {
    for (int64_t i = 0; i < lv->M[l]; ++i) {
      double* row = out + (lv->off[l] + i) * d;
      double cnt = 0.0;
      for (int j = 0; j < d; ++j) row[j] = 0.0;
      for (int c = 0; c < g; ++c) {
        int64_t ch = i * g + c;
        if (ch >= lv->M[l - 1]) break;
        double w = (double)(node_end(lv, l - 1, ch) - node_start(lv, l - 1, ch));
        const double* crow = out + (lv->off[l - 1] + ch) * d;
        for (int j = 0; j < d; ++j) row[j] += w * crow[j];
        cnt += w;
      }
      for (int j = 0; j < d; ++j) row[j] /= cnt;
    }
  }
}

/* Pyramid over the first n tokens of every sequence.  keys: [B][n_cap][Hkv][d];
 * out: [B][Hkv][total_nodes(n)][d], levels leaf-first.  recursive != 0 selects
 * the count-weighted merge route instead of the direct mean. */
int pisa_oracle_build_pyramid(const float* keys, int B, int64_t n_cap, int64_t n, int Hkv, int d,
                              int C, int g, int recursive, double* out) {
  oracle_levels lv;
  if (n > n_cap || levels_init(&lv, n, C, g)) return -1;
  for (int b = 0; b < B; ++b)
    for (int kv = 0; kv < Hkv; ++kv) {
      double* o = out + ((int64_t)b * Hkv + kv) * lv.total * d;
      if (recursive)
        build_recursive(keys, n_cap, Hkv, d, b, kv, g, &lv, o);
      else
        build_direct(keys, n_cap, Hkv, d, b, kv, &lv, o);
    }
  return 0;
}

/* log(sum_i exp(x_i)) with the largest term factored out; x has m >= 1 terms. */
static double lse(const double* x, int m) {
  double mx = x[0];
  for (int i = 1; i < m; ++i)
    if (x[i] > mx) mx = x[i];
  double s = 0.0;
  for (int i = 0; i < m; ++i) s += exp(x[i] - mx);
  return mx + log(s);
}

typedef struct {
  const float* q;      /* [Hq][d] rows of this query (fp32 holding bf16)          */
  const float* keys;   /* [B][n_cap][Hkv][d]                                       */
  const double* pyr;   /* [total][d] summaries of this (b, kv)                     */
  const oracle_levels* lv;
  int64_t n_cap;
  int b, kv, Hkv, G, d, g, causal;
  int64_t t;           /* query position                                           */
  double scale;        /* 1/sqrt(d)                                                */
  double* work;        /* scratch of >= max(C, g) doubles                          */
  int mode;            /* block score: 0 LSE, 1 mean (PISA-1), 2 mean + var/2 (PISA-2) */
} walk_ctx;

/* ["Scoring: LogSumExp"]: the Taylor expansion of log sum_i e^{z_i} around the mean,
 * without the log m term, truncated at first order gives the mean of the logits
 * (the PISA-1 ablation) and at second order the mean plus half their variance (PISA-2).
 * Mean and (population) variance over the m logits present. */
static double mode_score(const double* x, int m, int mode) {
  if (mode == 0) return lse(x, m);
  double mean = 0.0;
  for (int i = 0; i < m; ++i) mean += x[i];
  mean /= m;
  if (mode == 1) return mean;
  double var = 0.0;
  for (int i = 0; i < m; ++i) var += (x[i] - mean) * (x[i] - mean);
  return mean + 0.5 * (var / m);
}

static int eligible(const walk_ctx* w, int l, int64_t i) {
  return !w->causal || node_start(w->lv, l, i) <= w->t;
}

/* ["Scoring: LogSumExp"] + [§4.1]: the score of candidate c at level l is, summed
 * over the query heads of the KV group, log sum_r exp(q_h . kbar_r / sqrt(d))
 * over c's eligible children r at level l-1 (raw keys when l == 1). */
static double block_score(const walk_ctx* w, int l, int64_t c) {
  const oracle_levels* lv = w->lv;
  double total = 0.0;
  for (int h = 0; h < w->G; ++h) {
    const float* qh = w->q + (int64_t)(w->kv * w->G + h) * w->d;
    int m = 0;
    if (l == 1) {
      int64_t s = node_start(lv, 1, c), e = node_end(lv, 1, c);
      for (int64_t r = s; r < e; ++r) {
        if (w->causal && r > w->t) break;
        double dot = 0.0;
        for (int j = 0; j < w->d; ++j)
          dot += (double)qh[j] * key_at(w->keys, w->n_cap, w->Hkv, w->d, w->b, r, w->kv, j);
        w->work[m++] = dot * w->scale;
      }
    } else {
      for (int k = 0; k < w->g; ++k) {
        int64_t r = c * w->g + k;
        if (r >= lv->M[l - 1] || !eligible(w, l - 1, r)) continue;
        const double* kb = w->pyr + (lv->off[l - 1] + r) * w->d;
        double dot = 0.0;
        for (int j = 0; j < w->d; ++j) dot += (double)qh[j] * kb[j];
        w->work[m++] = dot * w->scale;
      }
    }
    total += mode_score(w->work, m, w->mode); /* m >= 1: an eligible candidate's first child is */
  }
  return total;
}

/* Order for the Top-K: higher score first, lower node index on equal scores. */
static int better(double sa, int64_t ia, double sb, int64_t ib) {
  return sa > sb || (sa == sb && ia < ib);
}

/* [§3.2] coarse-to-fine walk for one query.  Writes the selected leaves in
 * ascending order (padded with -1) and their exact leaf scores (-inf padding).
 * Returns the number of levels that were scored; *min_gap receives the smallest
 * (K-th best - (K+1)-th best) score gap over those levels (+inf if none). */
static int walk_one(walk_ctx* w, int K, int32_t* idx_out, double* score_out, double* min_gap,
                    int64_t* S, int64_t* cand, double* cs, int64_t* order) {
  const oracle_levels* lv = w->lv;
  int nS = 1;
  S[0] = 0; /* the root */
  int n_scored = 0;
  double gap_min = INFINITY;
  for (int l = lv->L - 1; l >= 1; --l) {
    /* candidates: eligible children of the survivors, ascending */
    int nc = 0;
    for (int s = 0; s < nS; ++s)
      for (int k = 0; k < w->g; ++k) {
        int64_t c = S[s] * w->g + k;
        if (c < lv->M[l] && eligible(w, l, c)) cand[nc++] = c;
      }
    if (nc <= K) { /* [§3.2] at most K candidates: keep them all, no scoring */
      for (int i = 0; i < nc; ++i) S[i] = cand[i];
      nS = nc;
      continue;
    }
    ++n_scored;
    for (int i = 0; i < nc; ++i) cs[i] = block_score(w, l, cand[i]);
    /* rank candidates by (score desc, index asc): selection sort is enough here */
    for (int i = 0; i < nc; ++i) order[i] = i;
    for (int i = 0; i < nc; ++i) {
      int best = i;
      for (int j = i + 1; j < nc; ++j)
        if (better(cs[order[j]], cand[order[j]], cs[order[best]], cand[order[best]])) best = j;
      int64_t tmp = order[i];
      order[i] = order[best];
      order[best] = tmp;
    }
    double gap = cs[order[K - 1]] - cs[order[K]];
    if (gap < gap_min) gap_min = gap;
    /* survivors in ascending node order */
    nS = 0;
    for (int i = 0; i < nc; ++i) {
      int keep = 0;
      for (int j = 0; j < K; ++j)
        if (order[j] == i) keep = 1;
      if (keep) S[nS++] = cand[i];
    }
  }
  if (lv->L == 1) { /* a single leaf is the root */
    nS = 1;
    S[0] = 0;
  }
  for (int i = 0; i < K; ++i) {
    if (i < nS) {
      idx_out[i] = (int32_t)S[i];
      if (score_out) score_out[i] = block_score(w, 1, S[i]);
    } else {
      idx_out[i] = -1;
      if (score_out) score_out[i] = -INFINITY;
    }
  }
  if (min_gap) *min_gap = gap_min;
  return n_scored;
}

static int resolve_threads(int n_threads) {
#ifdef _OPENMP
  return n_threads > 0 ? n_threads : omp_get_max_threads();
#else
  (void)n_threads;
  return 1;
#endif
}

int pisa_oracle_max_threads(void) { return resolve_threads(0); }

/*
 * Prefill selection for a list of query positions.
 *   q      : [B][n_t][Hq][d]   query rows for the listed positions (fp32 of bf16)
 *   keys   : [B][N][Hkv][d]
 *   t_list : [n_t] query positions (each in [0, N))
 *   idx    : [B][Hkv][n_t][K]  selected leaves, ascending, -1 padded
 *   scores : [B][Hkv][n_t][K]  exact leaf scores of the selected leaves (nullable)
 *   min_gap: [B][Hkv][n_t]     smallest K-th minus (K+1)-th gap on the path (nullable)
 *   n_scored:[B][Hkv][n_t]     scored levels on the path (nullable)
 * Returns 0, or -1 on bad arguments.
 */
int pisa_oracle_select(const float* q, const float* keys, int B, int64_t N, int Hq, int Hkv, int d,
                       int C, int g, int K, int causal, const int64_t* t_list, int64_t n_t,
                       int32_t* idx, double* scores, double* min_gap, int32_t* n_scored,
                       int n_threads, int mode) {
  oracle_levels lv;
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || K < 1 || levels_init(&lv, N, C, g)) return -1;
  for (int64_t i = 0; i < n_t; ++i)
    if (t_list[i] < 0 || t_list[i] >= N) return -1;
  const int G = Hq / Hkv;
  double* pyr = (double*)malloc(sizeof(double) * (size_t)B * Hkv * lv.total * d);
  if (!pyr) return -1;
  pisa_oracle_build_pyramid(keys, B, N, N, Hkv, d, C, g, 0, pyr);
  const int64_t jobs = (int64_t)B * Hkv * n_t;
  const int nt = resolve_threads(n_threads);
  const int cap = 2 * g * K + 8;
#pragma omp parallel num_threads(nt)
  {
    int64_t* S = (int64_t*)malloc(sizeof(int64_t) * cap);
    int64_t* cand = (int64_t*)malloc(sizeof(int64_t) * cap);
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * cap);
    double* cs = (double*)malloc(sizeof(double) * cap);
    double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
#pragma omp for schedule(dynamic, 16)
    for (int64_t job = 0; job < jobs; ++job) {
      int64_t it = job % n_t;
      int kv = (int)((job / n_t) % Hkv);
      int b = (int)(job / (n_t * Hkv));
      walk_ctx w;
      w.q = q + ((int64_t)b * n_t + it) * Hq * d;
      w.keys = keys;
      w.pyr = pyr + ((int64_t)b * Hkv + kv) * lv.total * d;
      w.lv = &lv;
      w.n_cap = N;
      w.b = b;
      w.kv = kv;
      w.Hkv = Hkv;
      w.G = G;
      w.d = d;
      w.g = g;
      w.causal = causal;
      w.t = t_list[it];
      w.scale = 1.0 / sqrt((double)d);
      w.work = work;
      w.mode = mode;
      int64_t o = ((int64_t)b * Hkv + kv) * n_t + it;
      int ns = walk_one(&w, K, idx + o * K, scores ? scores + o * K : NULL,
                        min_gap ? min_gap + o : NULL, S, cand, cs, order);
      if (n_scored) n_scored[o] = ns;
    }
    free(S);
    free(cand);
    free(order);
    free(cs);
    free(work);
  }
  free(pyr);
  return 0;
}

/*
 * Flat block selection, the conventional stage-1 baseline ([P1]: block-sparse
 * attention such as BSA scores all N/C key blocks for every query): every
 * eligible leaf gets the leaf score of ["Scoring: LogSumExp"] (exact raw-key
 * LSE summed over the group's heads, keys after t masked when causal) and the K
 * best are kept, ties to the lower index, listed ascending with -1 padding.
 *   idx    : [B][Hkv][n_t][K], scores: [B][Hkv][n_t][K] (nullable)
 *   min_gap: [B][Hkv][n_t] K-th best minus (K+1)-th best (+inf when at most K
 *            leaves are eligible) (nullable)
 */
int pisa_oracle_flat_select(const float* q, const float* keys, int B, int64_t N, int Hq, int Hkv, int d,
                            int C, int g, int K, int causal, const int64_t* t_list, int64_t n_t,
                            int32_t* idx, double* scores, double* min_gap, int n_threads, int mode) {
  oracle_levels lv;
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || K < 1 || levels_init(&lv, N, C, g)) return -1;
  for (int64_t i = 0; i < n_t; ++i)
    if (t_list[i] < 0 || t_list[i] >= N) return -1;
  const int G = Hq / Hkv;
  const int64_t M1 = lv.M[1];
  const int64_t jobs = (int64_t)B * Hkv * n_t;
  const int nt = resolve_threads(n_threads);
#pragma omp parallel num_threads(nt)
  {
    double* cs = (double*)malloc(sizeof(double) * (size_t)M1);
    char* taken = (char*)malloc((size_t)M1);
    int64_t* best = (int64_t*)malloc(sizeof(int64_t) * (size_t)(K + 1));
    double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
#pragma omp for schedule(dynamic, 4)
    for (int64_t job = 0; job < jobs; ++job) {
      int64_t it = job % n_t;
      int kv = (int)((job / n_t) % Hkv);
      int b = (int)(job / (n_t * Hkv));
      walk_ctx w;
      memset(&w, 0, sizeof(w));
      w.q = q + ((int64_t)b * n_t + it) * Hq * d;
      w.keys = keys;
      w.lv = &lv;
      w.n_cap = N;
      w.b = b;
      w.kv = kv;
      w.Hkv = Hkv;
      w.G = G;
      w.d = d;
      w.g = g;
      w.causal = causal;
      w.t = t_list[it];
      w.scale = 1.0 / sqrt((double)d);
      w.work = work;
      w.mode = mode;
      int64_t nc = 0; /* eligible leaves are a prefix: 0 .. nc-1 */
      while (nc < M1 && eligible(&w, 1, nc)) ++nc;
      for (int64_t c = 0; c < nc; ++c) {
        cs[c] = block_score(&w, 1, c);
        taken[c] = 0;
      }
      /* the K+1 best by (score desc, index asc), one pass per rank */
      int nb = 0;
      for (; nb < K + 1 && nb < nc; ++nb) {
        int64_t pick = -1;
        for (int64_t c = 0; c < nc; ++c)
          if (!taken[c] && (pick < 0 || better(cs[c], c, cs[pick], pick))) pick = c;
        taken[pick] = 1;
        best[nb] = pick;
      }
      int64_t o = ((int64_t)b * Hkv + kv) * n_t + it;
      if (min_gap) min_gap[o] = nc > K ? cs[best[K - 1]] - cs[best[K]] : INFINITY;
      int w_out = 0;
      for (int64_t c = 0; c < nc && w_out < K; ++c)
        if (taken[c] && (nc <= K || c != best[K])) {
          idx[o * K + w_out] = (int32_t)c;
          if (scores) scores[o * K + w_out] = cs[c];
          ++w_out;
        }
      for (; w_out < K; ++w_out) {
        idx[o * K + w_out] = -1;
        if (scores) scores[o * K + w_out] = -INFINITY;
      }
    }
    free(cs);
    free(taken);
    free(best);
    free(work);
  }
  return 0;
}

/*
 * Stage two of block-sparse attention ([P2] "Background: two stages": each query
 * attends over the original keys and values inside its selected blocks).  For
 * query position t and query head h of KV group kv:
 *   o = sum_r softmax_r(q . k_r / sqrt(d)) v_r
 * over the keys r of the selected leaves idx[b][kv][it][0..K) (entries < 0 are
 * skipped), keys after t masked when causal; one softmax over all of them.
 *   q  : [B][n_t][Hq][d] rows of t_list; k, v: [B][N][Hkv][d]
 *   out: [B][n_t][Hq][d] (a row with no key is all zeros)
 */
int pisa_oracle_attention(const float* q, const float* keys, const float* vals, int B, int64_t N, int Hq,
                          int Hkv, int d, int C, int causal, const int64_t* t_list, int64_t n_t, int K,
                          const int32_t* idx, double* out, int n_threads) {
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || C <= 0 || K < 1) return -1;
  for (int64_t i = 0; i < n_t; ++i)
    if (t_list[i] < 0 || t_list[i] >= N) return -1;
  const int G = Hq / Hkv;
  const int nt = resolve_threads(n_threads);
  const int64_t jobs = (int64_t)B * n_t * Hq;
  const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel num_threads(nt)
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)K * C);
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)K * C);
#pragma omp for schedule(dynamic, 16)
    for (int64_t job = 0; job < jobs; ++job) {
      const int h = (int)(job % Hq);
      const int64_t it = (job / Hq) % n_t;
      const int b = (int)(job / (Hq * n_t));
      const int kv = h / G;
      const int64_t t = t_list[it];
      const float* qh = q + (((int64_t)b * n_t + it) * Hq + h) * d;
      const int32_t* sel = idx + (((int64_t)b * Hkv + kv) * n_t + it) * K;
      int m = 0;
      for (int i = 0; i < K; ++i) {
        if (sel[i] < 0) continue;
        for (int64_t r = (int64_t)sel[i] * C; r < (int64_t)(sel[i] + 1) * C && r < N; ++r) {
          if (causal && r > t) break;
          double dot = 0.0;
          for (int j = 0; j < d; ++j) dot += (double)qh[j] * key_at(keys, N, Hkv, d, b, r, kv, j);
          z[m] = dot * scale;
          rows[m++] = r;
        }
      }
      double* o = out + (((int64_t)b * n_t + it) * Hq + h) * d;
      for (int j = 0; j < d; ++j) o[j] = 0.0;
      if (m == 0) continue;
      double mx = z[0];
      for (int i = 1; i < m; ++i)
        if (z[i] > mx) mx = z[i];
      double den = 0.0;
      for (int i = 0; i < m; ++i) den += exp(z[i] - mx);
      for (int i = 0; i < m; ++i) {
        const double p = exp(z[i] - mx) / den;
        for (int j = 0; j < d; ++j) o[j] += p * key_at(vals, N, Hkv, d, b, rows[i], kv, j);
      }
    }
    free(z);
    free(rows);
  }
  return 0;
}

/*
 * Decode selection ([P1] decoding keeps a cached mean pyramid and walks for the
 * one new query).  By definition it equals the prefill walk of the last query
 * over the keys present, so this routine rebuilds the pyramid over the first
 * lengths[b] tokens of each sequence and walks t = lengths[b] - 1.
 *   q      : [B][Hq][d]         the new query of each sequence
 *   keys   : [B][n_cap][Hkv][d] key cache holding lengths[b] valid tokens
 *   idx    : [B][Hkv][K], scores: [B][Hkv][K] (nullable), min_gap: [B][Hkv]
 */
int pisa_oracle_select_last(const float* q, const float* keys, int B, int64_t n_cap,
                            const int64_t* lengths, int Hq, int Hkv, int d, int C, int g, int K,
                            int32_t* idx, double* scores, double* min_gap, int32_t* n_scored,
                            int n_threads) {
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || K < 1) return -1;
  for (int b = 0; b < B; ++b)
    if (lengths[b] < 1 || lengths[b] > n_cap) return -1;
  const int G = Hq / Hkv;
  const int nt = resolve_threads(n_threads);
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int64_t job = 0; job < (int64_t)B * Hkv; ++job) {
    int b = (int)(job / Hkv), kv = (int)(job % Hkv);
    oracle_levels lv;
    if (levels_init(&lv, lengths[b], C, g)) {
      err = 1;
      continue;
    }
    double* pyr = (double*)malloc(sizeof(double) * (size_t)lv.total * d);
    /* the same direct means, over this sequence's tokens only */
    const float* kb = keys + (int64_t)b * n_cap * Hkv * d;
    build_direct(kb, n_cap, Hkv, d, 0, kv, &lv, pyr);
    int cap = 2 * g * K + 8;
    int64_t* S = (int64_t*)malloc(sizeof(int64_t) * cap);
    int64_t* cand = (int64_t*)malloc(sizeof(int64_t) * cap);
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * cap);
    double* cs = (double*)malloc(sizeof(double) * cap);
    double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
    walk_ctx w;
    w.q = q + (int64_t)b * Hq * d;
    w.keys = kb;
    w.pyr = pyr;
    w.lv = &lv;
    w.n_cap = n_cap;
    w.b = 0;
    w.kv = kv;
    w.Hkv = Hkv;
    w.G = G;
    w.d = d;
    w.g = g;
    w.causal = 1;
    w.t = lengths[b] - 1;
    w.scale = 1.0 / sqrt((double)d);
    w.work = work;
    w.mode = 0; /* decode: LSE only */
    int64_t o = job;
    int ns = walk_one(&w, K, idx + o * K, scores ? scores + o * K : NULL,
                      min_gap ? min_gap + o : NULL, S, cand, cs, order);
    if (n_scored) n_scored[o] = ns;
    free(S);
    free(cand);
    free(order);
    free(cs);
    free(work);
    free(pyr);
  }
  return err ? -1 : 0;
}

/*
 * Exact leaf score of arbitrary leaves for given query positions: the summed
 * raw-key LSE of ["Scoring: LogSumExp"] at the leaf level.  Used to check the
 * validity of a selection that legitimately differs from the oracle's on a
 * near tie.  leaves: [B][Hkv][n_t][K] (-1 entries give -inf); out likewise.
 */
int pisa_oracle_leaf_scores(const float* q, const float* keys, int B, int64_t N, int Hq, int Hkv,
                            int d, int C, int g, int causal, const int64_t* t_list, int64_t n_t,
                            int K, const int32_t* leaves, double* out, int n_threads, int mode) {
  oracle_levels lv;
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || levels_init(&lv, N, C, g)) return -1;
  const int G = Hq / Hkv;
  const int nt = resolve_threads(n_threads);
  const int64_t jobs = (int64_t)B * Hkv * n_t;
#pragma omp parallel num_threads(nt)
  {
    double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
#pragma omp for schedule(dynamic, 16)
    for (int64_t job = 0; job < jobs; ++job) {
      int64_t it = job % n_t;
      int kv = (int)((job / n_t) % Hkv);
      int b = (int)(job / (n_t * Hkv));
      walk_ctx w;
      memset(&w, 0, sizeof(w));
      w.q = q + ((int64_t)b * n_t + it) * Hq * d;
      w.keys = keys;
      w.lv = &lv;
      w.n_cap = N;
      w.b = b;
      w.kv = kv;
      w.Hkv = Hkv;
      w.G = G;
      w.d = d;
      w.g = g;
      w.causal = causal;
      w.t = t_list[it];
      w.scale = 1.0 / sqrt((double)d);
      w.work = work;
      w.mode = mode;
      for (int k = 0; k < K; ++k) {
        int64_t o = job * K + k;
        int32_t c = leaves[o];
        if (c < 0 || c >= lv.M[1] || !eligible(&w, 1, c))
          out[o] = -INFINITY;
        else
          out[o] = block_score(&w, 1, c);
      }
    }
    free(work);
  }
  return 0;
}

/*
 * Score of one candidate node for one query, for the invariants of the tests:
 * level >= 2 uses the children's summaries (pyramid over all N tokens), level 1
 * the raw keys.  Returns the head-summed score of node c at level l for the
 * query q ([Hq][d]) of group kv at position t.
 */
double pisa_oracle_node_score(const float* q, const float* keys, int64_t N, int Hq, int Hkv, int d,
                              int C, int g, int causal, int kv, int64_t t, int level, int64_t c, int mode) {
  oracle_levels lv;
  if (levels_init(&lv, N, C, g) || level < 1 || level > lv.L || c < 0 || c >= lv.M[level])
    return NAN;
  double* pyr = (double*)malloc(sizeof(double) * (size_t)lv.total * d);
  build_direct(keys, N, Hkv, d, 0, kv, &lv, pyr);
  double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
  walk_ctx w;
  w.q = q;
  w.keys = keys;
  w.pyr = pyr;
  w.lv = &lv;
  w.n_cap = N;
  w.b = 0;
  w.kv = kv;
  w.Hkv = Hkv;
  w.G = Hq / Hkv;
  w.d = d;
  w.g = g;
  w.causal = causal;
  w.t = t;
  w.scale = 1.0 / sqrt((double)d);
  w.work = work;
  w.mode = mode;
  double s = block_score(&w, level, c);
  free(work);
  free(pyr);
  return s;
}

/* ------------------------------------------------------------------------------
 * Checking a selection that differs from the oracle's ([§3.2] walk, ["Scoring:
 * LogSumExp"] scores).  Where two candidates' scores are closer than `tie`,
 * either order is a correct answer, so more than one leaf set can be correct.
 * A leaf set is accepted iff some walk that breaks such near ties either way
 * produces it:
 *   - at a level with at most K eligible candidates every candidate is kept;
 *   - at a scored level the kept set S (|S| = K) is a near Top-K of the
 *     candidates: every candidate left out scores less than min_{s in S}
 *     score(s) + tie;
 *   - at the leaf level the kept set is the given leaf set itself.
 * At an intermediate level the kept set must contain the ancestors of the given
 * leaves; the other survivors are not visible in the output, so every near-Top-K
 * completion is tried (depth first; the number of completions is tiny unless
 * many candidates sit within `tie` of each other, and a node budget bounds it).
 * Verdict: 1 reachable, 0 not reachable (or malformed), -1 budget exhausted.
 * ---------------------------------------------------------------------------- */

typedef struct {
  walk_ctx* w;
  int K;
  double tie;
  int64_t budget;
  int cap;               /* g*K + 8: room for one level's candidates           */
  int64_t* anc;          /* [L+1][K]: ancestors of the given leaves per level */
  int n_anc[ORACLE_MAX_LEVELS + 1];
  int64_t* cand;         /* [L+1][cap] candidates per level                   */
  double* cs;            /* [L+1][cap] their scores                           */
  int64_t* rest;         /* [L+1][cap] candidates not among the ancestors     */
  double* rest_s;        /* [L+1][cap]                                        */
  int64_t* pick;         /* [L+1][cap] chosen completion                      */
  int64_t* next;         /* [L+1][cap] kept set handed to the level below     */
} check_ctx;

static int check_level(check_ctx* c, int l, const int64_t* S, int nS);

/* Depth-first search over the completions of level l: rest[] is sorted by score
 * (descending); `need` more members are still to be chosen from rest[pos..].
 * cur_min = lowest score kept so far (ancestors included), max_out = highest
 * score left out so far.  A completion is legal iff max_out - cur_min < tie. */
static int complete(check_ctx* c, int l, int pos, int nrest, int chosen, int need, double cur_min,
                    double max_out) {
  if (--c->budget < 0) return -1;
  int64_t* rest = c->rest + (int64_t)l * c->cap;
  double* rs = c->rest_s + (int64_t)l * c->cap;
  int64_t* pick = c->pick + (int64_t)l * c->cap;
  if (chosen == need) {
    double mo = max_out;
    if (pos < nrest && rs[pos] > mo) mo = rs[pos]; /* the rest are left out */
    if (!(mo - cur_min < c->tie)) return 0;
    /* kept set = ancestors + picks, ascending */
    const int64_t* A = c->anc + (int64_t)l * c->K;
    int nA = c->n_anc[l];
    int64_t* nx = c->next + (int64_t)l * c->cap;
    int n = 0;
    for (int i = 0; i < nA; ++i) nx[n++] = A[i];
    for (int i = 0; i < chosen; ++i) nx[n++] = pick[i];
    for (int i = 1; i < n; ++i) { /* insertion sort by index */
      int64_t v = nx[i];
      int j = i - 1;
      while (j >= 0 && nx[j] > v) {
        nx[j + 1] = nx[j];
        --j;
      }
      nx[j + 1] = v;
    }
    return check_level(c, l - 1, nx, n);
  }
  if (nrest - pos < need - chosen) return 0;
  int undecided = 0;
  /* keep rest[pos] */
  double nmin = rs[pos] < cur_min ? rs[pos] : cur_min;
  if (max_out - nmin < c->tie) {
    pick[chosen] = rest[pos];
    int r = complete(c, l, pos + 1, nrest, chosen + 1, need, nmin, max_out);
    if (r == 1) return 1;
    if (r < 0) undecided = 1;
  }
  /* leave rest[pos] out */
  double nmax = rs[pos] > max_out ? rs[pos] : max_out;
  if (nmax - cur_min < c->tie) {
    int r = complete(c, l, pos + 1, nrest, chosen, need, cur_min, nmax);
    if (r == 1) return 1;
    if (r < 0) undecided = 1;
  }
  return undecided ? -1 : 0;
}

/* Level l's candidates are the eligible children of the kept set S of level l+1. */
static int check_level(check_ctx* c, int l, const int64_t* S, int nS) {
  walk_ctx* w = c->w;
  const oracle_levels* lv = w->lv;
  const int K = c->K;
  int64_t* cand = c->cand + (int64_t)l * c->cap;
  double* cs = c->cs + (int64_t)l * c->cap;
  const int64_t* A = c->anc + (int64_t)l * K;
  const int nA = c->n_anc[l];
  int nc = 0;
  for (int s = 0; s < nS; ++s)
    for (int k = 0; k < w->g; ++k) {
      int64_t ch = S[s] * w->g + k;
      if (ch < lv->M[l] && eligible(w, l, ch)) cand[nc++] = ch;
    }
  /* the ancestors must be candidates (both lists ascending) */
  int member[64 * 2 + 8];
  int j = 0;
  for (int i = 0; i < nc; ++i) member[i] = 0;
  for (int a = 0; a < nA; ++a) {
    while (j < nc && cand[j] < A[a]) ++j;
    if (j == nc || cand[j] != A[a]) return 0;
    member[j] = 1;
  }
  if (nc <= K) { /* kept whole, unscored */
    if (l == 1) return nA == nc;
    return check_level(c, l - 1, cand, nc);
  }
  if (nA > K) return 0;
  for (int i = 0; i < nc; ++i) cs[i] = block_score(w, l, cand[i]);
  double min_in = INFINITY;
  for (int i = 0; i < nc; ++i)
    if (member[i] && cs[i] < min_in) min_in = cs[i];
  if (l == 1) { /* the kept set is the given leaf set */
    if (nA != K) return 0;
    for (int i = 0; i < nc; ++i)
      if (!member[i] && !(cs[i] - min_in < c->tie)) return 0;
    return 1;
  }
  /* the other survivors: near-Top-K completions of the ancestors */
  int64_t* rest = c->rest + (int64_t)l * c->cap;
  double* rs = c->rest_s + (int64_t)l * c->cap;
  int nr = 0;
  for (int i = 0; i < nc; ++i)
    if (!member[i]) {
      int p = nr++; /* insertion by (score desc, index asc) */
      while (p > 0 && (rs[p - 1] < cs[i] || (rs[p - 1] == cs[i] && rest[p - 1] > cand[i]))) {
        rs[p] = rs[p - 1];
        rest[p] = rest[p - 1];
        --p;
      }
      rs[p] = cs[i];
      rest[p] = cand[i];
    }
  return complete(c, l, 0, nr, 0, K - nA, min_in, -INFINITY);
}

/* Well-formed row: ascending distinct leaves, then -1 padding. */
static int row_well_formed(const int32_t* sel, int K, int64_t M1, int* n_sel) {
  int n = 0;
  while (n < K && sel[n] >= 0) ++n;
  for (int i = n; i < K; ++i)
    if (sel[i] != -1) return 0;
  for (int i = 0; i < n; ++i) {
    if (sel[i] >= M1) return 0;
    if (i && sel[i] <= sel[i - 1]) return 0;
  }
  *n_sel = n;
  return 1;
}

/* One query: the walk re-taken along the given leaves (flat = 0), or the flat
 * selection's near-Top-K rule over every eligible leaf (flat = 1). */
static int check_one(walk_ctx* w, int K, const int32_t* sel, double tie, int flat, int64_t budget,
                     check_ctx* c) {
  const oracle_levels* lv = w->lv;
  int n_sel;
  if (!row_well_formed(sel, K, lv->M[1], &n_sel)) return 0;
  if (flat) {
    int64_t nc = 0; /* eligible leaves are a prefix */
    while (nc < lv->M[1] && eligible(w, 1, nc)) ++nc;
    if (n_sel != (nc < K ? nc : K)) return 0;
    for (int i = 0; i < n_sel; ++i)
      if (sel[i] >= nc) return 0;
    if (nc <= K) return 1;
    double min_in = INFINITY;
    for (int i = 0; i < n_sel; ++i) {
      double s = block_score(w, 1, sel[i]);
      if (s < min_in) min_in = s;
    }
    int j = 0;
    for (int64_t leaf = 0; leaf < nc; ++leaf) {
      if (j < n_sel && sel[j] == leaf) {
        ++j;
        continue;
      }
      if (!(block_score(w, 1, leaf) - min_in < tie)) return 0;
    }
    return 1;
  }
  if (n_sel == 0) return 0;
  /* ancestors of the given leaves at every level (distinct, ascending) */
  for (int l = 1; l <= lv->L; ++l) {
    int64_t* A = c->anc + (int64_t)l * K;
    int n = 0;
    for (int i = 0; i < n_sel; ++i) {
      int64_t a = sel[i] / (lv->width[l] / lv->width[1]);
      if (n == 0 || A[n - 1] != a) A[n++] = a;
    }
    c->n_anc[l] = n;
  }
  if (lv->L == 1) return n_sel == 1 && sel[0] == 0; /* a single leaf is the root */
  c->w = w;
  c->K = K;
  c->tie = tie;
  c->budget = budget;
  int64_t root = 0;
  return check_level(c, lv->L - 1, &root, 1);
}

static int check_alloc(check_ctx* c, const oracle_levels* lv, int K, int g) {
  memset(c, 0, sizeof(*c));
  c->cap = g * K + 8;
  size_t n = (size_t)(lv->L + 1) * c->cap;
  c->anc = (int64_t*)malloc(sizeof(int64_t) * (size_t)(lv->L + 1) * K);
  c->cand = (int64_t*)malloc(sizeof(int64_t) * n);
  c->cs = (double*)malloc(sizeof(double) * n);
  c->rest = (int64_t*)malloc(sizeof(int64_t) * n);
  c->rest_s = (double*)malloc(sizeof(double) * n);
  c->pick = (int64_t*)malloc(sizeof(int64_t) * n);
  c->next = (int64_t*)malloc(sizeof(int64_t) * n);
  return c->anc && c->cand && c->cs && c->rest && c->rest_s && c->pick && c->next ? 0 : -1;
}

static void check_free(check_ctx* c) {
  free(c->anc);
  free(c->cand);
  free(c->cs);
  free(c->rest);
  free(c->rest_s);
  free(c->pick);
  free(c->next);
}

#define CHECK_BUDGET ((int64_t)1 << 22)

/*
 * Is each given prefill selection one that the walk (flat = 0) or the flat
 * selector (flat = 1) reaches when near ties (score differences below `tie`)
 * are broken either way?
 *   q      : [B][n_t][Hq][d] rows of t_list; keys: [B][N][Hkv][d]
 *   sel    : [B][Hkv][n_t][K] leaf sets to check (ascending, -1 padded)
 *   verdict: [B][Hkv][n_t]  1 reachable, 0 not (or malformed), -1 undecided
 */
int pisa_oracle_check_selection(const float* q, const float* keys, int B, int64_t N, int Hq, int Hkv,
                                int d, int C, int g, int K, int causal, const int64_t* t_list,
                                int64_t n_t, const int32_t* sel, double tie, int flat, int mode,
                                int32_t* verdict, int n_threads) {
  oracle_levels lv;
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || K < 1 || K > 64 || g > 2 || !(tie > 0) ||
      levels_init(&lv, N, C, g))
    return -1;
  for (int64_t i = 0; i < n_t; ++i)
    if (t_list[i] < 0 || t_list[i] >= N) return -1;
  const int G = Hq / Hkv;
  double* pyr = NULL;
  if (!flat) {
    pyr = (double*)malloc(sizeof(double) * (size_t)B * Hkv * lv.total * d);
    if (!pyr) return -1;
    pisa_oracle_build_pyramid(keys, B, N, N, Hkv, d, C, g, 0, pyr);
  }
  const int64_t jobs = (int64_t)B * Hkv * n_t;
  const int nt = resolve_threads(n_threads);
  int err = 0;
#pragma omp parallel num_threads(nt)
  {
    check_ctx c;
    double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
    if (check_alloc(&c, &lv, K, g) || !work) err = 1;
#pragma omp for schedule(dynamic, 4)
    for (int64_t job = 0; job < jobs; ++job) {
      if (err) continue;
      int64_t it = job % n_t;
      int kv = (int)((job / n_t) % Hkv);
      int b = (int)(job / (n_t * Hkv));
      walk_ctx w;
      memset(&w, 0, sizeof(w));
      w.q = q + ((int64_t)b * n_t + it) * Hq * d;
      w.keys = keys;
      w.pyr = pyr ? pyr + ((int64_t)b * Hkv + kv) * lv.total * d : NULL;
      w.lv = &lv;
      w.n_cap = N;
      w.b = b;
      w.kv = kv;
      w.Hkv = Hkv;
      w.G = G;
      w.d = d;
      w.g = g;
      w.causal = causal;
      w.t = t_list[it];
      w.scale = 1.0 / sqrt((double)d);
      w.work = work;
      w.mode = mode;
      int64_t o = ((int64_t)b * Hkv + kv) * n_t + it;
      verdict[o] = check_one(&w, K, sel + o * K, tie, flat, CHECK_BUDGET, &c);
    }
    check_free(&c);
    free(work);
  }
  free(pyr);
  return err ? -1 : 0;
}

/*
 * The same check for decode selections: sequence b's newest query (t =
 * lengths[b] - 1) over its lengths[b] keys, pyramid over those keys only.
 *   q: [B][Hq][d]; keys: [B][n_cap][Hkv][d]; sel: [B][Hkv][K]; verdict: [B][Hkv]
 */
int pisa_oracle_check_last(const float* q, const float* keys, int B, int64_t n_cap,
                           const int64_t* lengths, int Hq, int Hkv, int d, int C, int g, int K,
                           const int32_t* sel, double tie, int32_t* verdict, int n_threads) {
  if (B <= 0 || Hkv <= 0 || Hq % Hkv || K < 1 || K > 64 || g > 2 || !(tie > 0)) return -1;
  for (int b = 0; b < B; ++b)
    if (lengths[b] < 1 || lengths[b] > n_cap) return -1;
  const int G = Hq / Hkv;
  const int nt = resolve_threads(n_threads);
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int64_t job = 0; job < (int64_t)B * Hkv; ++job) {
    int b = (int)(job / Hkv), kv = (int)(job % Hkv);
    oracle_levels lv;
    check_ctx c;
    if (levels_init(&lv, lengths[b], C, g) || check_alloc(&c, &lv, K, g)) {
      err = 1;
      continue;
    }
    double* pyr = (double*)malloc(sizeof(double) * (size_t)lv.total * d);
    double* work = (double*)malloc(sizeof(double) * (C > g ? C : g));
    const float* kb = keys + (int64_t)b * n_cap * Hkv * d;
    build_direct(kb, n_cap, Hkv, d, 0, kv, &lv, pyr);
    walk_ctx w;
    memset(&w, 0, sizeof(w));
    w.q = q + (int64_t)b * Hq * d;
    w.keys = kb;
    w.pyr = pyr;
    w.lv = &lv;
    w.n_cap = n_cap;
    w.b = 0;
    w.kv = kv;
    w.Hkv = Hkv;
    w.G = G;
    w.d = d;
    w.g = g;
    w.causal = 1;
    w.t = lengths[b] - 1;
    w.scale = 1.0 / sqrt((double)d);
    w.work = work;
    w.mode = 0;
    verdict[job] = check_one(&w, K, sel + job * K, tie, 0, CHECK_BUDGET, &c);
    check_free(&c);
    free(pyr);
    free(work);
  }
  return err ? -1 : 0;
}
