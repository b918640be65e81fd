/*
 * spec_oracle.c -- CPU oracle for batched tree speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, fp64 statement of
 * what the verify step computes.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (cited by page and section):
 *   [tutorial]    "LLM speculative decoding: EAGLE" (jingming.pro), sections
 *                 1 (note on sampling transforms), 2.3 (accept/reject steps),
 *                 2.4 (worked example), 3.4 (candidate-tree verification).
 *   [eagle3]      EAGLE-3 article (mokono.cn), section 6 (worked verify example).
 *   [reading]     "EAGLE close reading" (edgeai1.github.io knowledge base),
 *                 section 3 (tree and distribution preservation), section 5
 *                 (greedy must match the target token by token).
 *   [translation] EAGLE / EAGLE-2 paper translation (modelers.csdn.net),
 *                 section 1.3.2 (verification: recursive speculative sampling at
 *                 every node, as in SpecInfer) and section 1.7 (multi-round
 *                 speculative sampling: after a rejection call the sampler again
 *                 on the next candidate; if all are rejected sample the adjusted
 *                 distribution).
 *   [philox]      Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *                 as 1, 2, 3", SC'11 -- the Philox4x32-10 bijection.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - transforms are applied in the order temperature -> top-k -> top-p, both
 *     to the target row p and the draft row q; ranking is by raw logit, ties to
 *     the lower vocabulary index; top-p keeps the shortest prefix whose
 *     normalised mass is >= top_p;
 *   - siblings are tried in increasing node index, each against the same q of
 *     their parent; acceptance is r <= p/q with r in (0, 1];
 *   - a residual whose mass is exactly zero leaves p unchanged;
 *   - the final token is drawn by inverse CDF in vocabulary-index order;
 *   - uniforms come from Philox4x32-10, key = seed, counter = (node, batch,
 *     offset_lo, offset_hi); word 0 drives the accept test at a child, word 1
 *     the final draw at a node; U = ((x >> 8) + 1) * 2^-24.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_NEAR 1e-6

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 ([philox], section 3: the Philox S-box is two 32x32->64     */
/* multiplications per round, ten rounds, the key advanced by the Weyl       */
/* constants between rounds).                                                */
/* ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
  const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = (uint64_t)mult0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)mult1 * (uint64_t)c2;
    uint32_t n0 = (uint32_t)(prod1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)prod1;
    uint32_t n2 = (uint32_t)(prod0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)prod0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* U(x) = ((x >> 8) + 1) * 2^-24, a uniform on (0, 1] that is exact in fp32. */
double oracle_uniform_from_word(uint32_t x) {
  return (double)((x >> 8) + 1u) * (1.0 / 16777216.0);
}

/* The uniform for (seed, offset, batch b, node n); word 0 = accept test, 1 = final draw. */
double oracle_uniform(uint64_t seed, uint64_t offset, int32_t b, int32_t node, int word) {
  uint32_t ctr[4] = {(uint32_t)node, (uint32_t)b, (uint32_t)offset, (uint32_t)(offset >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return oracle_uniform_from_word(out[word]);
}

/* ------------------------------------------------------------------------- */
/* Logit loading: fp32, or bf16 given as its raw 16 bits (exact widening).   */
/* ------------------------------------------------------------------------- */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

static double load_logit(const void* base, int dtype, int64_t elem) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[elem];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[elem]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Sampling transforms ([tutorial] section 1 note: p and q are compared       */
/* after temperature / top-k / top-p / argmax processing).                   */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t status;   /* 0 ok, 1 non-finite row (NaN or +inf present, or all -inf) */
  int32_t argmax;   /* lowest index of the maximum logit */
  int32_t kept;     /* number of tokens with nonzero filtered probability slot */
  int32_t cut_idx;  /* vocabulary index of the last kept token in rank order */
  double m;         /* maximum logit */
  double cut_z;     /* logit of the last kept token */
  double s_k;       /* sum over the top-k set of exp((z - m) / T) */
  double s_f;       /* sum over the kept set of exp((z - m) / T) */
  int32_t near;     /* top-p decision within ORACLE_NEAR of its threshold */
  int32_t pad;
  double margin;    /* distance of the top-p decision from top_p (normalised mass) */
} oracle_row_info;

typedef struct {
  double z;
  int32_t idx;
} ranked_t;

/* Rank order: larger logit first, equal logits by lower vocabulary index. */
static int rank_cmp(const void* a, const void* b) {
  const ranked_t* x = (const ranked_t*)a;
  const ranked_t* y = (const ranked_t*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/*
 * Filter one row of logits into a probability vector.
 *   T == 0     : one-hot at the argmax (greedy).
 *   T  > 0     : weights exp((z - m) / T); top-k keeps the first k in rank
 *                order (when 0 < k < V); top-p keeps the shortest rank-order
 *                prefix of the top-k set whose normalised mass is >= top_p
 *                (when top_p < 1); the kept weights are renormalised.
 * prob may be NULL.  Returns info->status.
 */
int oracle_filter_row(const void* row, int dtype, int V, double T, int top_k, double top_p,
                      double* prob, oracle_row_info* info) {
  memset(info, 0, sizeof *info);
  info->argmax = -1;
  info->cut_idx = -1;
  if (prob) for (int i = 0; i < V; ++i) prob[i] = 0.0;

  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  int bad = 0, all_neg_inf = 1;
  for (int i = 0; i < V; ++i) {
    z[i] = load_logit(row, dtype, i);
    if (isnan(z[i]) || (isinf(z[i]) && z[i] > 0)) bad = 1;
    if (!(isinf(z[i]) && z[i] < 0)) all_neg_inf = 0;
  }
  if (bad || all_neg_inf || V <= 0) {
    info->status = 1;
    free(z);
    return 1;
  }
  double m = z[0];
  int am = 0;
  for (int i = 1; i < V; ++i)
    if (z[i] > m) { m = z[i]; am = i; }
  info->m = m;
  info->argmax = am;

  if (T == 0.0) {
    info->kept = 1;
    info->cut_idx = am;
    info->cut_z = m;
    info->s_k = 1.0;
    info->s_f = 1.0;
    info->margin = INFINITY;
    if (prob) prob[am] = 1.0;
    free(z);
    return 0;
  }

  ranked_t* r = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)V);
  for (int i = 0; i < V; ++i) { r[i].z = z[i]; r[i].idx = i; }
  qsort(r, (size_t)V, sizeof(ranked_t), rank_cmp);

  int K = (top_k > 0 && top_k < V) ? top_k : V;
  double* w = (double*)malloc(sizeof(double) * (size_t)K);
  double s_k = 0.0;
  for (int j = 0; j < K; ++j) {
    w[j] = exp((r[j].z - m) / T);
    s_k += w[j];
  }

  int n_keep = K;
  double margin = INFINITY;
  if (top_p < 1.0) {
    double cum = 0.0;
    for (int j = 0; j < K; ++j) {
      double prev = cum;
      cum += w[j];
      if (cum / s_k >= top_p) {
        n_keep = j + 1;
        double above = cum / s_k - top_p;
        double below = top_p - prev / s_k;
        margin = above < below ? above : below;
        break;
      }
    }
  }
  double s_f = 0.0;
  for (int j = 0; j < n_keep; ++j) s_f += w[j];
  if (prob)
    for (int j = 0; j < n_keep; ++j) prob[r[j].idx] = w[j] / s_f;

  info->kept = n_keep;
  info->cut_idx = r[n_keep - 1].idx;
  info->cut_z = r[n_keep - 1].z;
  info->s_k = s_k;
  info->s_f = s_f;
  info->margin = margin;
  info->near = margin < ORACLE_NEAR;
  free(w);
  free(r);
  free(z);
  return 0;
}

/* Filter R rows laid out with a fixed row pitch (elements). */
void oracle_filter_rows(const void* rows, int dtype, int R, int V, int64_t row_pitch, double T,
                        int top_k, double top_p, double* probs /* [R, V] or NULL */,
                        oracle_row_info* infos) {
  for (int r = 0; r < R; ++r) {
    const void* row = (dtype == ORACLE_F32)
                          ? (const void*)((const float*)rows + (int64_t)r * row_pitch)
                          : (const void*)((const uint16_t*)rows + (int64_t)r * row_pitch);
    oracle_filter_row(row, dtype, V, T, top_k, top_p, probs ? probs + (int64_t)r * V : NULL,
                      &infos[r]);
  }
}

/* ------------------------------------------------------------------------- */
/* Tree walk: multi-round speculative sampling at every node                  */
/* ([translation] sections 1.3.2 and 1.7; [tutorial] section 2.3 steps 3-5).  */
/* ------------------------------------------------------------------------- */
enum {
  ORACLE_OK = 0,
  ORACLE_ROW_NONFINITE = 1,
  ORACLE_TREE_INVALID = 2,
};

typedef struct {
  const void* p;
  const void* q;
  int dtype, B, N, V;
  int64_t row_pitch, batch_stride;
  const int32_t* draft_tokens;
  const int32_t* parent_idx;
  int max_depth;
  double T, top_p;
  int top_k;
  uint64_t seed, offset;
  int32_t rng_b0;
  const double* u_accept;
  const double* u_final;
  int32_t* out_accept_len;
  int32_t* out_tokens;
  int32_t* out_path;
  double* out_alpha;
  int32_t* out_status;
  int32_t* out_near;
  double* out_final_dist;
} walk_args;

static const void* row_ptr(const walk_args* a, const void* base, int b, int n) {
  int64_t off = (int64_t)b * a->batch_stride + (int64_t)n * a->row_pitch;
  if (a->dtype == ORACLE_F32) return (const void*)((const float*)base + off);
  return (const void*)((const uint16_t*)base + off);
}

static void fail_tree(const walk_args* a, int b, int status) {
  int W = a->max_depth + 1;
  a->out_accept_len[b] = -1;
  for (int j = 0; j < W; ++j) {
    a->out_tokens[(int64_t)b * W + j] = -1;
    a->out_path[(int64_t)b * W + j] = -1;
  }
  if (a->out_status) a->out_status[b] = status;
}

/* Which decision of a tree fell within ORACLE_NEAR of its boundary (bits of
   out_near): a p row's or a q row's top-p cut, an accept test, the final draw. */
#define NEAR_P_CUT 1
#define NEAR_Q_CUT 2
#define NEAR_ACCEPT 4
#define NEAR_DRAW 8

/* Inverse CDF in index order: the smallest i with C_i >= r * C_V. */
static int inverse_cdf(const double* P, int V, double r, int* near) {
  double total = 0.0;
  for (int i = 0; i < V; ++i) total += P[i];
  double target = r * total;
  double cum = 0.0;
  int pick = -1;
  for (int i = 0; i < V; ++i) {
    double prev = cum;
    cum += P[i];
    if (P[i] > 0.0 && cum >= target) {
      pick = i;
      if (fabs(target - prev) < ORACLE_NEAR * total || fabs(target - cum) < ORACLE_NEAR * total)
        *near |= NEAR_DRAW;
      break;
    }
  }
  if (pick < 0) /* r == 1 and rounding: take the last token with mass */
    for (int i = V - 1; i >= 0; --i)
      if (P[i] > 0.0) { pick = i; *near |= NEAR_DRAW; break; }
  return pick;
}

static void walk_one_tree(const walk_args* a, int b) {
  const int N = a->N, V = a->V, W = a->max_depth + 1;
  const int32_t* par = a->parent_idx + (int64_t)b * N;
  const int32_t* tok = a->draft_tokens + (int64_t)b * N;
  if (a->out_status) a->out_status[b] = ORACLE_OK;
  if (a->out_near) a->out_near[b] = 0;
  if (a->out_alpha)
    for (int n = 0; n < N; ++n) a->out_alpha[(int64_t)b * N + n] = NAN;

  /* Tree checks: node 0 is the root, every other node's parent precedes it,
     every draft token is a vocabulary index, and no node is deeper than max_depth. */
  if (N < 1 || par[0] != -1) { fail_tree(a, b, ORACLE_TREE_INVALID); return; }
  int* depth = (int*)malloc(sizeof(int) * (size_t)N);
  depth[0] = 0;
  for (int n = 1; n < N; ++n) {
    if (par[n] < 0 || par[n] >= n || tok[n] < 0 || tok[n] >= V) {
      free(depth);
      fail_tree(a, b, ORACLE_TREE_INVALID);
      return;
    }
    depth[n] = depth[par[n]] + 1;
    if (depth[n] > a->max_depth) {
      free(depth);
      fail_tree(a, b, ORACLE_TREE_INVALID);
      return;
    }
  }
  free(depth);

  double* P = (double*)malloc(sizeof(double) * (size_t)V);
  double* Q = (double*)malloc(sizeof(double) * (size_t)V);
  int near = 0;
  int u = 0, n_acc = 0;
  int32_t path[W];
  int32_t toks[W];
  path[0] = 0;
  int final_tok = -1;

  for (;;) {
    oracle_row_info pi, qi;
    if (oracle_filter_row(row_ptr(a, a->p, b, u), a->dtype, V, a->T, a->top_k, a->top_p, P, &pi)) {
      free(P); free(Q);
      fail_tree(a, b, ORACLE_ROW_NONFINITE);
      return;
    }
    if (pi.near) near |= NEAR_P_CUT;
    int has_child = 0;
    for (int c = u + 1; c < N; ++c)
      if (par[c] == u) { has_child = 1; break; }

    if (a->T == 0.0) {
      /* Greedy ([reading] sections 3 and 5): accept the first child whose token is
         the target argmax; otherwise emit the argmax. */
      int next = -1;
      for (int c = u + 1; c < N && next < 0; ++c) {
        if (par[c] != u) continue;
        int ok = (tok[c] == pi.argmax);
        if (a->out_alpha) a->out_alpha[(int64_t)b * N + c] = ok ? 1.0 : 0.0;
        if (ok) next = c;
      }
      if (next >= 0) {
        toks[n_acc] = tok[next];
        path[++n_acc] = next;
        u = next;
        continue;
      }
      final_tok = pi.argmax;
      if (a->out_final_dist) {
        double* fd = a->out_final_dist + (int64_t)b * V;
        for (int i = 0; i < V; ++i) fd[i] = P[i];
      }
      break;
    }

    if (has_child) {
      if (oracle_filter_row(row_ptr(a, a->q, b, u), a->dtype, V, a->T, a->top_k, a->top_p, Q, &qi)) {
        free(P); free(Q);
        fail_tree(a, b, ORACLE_ROW_NONFINITE);
        return;
      }
      if (qi.near) near |= NEAR_Q_CUT;
    }

    int next = -1;
    for (int c = u + 1; c < N && next < 0; ++c) {
      if (par[c] != u) continue;
      int x = tok[c];
      /* Accept probability min(1, p(x)/q(x)) ([tutorial] section 2.3 step 3);
         q(x) == 0 accepts exactly when p(x) > 0. */
      double alpha;
      if (Q[x] > 0.0)
        alpha = fmin(1.0, P[x] / Q[x]);
      else
        alpha = (P[x] > 0.0) ? 1.0 : 0.0;
      double r = a->u_accept ? a->u_accept[(int64_t)b * N + c]
                             : oracle_uniform(a->seed, a->offset, a->rng_b0 + b, c, 0);
      if (a->out_alpha) a->out_alpha[(int64_t)b * N + c] = alpha;
      if (fabs(r - alpha) < ORACLE_NEAR) near |= NEAR_ACCEPT;
      if (r <= alpha) {
        next = c;
      } else {
        /* Rejected: p <- norm(max(0, p - q)) ([tutorial] section 2.3 step 4),
           then the next sibling is tried against the adjusted p
           ([translation] section 1.7). */
        double z = 0.0;
        for (int i = 0; i < V; ++i) z += fmax(0.0, P[i] - Q[i]);
        if (z > 0.0)
          for (int i = 0; i < V; ++i) P[i] = fmax(0.0, P[i] - Q[i]) / z;
      }
    }
    if (next >= 0) {
      toks[n_acc] = tok[next];
      path[++n_acc] = next;
      u = next;
      continue;
    }
    /* No child accepted (or u is a leaf): draw the correction / bonus token from
       the current p ([tutorial] section 2.3 step 4, both cases). */
    double r = a->u_final ? a->u_final[(int64_t)b * N + u]
                          : oracle_uniform(a->seed, a->offset, a->rng_b0 + b, u, 1);
    final_tok = inverse_cdf(P, V, r, &near);
    if (a->out_final_dist) {
      double* fd = a->out_final_dist + (int64_t)b * V;
      for (int i = 0; i < V; ++i) fd[i] = P[i];
    }
    break;
  }
  free(P);
  free(Q);

  /* Outputs: accepted tokens then the final token ([tutorial] section 2.3 step 5:
     n accepted + 1), padded with -1; the path starts at the root. */
  a->out_accept_len[b] = n_acc;
  for (int j = 0; j < W; ++j) {
    a->out_tokens[(int64_t)b * W + j] = -1;
    a->out_path[(int64_t)b * W + j] = -1;
  }
  for (int j = 0; j < n_acc; ++j) a->out_tokens[(int64_t)b * W + j] = toks[j];
  a->out_tokens[(int64_t)b * W + n_acc] = final_tok;
  for (int j = 0; j <= n_acc; ++j) a->out_path[(int64_t)b * W + j] = path[j];
  if (a->out_near) a->out_near[b] = near;
}

typedef struct {
  const walk_args* a;
  int b0, b1;
} walk_slice;

static void* walk_slice_main(void* arg) {
  walk_slice* s = (walk_slice*)arg;
  for (int b = s->b0; b < s->b1; ++b) walk_one_tree(s->a, b);
  return NULL;
}

/*
 * Verify B draft trees.  Logit element (b, n, v) sits at
 * b * batch_stride + n * row_pitch + v.  Tree b draws its uniforms as batch
 * index rng_b0 + b (so a slice of a larger batch reproduces the same draws).
 * u_accept / u_final, when non-NULL,
 * replace the Philox uniforms ([B, N] each, indexed by the tested child /
 * the node of the final draw).  out_alpha [B, N] (NaN where untested),
 * out_near [B] (the NEAR_* bits of the decisions that fell within ORACLE_NEAR of
 * their boundary, 0 if none), out_final_dist [B, V] are optional.  Returns 0.
 */
int oracle_verify_tree(const void* logits_p, const void* logits_q, int dtype, int B, int N, int V,
                       int64_t row_pitch, int64_t batch_stride, const int32_t* draft_tokens,
                       const int32_t* parent_idx, int max_depth, double temperature, int top_k,
                       double top_p, uint64_t seed, uint64_t offset, int32_t rng_b0,
                       const double* u_accept,
                       const double* u_final, int32_t* out_accept_len, int32_t* out_tokens,
                       int32_t* out_path, double* out_alpha, int32_t* out_status, int32_t* out_near,
                       double* out_final_dist, int nthreads) {
  walk_args a = {logits_p, logits_q, dtype, B, N, V, row_pitch, batch_stride, draft_tokens,
                 parent_idx, max_depth, temperature, top_p, top_k, seed, offset, rng_b0, u_accept,
                 u_final, out_accept_len, out_tokens, out_path, out_alpha, out_status, out_near,
                 out_final_dist};
  if (nthreads <= 1 || B <= 1) {
    for (int b = 0; b < B; ++b) walk_one_tree(&a, b);
    return 0;
  }
  if (nthreads > B) nthreads = B;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  walk_slice* sl = (walk_slice*)malloc(sizeof(walk_slice) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t) {
    sl[t].a = &a;
    sl[t].b0 = (int)((int64_t)B * t / nthreads);
    sl[t].b1 = (int)((int64_t)B * (t + 1) / nthreads);
    pthread_create(&th[t], NULL, walk_slice_main, &sl[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(sl);
  return 0;
}
