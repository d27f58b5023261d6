/*
 * CPU oracle of the tree verify forward pass -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check and the benchmark's CPU-baseline leg load this
 * file's library.  The product path never does: it shares no code with this
 * file and must fail loudly when its CUDA library is missing.
 *
 * What it computes (the definition, written out plainly):
 *
 *   Every node of a draft tree is scored by one "row".  Row i processes the
 *   node's own token at position ctx + depth(i) and attends to the cached
 *   context plus the root-to-i path (i included); its output distribution
 *   scores the children of i.  This is the query convention of
 *   [Algorithm and correctness contract, §Target position and batching]: the
 *   query that scores node x holds the prompt and x's ancestors, excluding x,
 *   and siblings share it.  Tree attention is "an ancestor mask and a position
 *   equal to its depth" [Drafters and tree verify, §Tree verify through
 *   recurrent layers].  Greedy verify must reproduce plain one-token-at-a-time
 *   decoding [Exactness, §The promise]; orc_decode_sequence below is that
 *   plain decoder, and each tree row must equal it on the row's own path.
 *
 *   The layer (the pages do not give one; this is the plainest reading):
 *     x   = E[token]
 *     h   = bf16( x / sqrt(mean(x^2) + eps) * g1 )
 *     q,k,v = h W_qkv^T ; q,k rotated by RoPE (rotate-half, base theta) at pos
 *     q,k,v -> bf16 (k and v are what the cache stores)
 *     o   = bf16( softmax(q k^T / sqrt(D)) v )   per query head, GQA
 *     r   = bf16( x + o W_o^T )
 *     hf  = bf16( r / sqrt(mean(r^2) + eps) * g_f )
 *     logits = fp32( hf W_lm^T )   -- "The head returns fp32 logits" [Exactness,
 *                                     §The one exception: near ties]
 *
 * Arithmetic: every sum, product, exp and sqrt in fp64, each dot product summed
 * in increasing index order.  bf16 rounding happens only at the storage points
 * listed above, round-to-nearest-even through fp32.  No blocking, fusion or
 * reordering: loops over independent outputs run in parallel (OpenMP) but no
 * single sum changes order.  Compile with -ffp-contract=off so that no a*b+c is
 * fused and the results are the same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int32_t hidden, n_q_heads, n_kv_heads, head_dim, vocab;
  double rope_theta, rms_eps;
  const uint16_t *embed;   /* [V][H]            */
  const uint16_t *ln1;     /* [H]               */
  const uint16_t *wqkv;    /* [(Hq+2Hkv)D][H]   */
  const uint16_t *wo;      /* [H][Hq D]         */
  const uint16_t *ln_f;    /* [H]               */
  const uint16_t *lm_head; /* [V][H]            */
} orc_model;

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the following calls (timing only: every sum keeps its order, so
 * the results do not depend on it). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ---- bf16 <-> fp64 ---------------------------------------------------- */

static double bf(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round to bf16: first to fp32 (the C conversion, round-to-nearest-even), then
 * to the 8-bit significand of bf16, ties to even. */
uint16_t orc_round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) {          /* inf or nan */
    if (u & 0x007fffffu) return (uint16_t)((u >> 16) | 0x0040u);
    return (uint16_t)(u >> 16);
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static double rb(double x) { return bf(orc_round_bf16(x)); }

/* ---- building blocks ---------------------------------------------------- */

/* y = bf16( x / sqrt(mean(x^2) + eps) * g ) */
static void rmsnorm_bf16(const double *x, const uint16_t *g, int H, double eps, double *y) {
  double ss = 0.0;
  for (int k = 0; k < H; ++k) ss += x[k] * x[k];
  double inv = 1.0 / sqrt(ss / (double)H + eps);
  for (int k = 0; k < H; ++k) y[k] = rb(x[k] * inv * bf(g[k]));
}

/* out[o] = sum_k W[o][k] * in[k], k ascending */
static double dot_w(const uint16_t *wrow, const double *in, int K) {
  double acc = 0.0;
  for (int k = 0; k < K; ++k) acc += bf(wrow[k]) * in[k];
  return acc;
}

/* Rotate-half RoPE at integer position pos: pairs (d, d + D/2), angle
 * pos * theta^(-2d/D). */
static void rope(double *x, int D, long pos, double theta) {
  int half = D / 2;
  for (int d = 0; d < half; ++d) {
    double inv_freq = pow(theta, -2.0 * (double)d / (double)D);
    double a = (double)pos * inv_freq;
    double c = cos(a), s = sin(a);
    double x1 = x[d], x2 = x[d + half];
    x[d] = x1 * c - x2 * s;
    x[d + half] = x2 * c + x1 * s;
  }
}

/* Front half of one token: embedding, norm, projections, RoPE.  Writes
 * x (fp64 copy of the embedding row), q [Hq*D], k [Hkv*D], v [Hkv*D] as bf16. */
static void token_front(const orc_model *m, int token, long pos, double *x,
                        uint16_t *q, uint16_t *k, uint16_t *v) {
  const int H = m->hidden, D = m->head_dim, Hq = m->n_q_heads, Hkv = m->n_kv_heads;
  double *h = (double *)malloc(sizeof(double) * H);
  double *t = (double *)malloc(sizeof(double) * D);
  for (int c = 0; c < H; ++c) x[c] = bf(m->embed[(size_t)token * H + c]);
  rmsnorm_bf16(x, m->ln1, H, m->rms_eps, h);
  for (int head = 0; head < Hq + 2 * Hkv; ++head) {
    for (int d = 0; d < D; ++d)
      t[d] = dot_w(m->wqkv + ((size_t)head * D + d) * H, h, H);
    if (head < Hq + Hkv) rope(t, D, pos, m->rope_theta);   /* q and k heads */
    uint16_t *dst = head < Hq ? q + (size_t)head * D
                  : head < Hq + Hkv ? k + (size_t)(head - Hq) * D
                  : v + (size_t)(head - Hq - Hkv) * D;
    for (int d = 0; d < D; ++d) dst[d] = orc_round_bf16(t[d]);
  }
  free(t);
  free(h);
}

/* Attention of one query row over an explicit list of keys.
 * kp[j*Hkv + g], vp[j*Hkv + g] point at key/value j of KV head g ([D] bf16).
 * o [Hq*D] bf16 = softmax(q.k / sqrt(D)) v per query head; query head hq reads
 * KV head hq / (Hq / Hkv). */
static void attend(const orc_model *m, const uint16_t *q, int n_keys,
                   const uint16_t *const *kp, const uint16_t *const *vp, uint16_t *o) {
  const int D = m->head_dim, Hq = m->n_q_heads, Hkv = m->n_kv_heads;
  const int group = Hq / Hkv;
  const double scale = 1.0 / sqrt((double)D);
  double *s = (double *)malloc(sizeof(double) * (size_t)n_keys);
  double *acc = (double *)malloc(sizeof(double) * D);
  for (int hq = 0; hq < Hq; ++hq) {
    const int g = hq / group;
    const uint16_t *qh = q + (size_t)hq * D;
    double mx = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
      const uint16_t *kj = kp[(size_t)j * Hkv + g];
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += bf(qh[d]) * bf(kj[d]);
      s[j] = dot * scale;
      if (s[j] > mx) mx = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < n_keys; ++j) {
      s[j] = exp(s[j] - mx);
      z += s[j];
    }
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j < n_keys; ++j) {
      const uint16_t *vj = vp[(size_t)j * Hkv + g];
      double p = s[j] / z;
      for (int d = 0; d < D; ++d) acc[d] += p * bf(vj[d]);
    }
    for (int d = 0; d < D; ++d) o[(size_t)hq * D + d] = orc_round_bf16(acc[d]);
  }
  free(acc);
  free(s);
}

/* Back half of one row: O projection, residual, final norm.  hf [H] as fp64
 * (holding bf16 values). */
static void token_back(const orc_model *m, const double *x, const uint16_t *o, double *hf) {
  const int H = m->hidden, QD = m->n_q_heads * m->head_dim;
  double *od = (double *)malloc(sizeof(double) * QD);
  double *r = (double *)malloc(sizeof(double) * H);
  for (int c = 0; c < QD; ++c) od[c] = bf(o[c]);
  for (int c = 0; c < H; ++c) r[c] = rb(x[c] + dot_w(m->wo + (size_t)c * QD, od, QD));
  rmsnorm_bf16(r, m->ln_f, H, m->rms_eps, hf);
  free(r);
  free(od);
}

/* logits[i][v] = fp32( sum_k hf_i[k] * W_lm[v][k] ) for n rows. */
static void head_logits(const orc_model *m, const double *hf, int n, float *logits) {
  const int H = m->hidden, V = m->vocab;
#pragma omp parallel for schedule(static)
  for (int v = 0; v < V; ++v)
    for (int i = 0; i < n; ++i)
      logits[(size_t)i * V + v] = (float)dot_w(m->lm_head + (size_t)v * H, hf + (size_t)i * H, H);
}

/* ---- the tree verify ---------------------------------------------------- */

/*
 * One request's verify.  cache_k/cache_v: [Hkv][capacity][D] bf16, slots
 * [0, ctx) valid.  parent[0] = -1 and parent[i] < i (the caller validated).
 * Outputs (any may be NULL):
 *   logits [n][V] fp32, q_out [n][Hq*D], k_out/v_out [n][Hkv*D] (the tree rows'
 *   K/V, i.e. what verify writes to cache slot ctx+i), attn_out [n][Hq*D],
 *   hf_out [n][H] (bf16 bits).
 * Returns 0, or -1 on allocation failure.
 */
int orc_verify_tree(const orc_model *m, const uint16_t *cache_k, const uint16_t *cache_v,
                    int ctx, int capacity, const int32_t *parent, const int32_t *token, int n,
                    float *logits, uint16_t *q_out, uint16_t *k_out, uint16_t *v_out,
                    uint16_t *attn_out, uint16_t *hf_out) {
  const int H = m->hidden, D = m->head_dim, Hq = m->n_q_heads, Hkv = m->n_kv_heads;
  const int QD = Hq * D, KD = Hkv * D;
  int *depth = (int *)malloc(sizeof(int) * n);
  double *x = (double *)malloc(sizeof(double) * (size_t)n * H);
  uint16_t *q = (uint16_t *)malloc(2 * (size_t)n * QD);
  uint16_t *k = (uint16_t *)malloc(2 * (size_t)n * KD);
  uint16_t *v = (uint16_t *)malloc(2 * (size_t)n * KD);
  uint16_t *o = (uint16_t *)malloc(2 * (size_t)n * QD);
  double *hf = (double *)malloc(sizeof(double) * (size_t)n * H);
  if (!depth || !x || !q || !k || !v || !o || !hf) return -1;

  /* position of node i = ctx + depth(i); the root has depth 0 */
  for (int i = 0; i < n; ++i) depth[i] = i == 0 ? 0 : depth[parent[i]] + 1;

#pragma omp parallel for schedule(dynamic)
  for (int i = 0; i < n; ++i)
    token_front(m, token[i], (long)ctx + depth[i], x + (size_t)i * H,
                q + (size_t)i * QD, k + (size_t)i * KD, v + (size_t)i * KD);

#pragma omp parallel for schedule(dynamic)
  for (int i = 0; i < n; ++i) {
    /* keys of row i: cache slots 0..ctx-1, then the root-to-i path in increasing
     * node index (= increasing depth, since a parent precedes its child) */
    int path[64], len = 0;
    for (int a = i; a >= 0; a = parent[a]) path[len++] = a;
    int n_keys = ctx + len;
    const uint16_t **kp = (const uint16_t **)malloc(sizeof(void *) * (size_t)n_keys * Hkv);
    const uint16_t **vp = (const uint16_t **)malloc(sizeof(void *) * (size_t)n_keys * Hkv);
    for (int g = 0; g < Hkv; ++g) {
      for (int j = 0; j < ctx; ++j) {
        kp[(size_t)j * Hkv + g] = cache_k + ((size_t)g * capacity + j) * D;
        vp[(size_t)j * Hkv + g] = cache_v + ((size_t)g * capacity + j) * D;
      }
      for (int t = 0; t < len; ++t) {
        int a = path[len - 1 - t];
        kp[(size_t)(ctx + t) * Hkv + g] = k + (size_t)a * KD + (size_t)g * D;
        vp[(size_t)(ctx + t) * Hkv + g] = v + (size_t)a * KD + (size_t)g * D;
      }
    }
    attend(m, q + (size_t)i * QD, n_keys, kp, vp, o + (size_t)i * QD);
    free(kp);
    free(vp);
    token_back(m, x + (size_t)i * H, o + (size_t)i * QD, hf + (size_t)i * H);
  }

  if (logits) head_logits(m, hf, n, logits);
  if (q_out) memcpy(q_out, q, 2 * (size_t)n * QD);
  if (k_out) memcpy(k_out, k, 2 * (size_t)n * KD);
  if (v_out) memcpy(v_out, v, 2 * (size_t)n * KD);
  if (attn_out) memcpy(attn_out, o, 2 * (size_t)n * QD);
  if (hf_out)
    for (size_t c = 0; c < (size_t)n * H; ++c) hf_out[c] = orc_round_bf16(hf[c]);
  free(depth); free(x); free(q); free(k); free(v); free(o); free(hf);
  return 0;
}

/*
 * Plain greedy-style decoding of a fixed token sequence, one token at a time:
 * token t sits at position ctx + t and attends to the cache and to tokens
 * 0..t, whose K/V were appended as they were decoded.  This is the reference
 * the tree verify must equal row by row [Exactness, §The promise].
 * Outputs as orc_verify_tree, one row per token.
 */
int orc_decode_sequence(const orc_model *m, const uint16_t *cache_k, const uint16_t *cache_v,
                        int ctx, int capacity, const int32_t *tokens, int len,
                        float *logits, uint16_t *k_out, uint16_t *v_out, uint16_t *attn_out,
                        uint16_t *hf_out) {
  const int H = m->hidden, D = m->head_dim, Hq = m->n_q_heads, Hkv = m->n_kv_heads;
  const int QD = Hq * D, KD = Hkv * D;
  /* the growing cache: ctx cached rows followed by the decoded rows */
  uint16_t *kc = (uint16_t *)malloc(2 * (size_t)(ctx + len) * KD);
  uint16_t *vc = (uint16_t *)malloc(2 * (size_t)(ctx + len) * KD);
  const uint16_t **kp = (const uint16_t **)malloc(sizeof(void *) * (size_t)(ctx + len) * Hkv);
  const uint16_t **vp = (const uint16_t **)malloc(sizeof(void *) * (size_t)(ctx + len) * Hkv);
  double *x = (double *)malloc(sizeof(double) * H);
  double *hf = (double *)malloc(sizeof(double) * (size_t)len * H);
  uint16_t *q = (uint16_t *)malloc(2 * (size_t)QD);
  uint16_t *o = (uint16_t *)malloc(2 * (size_t)QD);
  if (!kc || !vc || !kp || !vp || !x || !hf || !q || !o) return -1;
  for (int j = 0; j < ctx; ++j)
    for (int g = 0; g < Hkv; ++g) {
      memcpy(kc + (size_t)j * KD + (size_t)g * D, cache_k + ((size_t)g * capacity + j) * D, 2 * (size_t)D);
      memcpy(vc + (size_t)j * KD + (size_t)g * D, cache_v + ((size_t)g * capacity + j) * D, 2 * (size_t)D);
    }
  for (int t = 0; t < len; ++t) {
    const int slot = ctx + t;
    token_front(m, tokens[t], (long)slot, x, q, kc + (size_t)slot * KD, vc + (size_t)slot * KD);
    for (int j = 0; j <= slot; ++j)
      for (int g = 0; g < Hkv; ++g) {
        kp[(size_t)j * Hkv + g] = kc + (size_t)j * KD + (size_t)g * D;
        vp[(size_t)j * Hkv + g] = vc + (size_t)j * KD + (size_t)g * D;
      }
    attend(m, q, slot + 1, kp, vp, o);
    token_back(m, x, o, hf + (size_t)t * H);
    if (k_out) memcpy(k_out + (size_t)t * KD, kc + (size_t)slot * KD, 2 * (size_t)KD);
    if (v_out) memcpy(v_out + (size_t)t * KD, vc + (size_t)slot * KD, 2 * (size_t)KD);
    if (attn_out) memcpy(attn_out + (size_t)t * QD, o, 2 * (size_t)QD);
  }
  if (logits) head_logits(m, hf, len, logits);
  if (hf_out)
    for (size_t c = 0; c < (size_t)len * H; ++c) hf_out[c] = orc_round_bf16(hf[c]);
  free(kc); free(vc); free(kp); free(vp); free(x); free(hf); free(q); free(o);
  return 0;
}

/* Logits of n rows of hf (bf16 bits [n][H]) for a list of vocab ids only:
 * out[i][t] = fp32( sum_k hf_i[k] W_lm[vid[t]][k] ).  Used to spot-check the
 * full-vocabulary head one output at a time. */
int orc_head_rows(const orc_model *m, const uint16_t *hf_bits, int n, const int32_t *vid, int n_vid,
                  float *out) {
  const int H = m->hidden;
  double *hf = (double *)malloc(sizeof(double) * (size_t)n * H);
  if (!hf) return -1;
  for (size_t c = 0; c < (size_t)n * H; ++c) hf[c] = bf(hf_bits[c]);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < n_vid; ++t)
    for (int i = 0; i < n; ++i)
      out[(size_t)i * n_vid + t] = (float)dot_w(m->lm_head + (size_t)vid[t] * H, hf + (size_t)i * H, H);
  free(hf);
  return 0;
}

/* y[i][o] = sum_k W[o][k] * x[i][k] (k ascending, fp64) for n input rows; W is
 * [M][K] bf16 bits.  The plain projection the layer-stack oracle builds on:
 * every output is one sequential dot product, so the result does not depend
 * on n, on the thread count or on which other rows are projected with it. */
int orc_matvec_rows(const uint16_t *W, int M, int K, const double *x, int n, double *y) {
#pragma omp parallel for schedule(static)
  for (int o = 0; o < M; ++o)
    for (int i = 0; i < n; ++i)
      y[(size_t)i * M + o] = dot_w(W + (size_t)o * K, x + (size_t)i * K, K);
  return 0;
}
