/*
 * hwref.c - float64 CPU oracle for concurrent decode attention over a shared,
 * block-structured KV cache (Hogwild! Inference), and for the block commit.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (page title, then section / equation):
 *  [N] "Hogwild! Inference: Parallel LLM Generation via Concurrent Attention"
 *      (paper-notes page, NeurIPS 2025):
 *        - "Key design 1: shared KV cache and concurrent attention" and its
 *          query-rotation equation rho(q,i_q)[rho(A,i_k^A) (+) ...] =
 *          rho(q,i_q-i_k^A)A (+) ...;
 *        - "Key design 2: cache structure" (combined layout, step commit:
 *          a finished step's KV is rotated and moved into the shared history);
 *        - implementation notes under "training strategy": each block stores its
 *          KV at block-local positions, the real position is applied by
 *          rotating the query.
 *  [A] omica.com.cn article on Hogwild! Inference:
 *        - section 2.1 (rotate_query: frequencies 1/base^(2i/dim), angle =
 *          offset * freq, q*cos + rotate_half(q)*sin);
 *        - section 3.2 (blockwise attention: per block, rotate q by the block
 *          offset, score = q_rot . k / sqrt(dim); one softmax across all blocks;
 *          weighted sum of V).
 *
 * Readings where the pages are silent or garbled (each also listed in the
 * design notes):
 *  - block-local positions are 0..len-1;
 *  - RoPE pairs element i with element i + D/2 (rotate_half), frequencies
 *    w_i = theta^(-2i/D), theta passed by the caller;
 *  - i_k^block in the equation is the block's start position in the viewing
 *    worker's own view; the query is rotated by i_q - i_k^block;
 *  - one max-subtracted softmax over the concatenation of all view blocks;
 *    an empty view gives out = 0 and lse = -inf;
 *  - GQA: q head h reads kv head h / (Hq/Hkv) unless a map is given;
 *  - FP8 caches (the omica.com.cn article, section 6, only names FP8
 *    attention as future work; storage as E4M3 with per-head scales): K and V
 *    hold E4M3 codes, a cached element is its decoded value times its kv
 *    head's scale, queries stay bf16.
 *
 * Everything is computed in double, elementwise, with no blocking, fusion or
 * reordering beyond what the definitions state.  Work is spread over POSIX
 * threads by (row, q head) item; each item is computed independently.
 *
 * Planted mistakes: building with -DHWREF_MUTANT=<n> introduces one plausible
 * mistake (see the MUTANT(...) sites) so that the tests can show that the pins
 * catch it.  The default build has none.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef HWREF_MUTANT
#define HWREF_MUTANT 0
#endif
#define MUTANT(n) (HWREF_MUTANT == (n))

enum { HWREF_F32 = 0, HWREF_BF16 = 1, HWREF_FP8 = 2 };
enum { HWREF_OK = 0, HWREF_EINVAL = -1, HWREF_ENOMEM = -2 };

/* ------------------------------------------------------------------------ */
/* element access                                                            */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the float whose upper 16 bits are the stored bits. */
static double e4m3_to_double(uint8_t b);

static double load_elem(const void *base, int dtype, int64_t idx) {
  if (dtype == HWREF_F32) return (double)((const float *)base)[idx];
  if (dtype == HWREF_FP8) return e4m3_to_double(((const uint8_t *)base)[idx]);
  uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16, ties to even, directly from the double
 * (no intermediate float rounding).  Returns the 16 stored bits. */
static uint16_t bf16_from_double(double x) {
  if (isnan(x)) return 0x7fc0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  double q;                /* a rounded to the bf16 grid */
  if (e - 1 < -126) {
    /* subnormal range: grid step 2^-133 */
    q = ldexp(nearbyint(ldexp(a, 133)), -133);
  } else {
    /* 8 significant bits: m * 2^8 in [128, 256) */
    q = ldexp(nearbyint(ldexp(m, 8)), e - 8);
  }
  if (q > 0x1.fep127) return sign | 0x7f80; /* beyond the largest finite bf16 */
  float f = (float)q; /* exact: q has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | ((u >> 16) & 0x7fff));
}

/* FP8 E4M3 (the "fn" variant of the OCP 8-bit floating point formats): sign,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal
 * (m * 2^-9), S.1111.111 is NaN, there is no infinity, the largest finite
 * value is S.1111.110 = 448. */
static double e4m3_to_double(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  double v;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(8.0 + m, e - (MUTANT(10) ? 11 : 10)); /* (1 + m/8) * 2^(e - 7) */
  return sign ? -v : v;
}

/* Round a double to E4M3, ties to even, directly from the double; magnitudes
 * beyond 448 saturate to 448 (no infinity to round to). */
static uint8_t e4m3_from_double(double x) {
  if (isnan(x)) return 0x7f;
  const uint8_t sign = signbit(x) ? 0x80 : 0;
  const double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int k = e - 1;
  if (k < -6) k = -6; /* below 2^-6 the subnormal grid keeps the step 2^-9 */
  double q = nearbyint(ldexp(a, 3 - k)); /* a on the grid of step 2^(k-3), in steps */
  q = ldexp(q, k - 3);
  if (q > 448.0) q = 448.0;
  if (q == 0.0) return sign;
  if (q < 0x1p-6) return sign | (uint8_t)ldexp(q, 9); /* subnormal: m * 2^-9 */
  frexp(q, &e); /* q may have rounded up into the next binade */
  k = e - 1;
  const int m = (int)ldexp(q, 3 - k) - 8;
  return sign | (uint8_t)(((k + 7) << 3) | m);
}

static void store_elem(void *base, int dtype, int64_t idx, double v) {
  if (dtype == HWREF_F32)
    ((float *)base)[idx] = (float)v; /* round to nearest even */
  else if (dtype == HWREF_FP8)
    ((uint8_t *)base)[idx] = e4m3_from_double(v);
  else
    ((uint16_t *)base)[idx] = bf16_from_double(v);
}

static void copy_elem(void *dst, const void *src, int dtype, int64_t di, int64_t si) {
  if (dtype == HWREF_F32)
    memcpy((float *)dst + di, (const float *)src + si, 4);
  else if (dtype == HWREF_FP8)
    memcpy((uint8_t *)dst + di, (const uint8_t *)src + si, 1);
  else
    memcpy((uint16_t *)dst + di, (const uint16_t *)src + si, 2);
}

/* ------------------------------------------------------------------------ */
/* RoPE                                                                      */
/* ------------------------------------------------------------------------ */

/* Frequencies w_i = theta^(-2i/D), i in [0, D/2). */
void hwref_rope_freqs(int D, double theta, double *w) {
  for (int i = 0; i < D / 2; ++i) {
    w[i] = pow(theta, -2.0 * i / D);
    if (MUTANT(2)) w[i] = pow(theta, -1.0 * i / D); /* wrong exponent */
  }
}

/* y = rho(x, pos):  y_i       = x_i cos(a_i) - x_{i+D/2} sin(a_i)
 *                   y_{i+D/2} = x_{i+D/2} cos(a_i) + x_i sin(a_i)
 * with a_i = pos * w_i.  x and y may alias. */
static void rope_with(const double *x, int D, const double *w, double pos, double *y) {
  int half = D / 2;
  if (MUTANT(3)) { /* adjacent (interleaved) pairing instead of halves */
    for (int i = 0; i < half; ++i) {
      double a = pos * w[i];
      double c = cos(a), s = sin(a);
      double lo = x[2 * i], hi = x[2 * i + 1];
      y[2 * i] = lo * c - hi * s;
      y[2 * i + 1] = hi * c + lo * s;
    }
    return;
  }
  for (int i = 0; i < half; ++i) {
    double a = pos * w[i];
    double c = cos(a), s = sin(a);
    double lo = x[i], hi = x[i + half];
    if (MUTANT(1)) s = -s; /* rotation in the wrong direction */
    y[i] = lo * c - hi * s;
    y[i + half] = hi * c + lo * s;
  }
}

/* Public single-vector RoPE in double. */
void hwref_rope(const double *x, int D, double theta, double pos, double *y) {
  double w[512];
  hwref_rope_freqs(D, theta, w);
  rope_with(x, D, w, pos, y);
}

/* ------------------------------------------------------------------------ */
/* decode attention                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t n_rows;          /* query tokens (one per worker per problem) */
  int32_t n_q_heads;       /* Hq */
  int32_t n_kv_heads;      /* Hkv */
  int32_t head_dim;        /* D */
  int32_t n_blocks;        /* blocks in the cache pool */
  int32_t max_view_blocks; /* width of the per-row view tables */
  int64_t cache_capacity;  /* tokens per head in the pool */
  int32_t dtype;           /* HWREF_F32, HWREF_BF16, or HWREF_FP8 (bf16 q, E4M3 K and V) */
  double rope_theta;
  double scale;
} hwref_desc;

typedef struct {
  const hwref_desc *d;
  const void *q, *k, *v;
  const int32_t *block_start, *block_len, *view_block, *view_offset, *q_pos, *q_to_kv;
  const int32_t *view_limit; /* [rows][V] or NULL: tokens of the entry's block the row sees */
  const float *k_scale, *v_scale; /* HWREF_FP8: [Hkv], a stored value times its head's scale */
  const int32_t *rows; /* rows to compute, n_items = n_sel * Hq */
  int32_t n_sel;
  int brute; /* 0: block form (the method), 1: brute-force re-encoding */
  double *out, *lse;
  int64_t next;
  pthread_mutex_t mu;
  int status;
} decode_job;

static int kv_head_of(const hwref_desc *d, const int32_t *q_to_kv, int h) {
  if (q_to_kv) return q_to_kv[h];
  int group = d->n_q_heads / d->n_kv_heads;
  if (MUTANT(6)) return h % d->n_kv_heads; /* strided instead of grouped */
  return h / group;
}

/* Tokens of view entry (row, v) the row attends: the block's first
 * min(limit, len) when the entry has a limit >= 0, else all len. */
static int entry_len(const decode_job *J, int32_t row, int v, int len) {
  if (!J->view_limit) return len;
  const int32_t lim = J->view_limit[(int64_t)row * J->d->max_view_blocks + v];
  if (MUTANT(9) && lim > 0 && lim < len) return lim - 1; /* the limit's own token left out */
  return lim >= 0 && lim < len ? lim : len;
}

/* One (row, q-head) item.  Returns 0 or an error code. */
static int decode_item(decode_job *J, int32_t row, int32_t h, double *scratch_q, double *scratch_t,
                       double *w) {
  const hwref_desc *d = J->d;
  const int D = d->head_dim, V = d->max_view_blocks;
  const int g = kv_head_of(d, J->q_to_kv, h);
  if (g < 0 || g >= d->n_kv_heads) return HWREF_EINVAL;
  const int64_t qbase = ((int64_t)row * d->n_q_heads + h) * D;
  const int qdt = d->dtype == HWREF_FP8 ? HWREF_BF16 : d->dtype;
  for (int i = 0; i < D; ++i) scratch_q[i] = load_elem(J->q, qdt, qbase + i);
  /* a cached K or V element is its stored value times the head's scale (E4M3) */
  const double ks = d->dtype == HWREF_FP8 ? (double)J->k_scale[MUTANT(11) ? g ^ 1 : g] : 1.0;
  const double vs = d->dtype == HWREF_FP8 ? (double)J->v_scale[g] : 1.0;
  const int64_t head_base = (int64_t)g * d->cache_capacity * D;
  const int32_t iq = J->q_pos[row];

  /* pass 1: all scores of the view, in view order */
  int64_t n_tok = 0;
  for (int v = 0; v < V; ++v) {
    int b = J->view_block[(int64_t)row * V + v];
    if (b < 0) continue;
    if (b >= d->n_blocks) return HWREF_EINVAL;
    int len = J->block_len[b];
    if (len < 0) return HWREF_EINVAL;
    if ((int64_t)J->block_start[b] + len > d->cache_capacity || J->block_start[b] < 0)
      return HWREF_EINVAL;
    n_tok += entry_len(J, row, v, len);
  }
  double *s = (double *)malloc(sizeof(double) * (size_t)(n_tok > 0 ? n_tok : 1));
  if (!s) return HWREF_ENOMEM;
  double qt[1024], kk[1024], ka[1024];
  int64_t t = 0;
  if (J->brute) rope_with(scratch_q, D, w, (double)iq, qt); /* rho(q, i_q) */
  for (int v = 0; v < V; ++v) {
    int b = J->view_block[(int64_t)row * V + v];
    if (b < 0) continue;
    int len = entry_len(J, row, v, J->block_len[b]);
    if (len == 0) continue;
    int32_t off = J->view_offset[(int64_t)row * V + v];
    if (!J->brute) {
      /* rho(q, i_q - i_k^block): one rotation per block */
      double rel = (double)iq - (double)off;
      if (MUTANT(4)) rel = (double)iq + (double)off;
      rope_with(scratch_q, D, w, rel, qt);
    }
    for (int j = 0; j < len; ++j) {
      int64_t kb = head_base + ((int64_t)J->block_start[b] + j) * D;
      double dot = 0.0;
      if (!J->brute) {
        for (int i = 0; i < D; ++i) dot += qt[i] * (ks * load_elem(J->k, d->dtype, kb + i));
      } else {
        /* stored key sits at block-local position j: undo that, then encode
         * it at its absolute position in this view, off + j */
        for (int i = 0; i < D; ++i) kk[i] = ks * load_elem(J->k, d->dtype, kb + i);
        rope_with(kk, D, w, -(double)j, kk);
        rope_with(kk, D, w, (double)off + (double)j, ka);
        for (int i = 0; i < D; ++i) dot += qt[i] * ka[i];
      }
      s[t++] = d->scale * dot;
    }
  }

  /* pass 2: one softmax over the concatenation, weighted sum of V */
  double *o = scratch_t;
  for (int i = 0; i < D; ++i) o[i] = 0.0;
  const int64_t obase = ((int64_t)row * d->n_q_heads + h);
  if (n_tok == 0) {
    for (int i = 0; i < D; ++i) J->out[obase * D + i] = 0.0;
    J->lse[obase] = -INFINITY;
    free(s);
    return HWREF_OK;
  }
  double M = -INFINITY;
  for (int64_t u = 0; u < n_tok; ++u) M = s[u] > M ? s[u] : M;
  double Z = 0.0;
  t = 0;
  for (int v = 0; v < V; ++v) {
    int b = J->view_block[(int64_t)row * V + v];
    if (b < 0) continue;
    int len = entry_len(J, row, v, J->block_len[b]);
    for (int j = 0; j < len; ++j) {
      double p = exp(s[t++] - M);
      Z += p;
      int64_t vb = head_base + ((int64_t)J->block_start[b] + j) * D;
      for (int i = 0; i < D; ++i) o[i] += p * (vs * load_elem(J->v, d->dtype, vb + i));
    }
  }
  for (int i = 0; i < D; ++i) J->out[obase * D + i] = o[i] / Z;
  J->lse[obase] = MUTANT(5) ? log(Z) : M + log(Z);
  free(s);
  return HWREF_OK;
}

static void *decode_worker(void *arg) {
  decode_job *J = (decode_job *)arg;
  const hwref_desc *d = J->d;
  double q[1024], t[1024], w[512];
  hwref_rope_freqs(d->head_dim, d->rope_theta, w);
  const int64_t n_items = (int64_t)J->n_sel * d->n_q_heads;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t it = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (it >= n_items) break;
    int32_t row = J->rows ? J->rows[it / d->n_q_heads] : (int32_t)(it / d->n_q_heads);
    int32_t h = (int32_t)(it % d->n_q_heads);
    int rc = decode_item(J, row, h, q, t, w);
    if (rc) {
      pthread_mutex_lock(&J->mu);
      J->status = rc;
      pthread_mutex_unlock(&J->mu);
    }
  }
  return NULL;
}

static int valid_desc(const hwref_desc *d) {
  if (!d) return 0;
  if (d->head_dim <= 0 || d->head_dim % 2 || d->head_dim > 1024) return 0;
  if (d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->n_q_heads % d->n_kv_heads) return 0;
  if (d->n_rows < 0 || d->n_blocks < 0 || d->max_view_blocks < 0) return 0;
  if (d->dtype != HWREF_F32 && d->dtype != HWREF_BF16 && d->dtype != HWREF_FP8) return 0;
  return 1;
}

/*
 * out [rows][Hq][D] and lse [rows][Hq] (natural log) for the selected rows
 * (rows == NULL: all rows, n_sel ignored).  Entries of unselected rows are not
 * touched.  brute = 0 computes the method (query rotated once per block);
 * brute = 1 re-encodes every key at its absolute view position instead.
 * view_limit [rows][V] or NULL: an entry with a limit >= 0 attends only the
 * first min(limit, len) tokens of its block (a chunk's causal order within
 * its own block).
 */
int hwref_attn_decode_scaled(const hwref_desc *d, const void *q, const void *k_cache,
                             const void *v_cache, const float *k_scale, const float *v_scale,
                             const int32_t *block_start, const int32_t *block_len,
                             const int32_t *view_block, const int32_t *view_offset,
                             const int32_t *q_pos, const int32_t *q_to_kv,
                             const int32_t *view_limit, const int32_t *rows, int32_t n_sel,
                             int brute, double *out, double *lse, int n_threads) {
  if (!valid_desc(d) || !out || !lse) return HWREF_EINVAL;
  if (d->dtype == HWREF_FP8 && (!k_scale || !v_scale)) return HWREF_EINVAL;
  decode_job J;
  memset(&J, 0, sizeof J);
  J.d = d;
  J.q = q;
  J.k = k_cache;
  J.v = v_cache;
  J.block_start = block_start;
  J.block_len = block_len;
  J.view_block = view_block;
  J.view_offset = view_offset;
  J.q_pos = q_pos;
  J.q_to_kv = q_to_kv;
  J.view_limit = view_limit;
  J.k_scale = k_scale;
  J.v_scale = v_scale;
  J.rows = rows;
  J.n_sel = rows ? n_sel : d->n_rows;
  J.brute = brute;
  J.out = out;
  J.lse = lse;
  pthread_mutex_init(&J.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < n_threads; ++i)
    if (pthread_create(&th[started], NULL, decode_worker, &J) == 0) ++started;
  decode_worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.status;
}

/* hwref_attn_decode_scaled for bf16 or fp32 caches (no scales). */
int hwref_attn_decode_limited(const hwref_desc *d, const void *q, const void *k_cache,
                              const void *v_cache, const int32_t *block_start,
                              const int32_t *block_len, const int32_t *view_block,
                              const int32_t *view_offset, const int32_t *q_pos,
                              const int32_t *q_to_kv, const int32_t *view_limit,
                              const int32_t *rows, int32_t n_sel, int brute, double *out,
                              double *lse, int n_threads) {
  if (d && d->dtype == HWREF_FP8) return HWREF_EINVAL;
  return hwref_attn_decode_scaled(d, q, k_cache, v_cache, NULL, NULL, block_start, block_len,
                                  view_block, view_offset, q_pos, q_to_kv, view_limit, rows,
                                  n_sel, brute, out, lse, n_threads);
}

/* hwref_attn_decode_limited without limits: every entry sees its whole block. */
int hwref_attn_decode(const hwref_desc *d, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_start, const int32_t *block_len,
                      const int32_t *view_block, const int32_t *view_offset, const int32_t *q_pos,
                      const int32_t *q_to_kv, const int32_t *rows, int32_t n_sel, int brute,
                      double *out, double *lse, int n_threads) {
  return hwref_attn_decode_limited(d, q, k_cache, v_cache, block_start, block_len, view_block,
                                   view_offset, q_pos, q_to_kv, NULL, rows, n_sel, brute, out, lse,
                                   n_threads);
}

/* ------------------------------------------------------------------------ */
/* block commit                                                              */
/* ------------------------------------------------------------------------ */

/*
 * A finished step's KV moves into the shared history, its keys rotated:
 *   K_dst[h][dst_offset + j] = rho(K_src[h][src_begin + j], pos_delta)
 *   V_dst[h][dst_offset + j] = V_src[h][src_begin + j]          (bit copy)
 * for h < Hkv, j < n.  The rotated key is computed in double and rounded once
 * to the storage type (round to nearest, ties to even; E4M3 saturates at
 * +-448).  E4M3 pools take no scale here: a rotation is linear, so the key's
 * head scale carries over unchanged when both pools share it.  Destination entries
 * outside [dst_offset, dst_offset + n) are left as they are.  If k_exact is
 * not NULL it receives the unrounded keys, [Hkv][n][D].
 * Heads are strided by *_head_stride elements.  src and dst must not overlap
 * (checked by the caller).
 */
int hwref_block_commit(int dtype, int32_t n_kv_heads, int32_t head_dim, double rope_theta,
                       const void *k_src, const void *v_src, int64_t src_head_stride,
                       int32_t src_begin, int32_t n_tokens, void *k_dst, void *v_dst,
                       int64_t dst_head_stride, int32_t dst_offset, int32_t pos_delta,
                       double *k_exact) {
  if (head_dim <= 0 || head_dim % 2 || head_dim > 1024 || n_kv_heads <= 0 || n_tokens < 0)
    return HWREF_EINVAL;
  if (dtype != HWREF_F32 && dtype != HWREF_BF16 && dtype != HWREF_FP8) return HWREF_EINVAL;
  const int D = head_dim;
  double w[512], x[1024], y[1024];
  hwref_rope_freqs(D, rope_theta, w);
  for (int h = 0; h < n_kv_heads; ++h) {
    for (int j = 0; j < n_tokens; ++j) {
      int64_t si = h * src_head_stride + (int64_t)(src_begin + j) * D;
      int64_t di = h * dst_head_stride + (int64_t)(dst_offset + j) * D;
      if (MUTANT(7)) /* tokens placed in reverse order */
        di = h * dst_head_stride + (int64_t)(dst_offset + n_tokens - 1 - j) * D;
      for (int i = 0; i < D; ++i) x[i] = load_elem(k_src, dtype, si + i);
      rope_with(x, D, w, MUTANT(8) ? -(double)pos_delta : (double)pos_delta, y);
      for (int i = 0; i < D; ++i) {
        store_elem(k_dst, dtype, di + i, y[i]);
        copy_elem(v_dst, v_src, dtype, di + i, si + i);
        if (k_exact) k_exact[((int64_t)h * n_tokens + j) * D + i] = y[i];
      }
    }
  }
  return HWREF_OK;
}

/* Exposed for the tests: the oracle's own double -> bf16 rounding, and its
 * E4M3 decoding and rounding. */
uint16_t hwref_bf16_from_double(double x) { return bf16_from_double(x); }
double hwref_e4m3_to_double(uint8_t b) { return e4m3_to_double(b); }
uint8_t hwref_e4m3_from_double(double x) { return e4m3_from_double(x); }
