/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for Multi-head Latent Attention
 * decode.  TEST INFRASTRUCTURE ONLY: it is called by the test-suite, by the
 * package's smoke check and by the benchmark's CPU-baseline leg, never by the
 * product path.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the UNABSORBED definition, written out directly from
 *   "DeepSeek-V3" (ekkoxiao.github.io), section "Multi-Head Latent Attention":
 *     - KeyValue:   k^C_{j,i} = W_i^UK c_j ,  v^C_{j,i} = W_i^UV c_j
 *                   (W_i^UK, W_i^UV are the d_h x d_c row blocks of head i),
 *                   k^R_j = RoPE_j(.)  shared by all heads;
 *     - Query:      q^R_{t,i} = RoPE_t(.);
 *     - 注意力计算 (attention computation):
 *                   s_{t,j,i} = (q^C . k^C_{j,i} + q^R . k^R_j) / sqrt(d_h + d_h^R),
 *                   a = softmax over the visible positions j,
 *                   o_{t,i} = sum_j a_{t,j,i} v^C_{j,i};
 *     - YaRN 扩展:  RoPE rotates the j-th 2-D component pair at position m by
 *                   the angle m * theta_j.
 * Every key and value is expanded per head and per position; nothing is
 * absorbed, fused, blocked or reordered.  The softmax is the textbook
 * two-pass form: all scores, then their maximum, then normalised weights.
 *
 * Readings taken where the pages leave a step open (all listed in the design
 * notes of the repository):
 *   - RoPE pairs are interleaved (x_{2j}, x_{2j+1}); theta_j = base^(-2j/d_r);
 *     the rotation is (x cos - y sin, x sin + y cos).
 *   - positions are 0-based: keys sit at 0..L_b-1, query s of S sits at
 *     L_b - S + s and sees keys 0..L_b - S + s inclusive.
 *   - the cache holds the PRE-RoPE k_R; the oracle rotates it itself.
 *   - YaRN ("YaRN 扩展", and "Long Context Extension" of the technical report
 *     reading): theta'_j = (1 - g_j) theta_j / s + g_j theta_j, where g_j = 1
 *     in the high-frequency band and 0 in the low one.  The pages give the band
 *     edges only as alpha = 1, beta = 32; the ramp taken here is linear in the
 *     number of turns a pair makes over the original context,
 *     r_j = L_orig theta_j / (2 pi):  g_j = clamp((r_j - alpha) / (beta - alpha), 0, 1).
 *     It applies to the whole decoupled RoPE branch (q^R and k^R), the only
 *     place RoPE is used.
 *
 * The step functions below (absorb, latent attention, up-projection) restate
 * the absorbed identities of section "潜在向量的作用" (role of the latent
 * vector) one step at a time, so that each CUDA kernel can be checked alone.
 * They too are plain loops in fp64.
 *
 * Inputs are either fp64 arrays or raw bf16 bit patterns (uint16); bf16 is
 * widened exactly (bits << 16 -> binary32 -> binary64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes of the input arrays */
#define ORACLE_F64 0
#define ORACLE_BF16 1

static inline double ld(const void *p, size_t i, int dtype) {
  if (dtype == ORACLE_F64) return ((const double *)p)[i];
  uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

int mla_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* theta_j = base^(-2j/d_r), j = 0 .. d_r/2 - 1 */
static void base_theta(double base, int d_r, double *theta) {
  for (int j = 0; j < d_r / 2; ++j) theta[j] = pow(base, -2.0 * (double)j / (double)d_r);
}

/*
 * YaRN frequencies ("YaRN 扩展"): theta'_j = (1 - g_j) theta_j / s + g_j theta_j,
 * g_j = 1 for pairs that turn many times over the original context (high
 * frequency, kept), 0 for pairs that turn less than once (low frequency,
 * divided by s), linear in between (see the reading above).
 */
int mla_oracle_yarn_theta(double base, int d_r, double s, double alpha, double beta,
                          double orig_len, double *theta) {
  if (d_r <= 0 || (d_r & 1) || !(s >= 1.0) || !(beta > alpha) || !(orig_len > 0.0)) return 1;
  const double two_pi = 6.283185307179586476925286766559;
  base_theta(base, d_r, theta);
  for (int j = 0; j < d_r / 2; ++j) {
    double r = orig_len * theta[j] / two_pi; /* turns over the original context */
    double g = (r - alpha) / (beta - alpha);
    if (g < 0.0) g = 0.0;
    if (g > 1.0) g = 1.0;
    theta[j] = (1.0 - g) * theta[j] / s + g * theta[j];
  }
  return 0;
}

/*
 * YaRN score factor ("Long Context Extension" of the technical report reading:
 * the attention scores are scaled by 0.1 ln s + 1; "YaRN 扩展" applies it to the
 * scores before the softmax): the softmax scale becomes
 * (0.1 ln s + 1) / sqrt(d_h + d_r) in place of 1 / sqrt(d_h + d_r).
 */
int mla_oracle_yarn_softmax_scale(double s, int d_h, int d_r, double *out) {
  if (!(s >= 1.0) || d_h <= 0 || d_r < 0 || !out) return 1;
  *out = (0.1 * log(s) + 1.0) / sqrt((double)(d_h + d_r));
  return 0;
}

/* RoPE of one d_r-vector at integer position pos ("YaRN 扩展": phi_{m,j} = m theta_j). */
static void rope_vec(const double *x, int d_r, double pos, const double *theta, double *y) {
  for (int j = 0; j < d_r / 2; ++j) {
    double phi = pos * theta[j];
    double c = cos(phi), s = sin(phi);
    double x0 = x[2 * j], x1 = x[2 * j + 1];
    y[2 * j] = x0 * c - x1 * s;
    y[2 * j + 1] = x0 * s + x1 * c;
  }
}

/* Public RoPE: x[n, d_r] rotated at positions pos[n] with frequencies theta[d_r/2]. */
int mla_oracle_rope_theta(const void *x, int dtype, const int64_t *pos, int n, int d_r,
                          const double *theta, double *out) {
  if (d_r <= 0 || (d_r & 1)) return 1;
  double *tmp = (double *)malloc(sizeof(double) * (size_t)d_r);
  if (!tmp) return 2;
  for (int r = 0; r < n; ++r) {
    for (int k = 0; k < d_r; ++k) tmp[k] = ld(x, (size_t)r * d_r + k, dtype);
    rope_vec(tmp, d_r, (double)pos[r], theta, out + (size_t)r * d_r);
  }
  free(tmp);
  return 0;
}

/* The same with theta_j = base^(-2j/d_r). */
int mla_oracle_rope(const void *x, int dtype, const int64_t *pos, int n, int d_r,
                    double base, double *out) {
  if (d_r <= 0 || (d_r & 1) || d_r > 1024) return 1;
  double theta[512];
  base_theta(base, d_r, theta);
  return mla_oracle_rope_theta(x, dtype, pos, n, d_r, theta, out);
}

/*
 * Unabsorbed decode for a list of output rows.
 *   q_nope [B,S,H,d_h]   q_rope [B,S,H,d_r] (pre-RoPE)
 *   c_kv   [B,Lmax,d_c]  k_r    [B,Lmax,d_r] (pre-RoPE)
 *   W_UK   [H,d_h,d_c]   W_UV   [H,d_v,d_c]
 *   seqlens[B]
 *   theta  : RoPE frequencies [d_r/2] (both q^R and k^R use them)
 *   rows   : flat indices (b*S + s)*H + h to compute (NULL -> all B*S*H rows)
 *   out    : [n_rows, d_v] fp64
 *   wsum   : optional [n_rows], the sum of the softmax weights of each row
 * Returns 0, or a nonzero code for an invalid argument.
 */
int mla_oracle_decode_theta(const void *q_nope, const void *q_rope, const void *c_kv,
                            const void *k_r, const void *W_UK, const void *W_UV, int dtype,
                            const int32_t *seqlens, int B, int S, int H, int Lmax, int d_c,
                            int d_h, int d_r, int d_v, double softmax_scale, const double *theta,
                            const int64_t *rows, int64_t n_rows, double *out, double *wsum) {
  if (B <= 0 || S <= 0 || H <= 0 || Lmax <= 0 || d_c <= 0 || d_h <= 0 || d_r < 0 ||
      (d_r & 1) || d_v <= 0)
    return 1;
  for (int b = 0; b < B; ++b)
    if (seqlens[b] < S || seqlens[b] > Lmax) return 3;
  int64_t total = (int64_t)B * S * H;
  if (rows == NULL) n_rows = total;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows && (rows[r] < 0 || rows[r] >= total)) return 4;
  int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t flat = rows ? rows[r] : r;
    int h = (int)(flat % H);
    int s = (int)((flat / H) % S);
    int b = (int)(flat / ((int64_t)H * S));
    int L = seqlens[b];
    int pos_q = L - S + s; /* the query's own position; keys 0..pos_q are visible */
    int nvis = pos_q + 1;

    double *qn = (double *)malloc(sizeof(double) * d_h);
    double *qr_raw = (double *)malloc(sizeof(double) * (d_r ? d_r : 1));
    double *qr = (double *)malloc(sizeof(double) * (d_r ? d_r : 1));
    double *kr_raw = (double *)malloc(sizeof(double) * (d_r ? d_r : 1));
    double *kr = (double *)malloc(sizeof(double) * (d_r ? d_r : 1));
    double *c = (double *)malloc(sizeof(double) * d_c);
    double *kc = (double *)malloc(sizeof(double) * d_h);
    double *vc = (double *)malloc(sizeof(double) * d_v);
    double *score = (double *)malloc(sizeof(double) * nvis);
    if (!qn || !qr_raw || !qr || !kr_raw || !kr || !c || !kc || !vc || !score) {
#pragma omp atomic write
      bad = 2;
    } else {
      size_t qoff = (((size_t)b * S + s) * H + h);
      for (int d = 0; d < d_h; ++d) qn[d] = ld(q_nope, qoff * d_h + d, dtype);
      for (int d = 0; d < d_r; ++d) qr_raw[d] = ld(q_rope, qoff * d_r + d, dtype);
      rope_vec(qr_raw, d_r, (double)pos_q, theta, qr);

      /* pass 1: every score, with the key expanded per head */
      for (int j = 0; j < nvis; ++j) {
        size_t coff = ((size_t)b * Lmax + j);
        for (int k = 0; k < d_c; ++k) c[k] = ld(c_kv, coff * d_c + k, dtype);
        for (int d = 0; d < d_h; ++d) { /* k^C = W_i^UK c_j */
          double acc = 0.0;
          size_t woff = ((size_t)h * d_h + d) * d_c;
          for (int k = 0; k < d_c; ++k) acc += ld(W_UK, woff + k, dtype) * c[k];
          kc[d] = acc;
        }
        for (int d = 0; d < d_r; ++d) kr_raw[d] = ld(k_r, coff * d_r + d, dtype);
        rope_vec(kr_raw, d_r, (double)j, theta, kr); /* k^R_j = RoPE_j(.) */
        double dot = 0.0;
        for (int d = 0; d < d_h; ++d) dot += qn[d] * kc[d];
        for (int d = 0; d < d_r; ++d) dot += qr[d] * kr[d];
        score[j] = dot * softmax_scale;
      }
      /* softmax over the visible positions */
      double m = -INFINITY;
      for (int j = 0; j < nvis; ++j) m = score[j] > m ? score[j] : m;
      double den = 0.0;
      for (int j = 0; j < nvis; ++j) den += exp(score[j] - m);
      double *o = out + (size_t)r * d_v;
      for (int d = 0; d < d_v; ++d) o[d] = 0.0;
      double asum = 0.0;
      /* pass 2: o = sum_j a_j v^C_j with the value expanded per head */
      for (int j = 0; j < nvis; ++j) {
        double a = exp(score[j] - m) / den;
        asum += a;
        size_t coff = ((size_t)b * Lmax + j);
        for (int k = 0; k < d_c; ++k) c[k] = ld(c_kv, coff * d_c + k, dtype);
        for (int d = 0; d < d_v; ++d) { /* v^C = W_i^UV c_j */
          double acc = 0.0;
          size_t woff = ((size_t)h * d_v + d) * d_c;
          for (int k = 0; k < d_c; ++k) acc += ld(W_UV, woff + k, dtype) * c[k];
          vc[d] = acc;
        }
        for (int d = 0; d < d_v; ++d) o[d] += a * vc[d];
      }
      if (wsum) wsum[r] = asum;
    }
    free(qn); free(qr_raw); free(qr); free(kr_raw); free(kr);
    free(c); free(kc); free(vc); free(score);
  }
  return bad;
}

/* The same with theta_j = rope_base^(-2j/d_r). */
int mla_oracle_decode(const void *q_nope, const void *q_rope, const void *c_kv,
                      const void *k_r, const void *W_UK, const void *W_UV, int dtype,
                      const int32_t *seqlens, int B, int S, int H, int Lmax, int d_c,
                      int d_h, int d_r, int d_v, double softmax_scale, double rope_base,
                      const int64_t *rows, int64_t n_rows, double *out, double *wsum) {
  if (d_r < 0 || d_r > 1024) return 1;
  double theta[512];
  base_theta(rope_base, d_r, theta);
  return mla_oracle_decode_theta(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, dtype, seqlens, B, S, H,
                                 Lmax, d_c, d_h, d_r, d_v, softmax_scale, theta, rows, n_rows,
                                 out, wsum);
}

/*
 * Absorption step ("潜在向量的作用"): q~_{b,s,h} = (W_h^UK)^T q^C_{b,s,h}.
 *   q_nope [N,H,d_h], W_UK [H,d_h,d_c] -> out [N,H,d_c]
 */
int mla_oracle_absorb(const void *q_nope, const void *W_UK, int dtype, int N, int H,
                      int d_h, int d_c, double *out) {
  if (N < 0 || H <= 0 || d_h <= 0 || d_c <= 0) return 1;
#pragma omp parallel for collapse(2)
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h) {
      double *o = out + ((size_t)n * H + h) * d_c;
      for (int k = 0; k < d_c; ++k) {
        double acc = 0.0;
        for (int d = 0; d < d_h; ++d)
          acc += ld(W_UK, ((size_t)h * d_h + d) * d_c + k, dtype) *
                 ld(q_nope, ((size_t)n * H + h) * d_h + d, dtype);
        o[k] = acc;
      }
    }
  return 0;
}

/*
 * Up-projection step ("潜在向量的作用"): o_{b,s,h} = W_h^UV o^lat_{b,s,h}.
 *   o_lat [N,H,d_c], W_UV [H,d_v,d_c] -> out [N,H,d_v]
 */
int mla_oracle_up_project(const void *o_lat, const void *W_UV, int dtype, int N, int H,
                          int d_v, int d_c, double *out) {
  if (N < 0 || H <= 0 || d_v <= 0 || d_c <= 0) return 1;
#pragma omp parallel for collapse(2)
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h) {
      double *o = out + ((size_t)n * H + h) * d_v;
      for (int d = 0; d < d_v; ++d) {
        double acc = 0.0;
        for (int k = 0; k < d_c; ++k)
          acc += ld(W_UV, ((size_t)h * d_v + d) * d_c + k, dtype) *
                 ld(o_lat, ((size_t)n * H + h) * d_c + k, dtype);
        o[d] = acc;
      }
    }
  return 0;
}

/*
 * Latent-space attention step ("潜在向量的作用" + "注意力计算"), for checking
 * the decode kernel on its own.  Its query is the already absorbed and
 * rotated q_cat = [q~ ; RoPE(q^R)] and its keys the already rotated cache:
 *   s_j = (q~ . c_j + q^R . k^R_j) * scale ,  a = softmax_j ,  o^lat = sum_j a_j c_j
 *   q_cat [B,S,H,d_c+d_r], c_kv [B,Lmax,d_c], k_rot [B,Lmax,d_r], seqlens[B]
 *   rows : flat indices (b*S+s)*H+h (NULL -> all)      out : [n_rows, d_c]
 */
int mla_oracle_latent_attention(const void *q_cat, const void *c_kv, const void *k_rot,
                                int dtype, const int32_t *seqlens, int B, int S, int H,
                                int Lmax, int d_c, int d_r, double softmax_scale,
                                const int64_t *rows, int64_t n_rows, double *out) {
  if (B <= 0 || S <= 0 || H <= 0 || Lmax <= 0 || d_c <= 0 || d_r < 0) return 1;
  for (int b = 0; b < B; ++b)
    if (seqlens[b] < S || seqlens[b] > Lmax) return 3;
  int64_t total = (int64_t)B * S * H;
  if (rows == NULL) n_rows = total;
  int dq = d_c + d_r;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t flat = rows ? rows[r] : r;
    if (flat < 0 || flat >= total) {
#pragma omp atomic write
      bad = 4;
      continue;
    }
    int h = (int)(flat % H);
    int s = (int)((flat / H) % S);
    int b = (int)(flat / ((int64_t)H * S));
    int nvis = seqlens[b] - S + s + 1;
    double *score = (double *)malloc(sizeof(double) * nvis);
    if (!score) {
#pragma omp atomic write
      bad = 2;
      continue;
    }
    size_t qoff = (((size_t)b * S + s) * H + h) * dq;
    for (int j = 0; j < nvis; ++j) {
      size_t row = (size_t)b * Lmax + j;
      double dot = 0.0;
      for (int k = 0; k < d_c; ++k) dot += ld(q_cat, qoff + k, dtype) * ld(c_kv, row * d_c + k, dtype);
      for (int k = 0; k < d_r; ++k)
        dot += ld(q_cat, qoff + d_c + k, dtype) * ld(k_rot, row * d_r + k, dtype);
      score[j] = dot * softmax_scale;
    }
    double m = -INFINITY;
    for (int j = 0; j < nvis; ++j) m = score[j] > m ? score[j] : m;
    double den = 0.0;
    for (int j = 0; j < nvis; ++j) den += exp(score[j] - m);
    double *o = out + (size_t)r * d_c;
    for (int k = 0; k < d_c; ++k) o[k] = 0.0;
    for (int j = 0; j < nvis; ++j) {
      double a = exp(score[j] - m) / den;
      size_t row = (size_t)b * Lmax + j;
      for (int k = 0; k < d_c; ++k) o[k] += a * ld(c_kv, row * d_c + k, dtype);
    }
    free(score);
  }
  return bad;
}
