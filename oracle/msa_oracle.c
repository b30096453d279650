/*
 * msa_oracle.c -- plain CPU reference of the MiniMax Sparse Attention (MSA)
 * forward pass.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The product library
 * never links, loads or calls this file, and this file shares no code, header
 * or constant with the CUDA path.
 *
 * What it computes (one function per step, in the order the method runs):
 *
 *  1. msa_oracle_pooled -- Index Branch scores and block max-pool.
 *     "MiniMax Sparse Attention: let each query pick its own blocks",
 *     section "The mechanism, precisely", first bullet: one index-query head
 *     per GQA group, one shared index-key head, token scores Q_idx . K_idx^T,
 *     max-pooled to 128-token blocks.  The same page's Figure 1 (architecture
 *     diagram) shows the order: score matrix -> block max pooling -> top-k.
 *     Only keys at or before the query's own position enter a pool.
 *
 *  2. msa_oracle_select -- top-k block selection with the local block forced
 *     in.  Same section: keep the top-k blocks (k = 16 deployed), the block
 *     the query sits in is always kept; the atlas record of the report
 *     ("MiniMax M3 428B" architecture page, summary paragraph) states the
 *     local block is forced in and that selection is per query and per group.
 *     Ranking: pooled score descending, ties to the lower block index.
 *
 *     msa_oracle_index chains steps 1 and 2 (the Index Branch alone);
 *     msa_oracle_pooled_fp8 and msa_oracle_index_fp8 do the same over E4M3
 *     index inputs (see the fp8 notes near the end of the file).
 *
 *  3. msa_oracle_attention -- Main Branch: exact softmax attention of every
 *     query head over only the tokens of its group's selected blocks.  Same
 *     section, second bullet: attention stays exact but covers only the
 *     selected blocks, and all heads of a group share one block set.
 *
 * Precision.  The pages fix no precision.  Token index scores are formed in
 * double from the exact bf16 inputs and rounded once to fp32; pooling and
 * ranking then run in fp32, because a float comparison there decides an
 * integer (which blocks are kept) and the GPU path takes that decision in
 * fp32.  The Main Branch runs entirely in double.
 *
 * Layout (packed variable-length batch, row-major, contiguous):
 *   q      [total_q][hq][head_dim]      bf16 bits (uint16)
 *   k, v   [total_k][hkv][head_dim]     bf16 bits
 *   q_idx  [total_q][hkv][d_idx]        bf16 bits
 *   k_idx  [total_k][d_idx]             bf16 bits
 *   cu_q, cu_k  [num_seqs + 1] prefix sums of per-sequence query / key counts.
 * Query t of sequence s sits at key position pos = kv_len - q_len + t
 * (queries are the last q_len positions of the sequence; a decode step is
 * q_len = 1).  Head h belongs to group h / (hq / hkv).
 *
 * Every function returns 0 on success and a negative code on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* sum_d q[d] * k[d], accumulated in double in order d = 0 .. n-1, for bf16
 * vectors already widened to double (exactly; so are their products). */
static double dot_wide(const double *q, const double *k, int n) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) acc += q[d] * k[d];
  return acc;
}

/* dot_wide(q, k + u * n, n) for the four consecutive rows u = 0..3 of k,
 * computed side by side (four independent sums, each in the same order). */
static void dot4_wide(const double *q, const double *k, int n, double out[4]) {
  double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
  for (int d = 0; d < n; ++d) {
    a0 += q[d] * k[d];
    a1 += q[d] * k[n + d];
    a2 += q[d] * k[2 * n + d];
    a3 += q[d] * k[3 * n + d];
  }
  out[0] = a0;
  out[1] = a1;
  out[2] = a2;
  out[3] = a3;
}

/* Checks the two prefix-sum arrays: nondecreasing, start at 0, and every
 * sequence has at least as many keys as queries. */
static int check_seqlens(int num_seqs, const int32_t *cu_q, const int32_t *cu_k) {
  if (num_seqs < 0 || !cu_q || !cu_k) return ORACLE_EINVAL;
  if (cu_q[0] != 0 || cu_k[0] != 0) return ORACLE_EINVAL;
  for (int s = 0; s < num_seqs; ++s) {
    int q_len = cu_q[s + 1] - cu_q[s];
    int kv_len = cu_k[s + 1] - cu_k[s];
    if (q_len < 0 || kv_len < 0 || kv_len < q_len) return ORACLE_EINVAL;
  }
  return ORACLE_OK;
}

/* Sequence that owns packed query row i (linear scan: plain, not fast). */
static int seq_of_query(int num_seqs, const int32_t *cu_q, int i) {
  for (int s = 0; s < num_seqs; ++s)
    if (i >= cu_q[s] && i < cu_q[s + 1]) return s;
  return -1;
}

int msa_oracle_num_blocks(int pos, int block) { return pos / block + 1; }

double msa_oracle_e4m3_value(uint8_t code);

/* The inputs of step 1, in one of two forms: bf16 bits (q_idx, k_idx), or
 * E4M3 codes with fp32 scales (q8, k8; the fp8 index notes below), each
 * element then read as value(code) * scale.  The scores are the same
 * definition on those values. */
typedef struct {
  const uint16_t *q_idx, *k_idx; /* bf16: [total_q][hkv][d_idx], [total_k][d_idx] */
  const uint8_t *q8, *k8;        /* E4M3: same shapes */
  const float *q_scale;          /* [total_q][hkv]: one per (query row, group) */
  const float *k_scale;          /* [n_key_blocks]: one per key block of a sequence */
} index_inputs;

/* Index keys of sequence s widened to double, kd[j * d_idx + d] for its
 * kv_len keys; blk0 = scale row of the sequence's first key block. */
static void widen_keys(const index_inputs *in, const int32_t *cu_k, int s, int d_idx, int block, int blk0,
                       double *kd) {
  const int kv_len = cu_k[s + 1] - cu_k[s];
  for (int j = 0; j < kv_len; ++j)
    for (int d = 0; d < d_idx; ++d) {
      const size_t e = (size_t)(cu_k[s] + j) * d_idx + d;
      kd[(size_t)j * d_idx + d] = in->k8 ? msa_oracle_e4m3_value(in->k8[e]) * (double)in->k_scale[blk0 + j / block]
                                         : bf16_bits_to_double(in->k_idx[e]);
    }
}

/* Index query row i (all groups) widened to double, qd[g * d_idx + d]. */
static void widen_query(const index_inputs *in, int i, int hkv, int d_idx, double *qd) {
  for (int g = 0; g < hkv; ++g)
    for (int d = 0; d < d_idx; ++d) {
      const size_t e = ((size_t)i * hkv + g) * d_idx + d;
      qd[g * d_idx + d] = in->q8 ? msa_oracle_e4m3_value(in->q8[e]) * (double)in->q_scale[(size_t)i * hkv + g]
                                 : bf16_bits_to_double(in->q_idx[e]);
    }
}

/*
 * Step 1.  pooled[r][g][b] for query row rows[r] (all rows when rows == NULL,
 * then n_rows must equal total_q) and group g:
 *     s_j      = fp32( sum_d q_idx[i][g][d] * k_idx[key j][d] )   (sum in double)
 *     pooled_b = max over keys j of block b with j <= pos of s_j  (fp32)
 * for b = 0 .. pos / block.  Entries b > pos / block are set to -INFINITY.
 * The bf16 inputs and their products are exact in double; so are E4M3 values
 * times fp32 scales, whose products carry up to 56 significant bits and are
 * rounded to double (far below the final rounding to fp32).
 */
static int pooled_core(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                       int hkv, int d_idx, int block, const index_inputs *in,
                       int n_rows, const int32_t *rows,
                       int nb_stride, float *pooled) {
  if (check_seqlens(num_seqs, cu_q, cu_k)) return ORACLE_EINVAL;
  if (hkv <= 0 || d_idx <= 0 || block <= 0 || n_rows < 0 || !pooled) return ORACLE_EINVAL;
  if (in->q8 ? (!in->k8 || !in->q_scale || !in->k_scale) : (!in->q_idx || !in->k_idx)) return ORACLE_EINVAL;
  const int total_q = cu_q[num_seqs];
  if (!rows && n_rows != total_q) return ORACLE_EINVAL;
  /* The rows are processed one sequence at a time, with that sequence's index
   * keys widened once to double while its rows are scored. */
  int bad = 0;
  int *row_seq = (int *)malloc(sizeof(int) * (size_t)(n_rows > 0 ? n_rows : 1));
  if (!row_seq) return ORACLE_ENOMEM;
  for (int r = 0; r < n_rows; ++r) {
    const int i = rows ? rows[r] : r;
    row_seq[r] = (i >= 0 && i < total_q) ? seq_of_query(num_seqs, cu_q, i) : -1;
    if (row_seq[r] < 0) bad = 1;
  }
  int blk0 = 0; /* scale row of sequence s's first key block */
  for (int s = 0; s < num_seqs && !bad; blk0 += (cu_k[s + 1] - cu_k[s] + block - 1) / block, ++s) {
    int used = 0;
    for (int r = 0; r < n_rows && !used; ++r) used = (row_seq[r] == s);
    if (!used) continue;
    const int q_len = cu_q[s + 1] - cu_q[s];
    const int kv_len = cu_k[s + 1] - cu_k[s];
    double *kd = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1) * d_idx);
    if (!kd) { bad = 1; break; }
    widen_keys(in, cu_k, s, d_idx, block, blk0, kd);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < n_rows; ++r) {
      if (row_seq[r] != s) continue;
      const int i = rows ? rows[r] : r;
      const int pos = kv_len - q_len + (i - cu_q[s]);
      const int nb = msa_oracle_num_blocks(pos, block);
      if (nb > nb_stride) { bad = 1; continue; }
      double *qd = (double *)malloc(sizeof(double) * (size_t)hkv * d_idx);  /* qd[g * d_idx + d] */
      if (!qd) { bad = 1; continue; }
      widen_query(in, i, hkv, d_idx, qd);
      float *out = pooled + (size_t)r * hkv * nb_stride;  /* out[g * nb_stride + b] */
      for (int e = 0; e < hkv * nb_stride; ++e) out[e] = -INFINITY;
      for (int b = 0; b < nb; ++b) {
        const int j_end = ((b + 1) * block < pos + 1) ? (b + 1) * block : pos + 1;
        int j = b * block;
        /* four keys at a time (every group's query against the same four key
         * rows): independent sums, each over d in order */
        for (; j + 4 <= j_end; j += 4)
          for (int g = 0; g < hkv; ++g) {
            double sc[4];
            dot4_wide(qd + (size_t)g * d_idx, kd + (size_t)j * d_idx, d_idx, sc);
            for (int u = 0; u < 4; ++u)
              if ((float)sc[u] > out[g * nb_stride + b]) out[g * nb_stride + b] = (float)sc[u];
          }
        for (; j < j_end; ++j)
          for (int g = 0; g < hkv; ++g) {
            const float sj = (float)dot_wide(qd + (size_t)g * d_idx, kd + (size_t)j * d_idx, d_idx);
            if (sj > out[g * nb_stride + b]) out[g * nb_stride + b] = sj;
          }
      }
      free(qd);
    }
    free(kd);
  }
  free(row_seq);
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}

int msa_oracle_pooled(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                      int hkv, int d_idx, int block,
                      const uint16_t *q_idx, const uint16_t *k_idx,
                      int n_rows, const int32_t *rows,
                      int nb_stride, float *pooled) {
  const index_inputs in = {q_idx, k_idx, NULL, NULL, NULL, NULL};
  return pooled_core(num_seqs, cu_q, cu_k, hkv, d_idx, block, &in, n_rows, rows, nb_stride, pooled);
}

/*
 * Step 2.  For one pooled row of nb valid blocks whose local block is
 * local = nb - 1 (the query's own block is the last causal one):
 *   take the min(k - 1, nb - 1) best non-local blocks, best meaning larger
 *   pooled score, equal scores going to the lower block index; add the local
 *   block; write the set in ascending block order to sel[0..k), padding with
 *   -1.  (When k <= 0 nothing is selected.)
 * *gap receives the relative gap between the last selected non-local block
 * and the best unselected non-local block, |a - b| / max(|a|, |b|, 1e-30),
 * or +INFINITY when every non-local block is selected or none is (no float
 * comparison decides the set).  Scores are compared as fp32 values; +0 and -0
 * compare equal.
 */
int msa_oracle_select(int nb, const float *pooled_row, int k, int32_t *sel, double *gap) {
  if (nb <= 0 || k < 0 || !pooled_row || (k > 0 && !sel)) return ORACLE_EINVAL;
  const int local = nb - 1;
  const int want = (k - 1 < nb - 1) ? k - 1 : nb - 1;
  char *taken = (char *)calloc((size_t)nb, 1);
  int32_t *chosen = (int32_t *)malloc(sizeof(int32_t) * (size_t)(want > 0 ? want : 1));
  if (!taken || !chosen) { free(taken); free(chosen); return ORACLE_ENOMEM; }
  if (k > 0) taken[local] = 1;
  float last_val = 0.f;
  for (int r = 0; r < want; ++r) {
    int best = -1;
    for (int b = 0; b < nb; ++b) {
      if (taken[b]) continue;
      /* scanning b upward with a strict '>' keeps the lower index on ties */
      if (best < 0 || pooled_row[b] > pooled_row[best]) best = b;
    }
    taken[best] = 1;
    chosen[r] = best;
    last_val = pooled_row[best];
  }
  if (gap) {
    *gap = INFINITY;
    if (want >= 1 && want < nb - 1) {
      int next = -1;
      for (int b = 0; b < nb; ++b) {
        if (taken[b]) continue;
        if (next < 0 || pooled_row[b] > pooled_row[next]) next = b;
      }
      double a = last_val, c = pooled_row[next];
      double den = fabs(a) > fabs(c) ? fabs(a) : fabs(c);
      if (den < 1e-30) den = 1e-30;
      *gap = fabs(a - c) / den;
    }
  }
  /* ascending block order, -1 padding at the tail */
  int n = 0;
  for (int b = 0; b < nb && n < k; ++b)
    if (taken[b]) sel[n++] = b;
  for (; n < k; ++n) sel[n] = -1;
  free(taken);
  free(chosen);
  return ORACLE_OK;
}

/*
 * Step 3.  For query row rows[r] and every head h (group g = h / (hq/hkv)),
 * with the group's selected blocks idx[r][g][0..topk) (-1 entries ignored):
 *   x_j  = scale * sum_d q[i][h][d] * k[key j][g][d]   over tokens j of the
 *          selected blocks with j <= pos
 *   m    = max_j x_j,  l = sum_j exp(x_j - m)
 *   o[r][h][:] = sum_j exp(x_j - m) v[key j][g][:] / l,  lse[r][h] = m + ln l
 * all in double.  A row with no token (impossible when the local block is
 * selected) gets o = 0 and lse = -INFINITY.
 */
int msa_oracle_attention(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                         int hq, int hkv, int head_dim, int block, int topk, double scale,
                         const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const int32_t *idx, int n_rows, const int32_t *rows,
                         double *o, double *lse) {
  if (check_seqlens(num_seqs, cu_q, cu_k)) return ORACLE_EINVAL;
  if (hq <= 0 || hkv <= 0 || hq % hkv || head_dim <= 0 || block <= 0 || topk <= 0) return ORACLE_EINVAL;
  if (!q || !k || !v || !idx || !o || !lse || n_rows < 0) return ORACLE_EINVAL;
  const int total_q = cu_q[num_seqs];
  if (!rows && n_rows != total_q) return ORACLE_EINVAL;
  const int G = hq / hkv;
  int bad = 0;
#pragma omp parallel reduction(| : bad)
  {
    double *x = (double *)malloc(sizeof(double) * (size_t)topk * block);
    int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk * block);
    if (!x || !key) bad = 1;
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
      if (!x || !key) continue;
      const int i = rows ? rows[r] : r;
      const int s = (i >= 0 && i < total_q) ? seq_of_query(num_seqs, cu_q, i) : -1;
      if (s < 0) { bad = 1; continue; }
      const int q_len = cu_q[s + 1] - cu_q[s];
      const int kv_len = cu_k[s + 1] - cu_k[s];
      const int pos = kv_len - q_len + (i - cu_q[s]);
      for (int h = 0; h < hq; ++h) {
        const int g = h / G;
        const int32_t *sel = idx + ((size_t)r * hkv + g) * topk;
        /* gather the attended token positions */
        int n = 0;
        for (int e = 0; e < topk; ++e) {
          const int b = sel[e];
          if (b < 0) continue;
          for (int j = b * block; j < (b + 1) * block && j <= pos; ++j) key[n++] = j;
        }
        const uint16_t *qh = q + ((size_t)i * hq + h) * head_dim;
        double *oh = o + ((size_t)r * hq + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) oh[d] = 0.0;
        if (n == 0) { lse[(size_t)r * hq + h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
          const uint16_t *kj = k + ((size_t)(cu_k[s] + key[t]) * hkv + g) * head_dim;
          double acc = 0.0;
          for (int d = 0; d < head_dim; ++d) acc += bf16_bits_to_double(qh[d]) * bf16_bits_to_double(kj[d]);
          x[t] = scale * acc;
          if (x[t] > m) m = x[t];
        }
        double l = 0.0;
        for (int t = 0; t < n; ++t) {
          const double p = exp(x[t] - m);
          l += p;
          const uint16_t *vj = v + ((size_t)(cu_k[s] + key[t]) * hkv + g) * head_dim;
          for (int d = 0; d < head_dim; ++d) oh[d] += p * bf16_bits_to_double(vj[d]);
        }
        for (int d = 0; d < head_dim; ++d) oh[d] /= l;
        lse[(size_t)r * hq + h] = m + log(l);
      }
    }
    free(x);
    free(key);
  }
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}

/*
 * Steps 1-2 chained (the Index Branch alone) for the query rows listed in rows
 * (all when NULL): idx [n_rows][hkv][topk] (ascending, -1 padded) and gap
 * [n_rows][hkv] (see msa_oracle_select).
 */
static int index_core(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                      int hkv, int d_idx, int block, int topk, const index_inputs *in,
                      int n_rows, const int32_t *rows,
                      int32_t *idx, double *gap) {
  if (check_seqlens(num_seqs, cu_q, cu_k)) return ORACLE_EINVAL;
  if (hkv <= 0 || block <= 0 || topk <= 0 || !idx || n_rows < 0) return ORACLE_EINVAL;
  int max_nb = 1;
  for (int s = 0; s < num_seqs; ++s) {
    int kv_len = cu_k[s + 1] - cu_k[s];
    if (kv_len > 0) {
      int nb = msa_oracle_num_blocks(kv_len - 1, block);
      if (nb > max_nb) max_nb = nb;
    }
  }
  float *pooled = (float *)malloc(sizeof(float) * (size_t)(n_rows > 0 ? n_rows : 1) * hkv * max_nb);
  if (!pooled) return ORACLE_ENOMEM;
  int rc = pooled_core(num_seqs, cu_q, cu_k, hkv, d_idx, block, in, n_rows, rows, max_nb, pooled);
  if (rc) { free(pooled); return rc; }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(| : bad)
  for (int r = 0; r < n_rows; ++r) {
    const int i = rows ? rows[r] : r;
    const int s = seq_of_query(num_seqs, cu_q, i);
    const int pos = (cu_k[s + 1] - cu_k[s]) - (cu_q[s + 1] - cu_q[s]) + (i - cu_q[s]);
    const int nb = msa_oracle_num_blocks(pos, block);
    for (int g = 0; g < hkv; ++g)
      bad |= msa_oracle_select(nb, pooled + ((size_t)r * hkv + g) * max_nb, topk,
                               idx + ((size_t)r * hkv + g) * topk,
                               gap ? gap + (size_t)r * hkv + g : NULL) != 0;
  }
  free(pooled);
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}

int msa_oracle_index(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                     int hkv, int d_idx, int block, int topk,
                     const uint16_t *q_idx, const uint16_t *k_idx,
                     int n_rows, const int32_t *rows,
                     int32_t *idx, double *gap) {
  const index_inputs in = {q_idx, k_idx, NULL, NULL, NULL, NULL};
  return index_core(num_seqs, cu_q, cu_k, hkv, d_idx, block, topk, &in, n_rows, rows, idx, gap);
}

/*
 * Steps 1-3 chained for the query rows listed in rows (all when NULL).
 * Outputs: idx [n_rows][hkv][topk] (ascending, -1 padded), gap
 * [n_rows][hkv] (see msa_oracle_select), o [n_rows][hq][head_dim] and
 * lse [n_rows][hq] in double.
 */
int msa_oracle_forward(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                       int hq, int hkv, int head_dim, int d_idx, int block, int topk, double scale,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const uint16_t *q_idx, const uint16_t *k_idx,
                       int n_rows, const int32_t *rows,
                       int32_t *idx, double *gap, double *o, double *lse) {
  int rc = msa_oracle_index(num_seqs, cu_q, cu_k, hkv, d_idx, block, topk, q_idx, k_idx,
                            n_rows, rows, idx, gap);
  if (rc) return rc;
  return msa_oracle_attention(num_seqs, cu_q, cu_k, hq, hkv, head_dim, block, topk, scale,
                              q, k, v, idx, n_rows, rows, o, lse);
}

/*
 * fp8 K/V (the atlas record of the report, provenance of section 4.2: the
 * kernels handle fp8 as well; the pages give no format, so this follows the
 * plainest reading, stated with the build's design notes):
 *   * codes are OCP FP8 E4M3 ("E4M3FN"): sign, 4 exponent bits with bias 7,
 *     3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); no infinities;
 *     S.1111.111 is NaN; the largest finite value is 1.75 * 2^8 = 448;
 *   * one fp32 scale per (key block of 128 tokens of a sequence, KV head), for
 *     K and V separately: s = amax / 448 over the block's rows of that head
 *     (s = 1 when amax = 0), code = round-to-nearest-even(x / s) with x / s
 *     computed in fp32 and saturated to +-448;
 *   * value = decode(code) * s.
 * Scales are stored [n_key_blocks][hkv], key block b of sequence s at row
 * sum_{s' < s} ceil(kv_len_s' / block) + b.
 */

/* Value of an E4M3 code, from the definition above (NaN for the NaN codes). */
double msa_oracle_e4m3_value(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* E4M3 code of x: the nearest finite E4M3 value, ties to the even code (the
 * one whose last mantissa bit is 0), magnitudes beyond 448 saturated to 448,
 * NaN to 0x7F.  Written as a search over the ordered non-negative codes. */
uint8_t msa_oracle_e4m3_code(float x) {
  if (x != x) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int c = 0;  /* largest non-negative code whose value is <= a */
  while (c + 1 <= 0x7E && msa_oracle_e4m3_value((uint8_t)(c + 1)) <= a) ++c;
  const double lo = msa_oracle_e4m3_value((uint8_t)c);
  if (lo == a) return (uint8_t)(sign | c);
  const double hi = msa_oracle_e4m3_value((uint8_t)(c + 1));
  int pick;
  if (a - lo < hi - a) pick = c;
  else if (hi - a < a - lo) pick = c + 1;
  else pick = (c % 2 == 0) ? c : c + 1;
  return (uint8_t)(sign | pick);
}

/* Number of key blocks of all sequences (rows of a scale array). */
int msa_oracle_key_blocks(int num_seqs, const int32_t *cu_k, int block) {
  int n = 0;
  for (int s = 0; s < num_seqs; ++s) n += (cu_k[s + 1] - cu_k[s] + block - 1) / block;
  return n;
}

/*
 * Quantizes x (bf16 bits, [total_k][hkv][head_dim]) to codes (same shape) and
 * scales ([n_key_blocks][hkv]) as described above.
 */
int msa_oracle_quantize_fp8(int num_seqs, const int32_t *cu_k, int hkv, int head_dim, int block,
                            const uint16_t *x, uint8_t *codes, float *scales) {
  if (num_seqs < 0 || !cu_k || hkv <= 0 || head_dim <= 0 || block <= 0 || !x || !codes || !scales)
    return ORACLE_EINVAL;
  if (cu_k[0] != 0) return ORACLE_EINVAL;
  int row = 0;  /* scale row of the current block */
  for (int s = 0; s < num_seqs; ++s) {
    const int kv_len = cu_k[s + 1] - cu_k[s];
    if (kv_len < 0) return ORACLE_EINVAL;
    for (int b = 0; b * block < kv_len; ++b, ++row) {
      const int j0 = cu_k[s] + b * block;
      const int j1 = cu_k[s] + ((b + 1) * block < kv_len ? (b + 1) * block : kv_len);
      for (int g = 0; g < hkv; ++g) {
        float amax = 0.f;
        for (int j = j0; j < j1; ++j)
          for (int d = 0; d < head_dim; ++d) {
            const float a = (float)fabs(bf16_bits_to_double(x[((size_t)j * hkv + g) * head_dim + d]));
            if (a > amax) amax = a;
          }
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        scales[(size_t)row * hkv + g] = sc;
        for (int j = j0; j < j1; ++j)
          for (int d = 0; d < head_dim; ++d) {
            const size_t e = ((size_t)j * hkv + g) * head_dim + d;
            const float xf = (float)bf16_bits_to_double(x[e]);
            const float q = xf / sc;
            codes[e] = msa_oracle_e4m3_code(q);
          }
      }
    }
  }
  return ORACLE_OK;
}

/*
 * fp8 index (the same provenance; the pages give no format, and the report
 * warns that quantizing the index changes which blocks are selected, so this
 * is an option beside the bf16 index, not a replacement): Q_idx and K_idx as
 * E4M3 codes with the quantizer above, K_idx with one scale per key block of a
 * sequence (msa_oracle_quantize_fp8 with hkv = 1, head_dim = d_idx) and Q_idx
 * with one scale per (query row, group) (the same quantizer over the query
 * rows with block = 1: scales [total_q][hkv]).  Steps 1 and 2 then run
 * unchanged on the dequantized values.
 */
int msa_oracle_pooled_fp8(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                          int hkv, int d_idx, int block,
                          const uint8_t *q8, const float *q_scale, const uint8_t *k8, const float *k_scale,
                          int n_rows, const int32_t *rows,
                          int nb_stride, float *pooled) {
  const index_inputs in = {NULL, NULL, q8, k8, q_scale, k_scale};
  if (!q8) return ORACLE_EINVAL;
  return pooled_core(num_seqs, cu_q, cu_k, hkv, d_idx, block, &in, n_rows, rows, nb_stride, pooled);
}

int msa_oracle_index_fp8(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                         int hkv, int d_idx, int block, int topk,
                         const uint8_t *q8, const float *q_scale, const uint8_t *k8, const float *k_scale,
                         int n_rows, const int32_t *rows,
                         int32_t *idx, double *gap) {
  const index_inputs in = {NULL, NULL, q8, k8, q_scale, k_scale};
  if (!q8) return ORACLE_EINVAL;
  return index_core(num_seqs, cu_q, cu_k, hkv, d_idx, block, topk, &in, n_rows, rows, idx, gap);
}

/*
 * Step 3 with fp8 K and V: as msa_oracle_attention, every key and value
 * element read as msa_oracle_e4m3_value(code) * scale of its (key block, KV
 * head); everything in double.
 */
int msa_oracle_attention_fp8(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                             int hq, int hkv, int head_dim, int block, int topk, double scale,
                             const uint16_t *q, const uint8_t *k8, const uint8_t *v8,
                             const float *k_scale, const float *v_scale,
                             const int32_t *idx, int n_rows, const int32_t *rows,
                             double *o, double *lse) {
  if (check_seqlens(num_seqs, cu_q, cu_k)) return ORACLE_EINVAL;
  if (hq <= 0 || hkv <= 0 || hq % hkv || head_dim <= 0 || block <= 0 || topk <= 0) return ORACLE_EINVAL;
  if (!q || !k8 || !v8 || !k_scale || !v_scale || !idx || !o || !lse || n_rows < 0) return ORACLE_EINVAL;
  const int total_q = cu_q[num_seqs];
  if (!rows && n_rows != total_q) return ORACLE_EINVAL;
  const int G = hq / hkv;
  int *blk0 = (int *)malloc(sizeof(int) * (size_t)(num_seqs + 1));  /* first scale row of each sequence */
  if (!blk0) return ORACLE_ENOMEM;
  blk0[0] = 0;
  for (int s = 0; s < num_seqs; ++s) blk0[s + 1] = blk0[s] + (cu_k[s + 1] - cu_k[s] + block - 1) / block;
  int bad = 0;
#pragma omp parallel reduction(| : bad)
  {
    double *x = (double *)malloc(sizeof(double) * (size_t)topk * block);
    int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk * block);
    if (!x || !key) bad = 1;
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
      if (!x || !key) continue;
      const int i = rows ? rows[r] : r;
      const int s = (i >= 0 && i < total_q) ? seq_of_query(num_seqs, cu_q, i) : -1;
      if (s < 0) { bad = 1; continue; }
      const int q_len = cu_q[s + 1] - cu_q[s];
      const int kv_len = cu_k[s + 1] - cu_k[s];
      const int pos = kv_len - q_len + (i - cu_q[s]);
      for (int h = 0; h < hq; ++h) {
        const int g = h / G;
        const int32_t *sel = idx + ((size_t)r * hkv + g) * topk;
        int n = 0;
        for (int e = 0; e < topk; ++e) {
          const int b = sel[e];
          if (b < 0) continue;
          for (int j = b * block; j < (b + 1) * block && j <= pos; ++j) key[n++] = j;
        }
        const uint16_t *qh = q + ((size_t)i * hq + h) * head_dim;
        double *oh = o + ((size_t)r * hq + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) oh[d] = 0.0;
        if (n == 0) { lse[(size_t)r * hq + h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
          const double sk = k_scale[(size_t)(blk0[s] + key[t] / block) * hkv + g];
          const uint8_t *kj = k8 + ((size_t)(cu_k[s] + key[t]) * hkv + g) * head_dim;
          double acc = 0.0;
          for (int d = 0; d < head_dim; ++d)
            acc += bf16_bits_to_double(qh[d]) * (msa_oracle_e4m3_value(kj[d]) * sk);
          x[t] = scale * acc;
          if (x[t] > m) m = x[t];
        }
        double l = 0.0;
        for (int t = 0; t < n; ++t) {
          const double p = exp(x[t] - m);
          l += p;
          const double sv = v_scale[(size_t)(blk0[s] + key[t] / block) * hkv + g];
          const uint8_t *vj = v8 + ((size_t)(cu_k[s] + key[t]) * hkv + g) * head_dim;
          for (int d = 0; d < head_dim; ++d) oh[d] += p * (msa_oracle_e4m3_value(vj[d]) * sv);
        }
        for (int d = 0; d < head_dim; ++d) oh[d] /= l;
        lse[(size_t)r * hq + h] = m + log(l);
      }
    }
    free(x);
    free(key);
  }
  free(blk0);
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}

/*
 * Index prologue: hidden states -> index query and key heads.  "MiniMax Sparse
 * Attention: let each query pick its own blocks", Figure 1: the Index Branch
 * takes the hidden states through a linear projection, a norm and RoPE to the
 * index query and key heads.  The atlas record of the report gives d_model =
 * 3072 and a RoPE dimension of 64 on 128-dim heads (provenance of section
 * 5.1); the norm type is not given.  Reading taken here, for each new token
 * (query row i at key position pos(i)):
 *   y_h = W_q[h] x_i  (h < hkv, d_idx each),  y_k = W_k x_i   (sums in double)
 *   RMSNorm per head: z = y / sqrt(mean_d y^2 + eps) * gamma  (gamma_q shared by
 *     the index query heads, gamma_k for the key head)
 *   RoPE on dims [0, rope_dim): pairs (j, j + rope_dim/2), angle
 *     pos(i) * base^(-2j / rope_dim), (a, b) -> (a cos - b sin, b cos + a sin);
 *     dims rope_dim .. d_idx - 1 pass unchanged.
 * Outputs are the unrounded values in double: q_out [n_rows][hkv][d_idx] and
 * k_out [n_rows][d_idx] (the key row of token i is k_start + pos(i)).
 */
int msa_oracle_index_prologue(int num_seqs, const int32_t *cu_q, const int32_t *cu_k,
                              int d_model, int hkv, int d_idx, int rope_dim, double rope_base, double eps,
                              const uint16_t *x, const uint16_t *wq, const uint16_t *wk,
                              const uint16_t *gamma_q, const uint16_t *gamma_k,
                              int n_rows, const int32_t *rows, double *q_out, double *k_out) {
  if (check_seqlens(num_seqs, cu_q, cu_k)) return ORACLE_EINVAL;
  if (d_model <= 0 || hkv <= 0 || d_idx <= 0 || rope_dim < 0 || rope_dim > d_idx || rope_dim % 2 ||
      !(rope_base > 0) || !(eps >= 0) || !x || !wq || !wk || !gamma_q || !gamma_k || !q_out || !k_out ||
      n_rows < 0)
    return ORACLE_EINVAL;
  const int total_q = cu_q[num_seqs];
  if (!rows && n_rows != total_q) return ORACLE_EINVAL;
  const int half = rope_dim / 2;
  int bad = 0;
#pragma omp parallel reduction(| : bad)
  {
    double *y = (double *)malloc(sizeof(double) * (size_t)d_idx);
    if (!y) bad = 1;
#pragma omp for schedule(dynamic, 16)
    for (int r = 0; r < n_rows; ++r) {
      if (!y) continue;
      const int i = rows ? rows[r] : r;
      const int s = (i >= 0 && i < total_q) ? seq_of_query(num_seqs, cu_q, i) : -1;
      if (s < 0) { bad = 1; continue; }
      const int pos = (cu_k[s + 1] - cu_k[s]) - (cu_q[s + 1] - cu_q[s]) + (i - cu_q[s]);
      const uint16_t *xi = x + (size_t)i * d_model;
      for (int h = 0; h <= hkv; ++h) {  /* h == hkv: the key head */
        const uint16_t *w = (h < hkv) ? wq + (size_t)h * d_idx * d_model : wk;
        const uint16_t *gamma = (h < hkv) ? gamma_q : gamma_k;
        double *out = (h < hkv) ? q_out + ((size_t)r * hkv + h) * d_idx : k_out + (size_t)r * d_idx;
        /* projection */
        for (int d = 0; d < d_idx; ++d) {
          double acc = 0.0;
          for (int c = 0; c < d_model; ++c)
            acc += bf16_bits_to_double(xi[c]) * bf16_bits_to_double(w[(size_t)d * d_model + c]);
          y[d] = acc;
        }
        /* RMSNorm */
        double ss = 0.0;
        for (int d = 0; d < d_idx; ++d) ss += y[d] * y[d];
        const double inv = 1.0 / sqrt(ss / d_idx + eps);
        for (int d = 0; d < d_idx; ++d) y[d] = y[d] * inv * bf16_bits_to_double(gamma[d]);
        /* RoPE on the first rope_dim dims */
        for (int d = 0; d < d_idx; ++d) out[d] = y[d];
        for (int j = 0; j < half; ++j) {
          const double ang = (double)pos * pow(rope_base, -2.0 * j / rope_dim);
          const double c = cos(ang), sn = sin(ang);
          out[j] = y[j] * c - y[j + half] * sn;
          out[j + half] = y[j + half] * c + y[j] * sn;
        }
      }
    }
    free(y);
  }
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}
