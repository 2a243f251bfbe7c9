/*
 * attn_oracle.c -- plain fp64 CPU oracle for causal / sliding-window GQA
 * attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never links, loads or calls
 * this file.  Only the test-suite, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no source, header, table or helper with the
 * CUDA path.
 *
 * What it computes is the plain definition of masked softmax attention, not
 * the tiled online-softmax algorithm that the fused kernels use.  The online
 * recurrence (running max m, running sum l, rescale of O, store LSE = m + log l)
 * described in the Graphcore flash-attention-ipu page
 * (flash_attention_qkv_packed.cpp, forward `flashAttentionQKVPackedWithStash`)
 * and in the forge page (flash_attention.metal, header "Online softmax") is
 * algebraically the same function, so the oracle is that function written out:
 *
 *   S[i][j] = scale * sum_d Q[b,i,h,d] K[b,j,g,d]         g = h / (H/HKV)
 *   S[i][j] = -inf   where not Visible(i, j)
 *   m_i = max_j S[i][j];  l_i = sum_j exp(S - m_i);  P = exp(S - m_i) / l_i
 *   LSE_i = m_i + ln l_i;   O_i = sum_j P_ij V_j
 *
 *   Visible(i, j) <=> (!causal || j <= i) && (window == 0 || i - j < window)
 *
 * The visibility rule, the GQA head map g = h / (H/HKV), the [B,T,H,D]
 * layouts, the fp32-sized LSE in [B,H,T] and the "keys kept, self included"
 * meaning of `window` follow the forge page (flash_attention.metal: struct
 * FlashParams and kernel flash_attn_fwd).  A row with no visible key gets
 * O = 0 and LSE = 0, the guard of the same kernel's epilogue (it cannot occur
 * for self-attention, where j = i is always visible).
 *
 * Queries and keys may differ in length (Tq query rows i, Tk key rows j):
 * the teeny-kernels page (flash_attn2.rs, `flash_attention2_forward`) takes
 * separate n_ctx_q and n_ctx_k and visits every key of every query row.  The
 * visibility rule above is applied as written for any (i, j); the CUDA path
 * accepts Tq != Tk only without causal or window masking, where it is
 * unconditional.
 *
 * Backward (the analytic gradient of the definition above; the same formulas
 * appear in the Graphcore page's `flashAttentionQKVPackedGrad`, the
 * teeny-kernels page flash_attn2.rs `flash_attention2_backward_dq` /
 * `_dkv` doc comments, and FlashMetal's flashback.metal):
 *
 *   dP_ij = sum_d dO[i,d] V[j,d]
 *   Delta_i = sum_j P_ij dP_ij                  (the definition; the identity
 *                                                Delta_i = sum_d dO_i O_i is
 *                                                checked by the tests)
 *   dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_{h in group g} sum_i dS_ij Q_i
 *   dV_j  =         sum_{h in group g} sum_i P_ij dO_i
 *
 * All arithmetic is IEEE double, each sum taken in index order by one thread.
 * OpenMP only spreads independent rows / columns over cores.
 *
 * Layouts (row-major, contiguous):
 *   Q, O, dO, dQ : [B, Tq, H,   D]
 *   K, V, dK, dV : [B, Tk, HKV, D]
 *   LSE, Delta   : [B, H, Tq]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

typedef struct {
  int B, T, H, HKV, D; /* T: query rows */
  double scale;
  int causal, window;
  int Tk; /* key rows */
} shape_t;

static int visible(const shape_t* s, long i, long j) {
  if (s->causal && j > i) return 0;
  if (s->window > 0 && i - j >= s->window) return 0;
  return 1;
}

static size_t q_index(const shape_t* s, long b, long t, long h) {
  return (((size_t)b * s->T + t) * s->H + h) * s->D;
}

static size_t kv_index(const shape_t* s, long b, long t, long g) {
  return (((size_t)b * s->Tk + t) * s->HKV + g) * s->D;
}

static size_t row_index(const shape_t* s, long b, long h, long t) {
  return ((size_t)b * s->H + h) * s->T + t;
}

static int check_shape(const shape_t* s) {
  if (s->B < 1 || s->T < 1 || s->Tk < 1 || s->H < 1 || s->HKV < 1 || s->D < 1) return 0;
  if (s->H % s->HKV != 0) return 0;
  if (s->window < 0) return 0;
  return 1;
}

static double dot(const double* a, const double* b, int n) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) acc += a[d] * b[d];
  return acc;
}

/* One row of masked scores: S_row[j] = scale * Q_i . K_j, or -inf. */
static void score_row(const shape_t* s, const double* Q, const double* K,
                      long b, long h, long i, double* S_row) {
  const long g = h / (s->H / s->HKV);
  const double* qi = Q + q_index(s, b, i, h);
  for (long j = 0; j < s->Tk; ++j) {
    if (visible(s, i, j))
      S_row[j] = s->scale * dot(qi, K + kv_index(s, b, j, g), s->D);
    else
      S_row[j] = -INFINITY;
  }
}

/*
 * Three-pass softmax of one score row of n keys, in place: S_row becomes P_row.
 * Returns LSE = m + ln l, or 0 for a row with no visible key (then P_row = 0).
 */
static double softmax_row(double* S_row, long n) {
  double m = -INFINITY;
  for (long j = 0; j < n; ++j)
    if (S_row[j] > m) m = S_row[j];
  if (m == -INFINITY) {
    for (long j = 0; j < n; ++j) S_row[j] = 0.0;
    return 0.0;
  }
  double l = 0.0;
  for (long j = 0; j < n; ++j) l += exp(S_row[j] - m);
  for (long j = 0; j < n; ++j) S_row[j] = exp(S_row[j] - m) / l;
  return m + log(l);
}

/* dP_row[j] = dO_i . V_j on visible (i, j), 0 elsewhere. */
static void dp_row(const shape_t* s, const double* V, const double* dO,
                   long b, long h, long i, double* dP_row) {
  const long g = h / (s->H / s->HKV);
  const double* doi = dO + q_index(s, b, i, h);
  for (long j = 0; j < s->Tk; ++j)
    dP_row[j] = visible(s, i, j) ? dot(doi, V + kv_index(s, b, j, g), s->D) : 0.0;
}

/* ------------------------------------------------------------------ forward */

/*
 * Full probability matrix of one (b, h): P[i*Tk + j].  Also LSE_head[i] if
 * not NULL.  This is the unfused Tq x Tk matrix the flash method avoids; the
 * oracle materialises it on purpose.
 */
int oracle_attn_probs(const double* Q, const double* K,
                      int B, int T, int Tk, int H, int HKV, int D,
                      double scale, int causal, int window,
                      int b, int h, double* P, double* LSE_head) {
  shape_t s = {B, T, H, HKV, D, scale, causal, window, Tk};
  if (!check_shape(&s) || b < 0 || b >= B || h < 0 || h >= H) return ORACLE_EINVAL;
#pragma omp parallel for schedule(dynamic, 16)
  for (long i = 0; i < T; ++i) {
    double* row = P + (size_t)i * Tk;
    score_row(&s, Q, K, b, h, i, row);
    const double lse = softmax_row(row, Tk);
    if (LSE_head) LSE_head[i] = lse;
  }
  return ORACLE_OK;
}

/* O = P V and LSE for every (b, h), one head's Tq x Tk matrix at a time. */
int oracle_attn_fwd(const double* Q, const double* K, const double* V,
                    int B, int T, int Tk, int H, int HKV, int D,
                    double scale, int causal, int window,
                    double* O, double* LSE) {
  shape_t s = {B, T, H, HKV, D, scale, causal, window, Tk};
  if (!check_shape(&s)) return ORACLE_EINVAL;
  double* P = (double*)malloc(sizeof(double) * (size_t)T * Tk);
  if (!P) return ORACLE_ENOMEM;
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < H; ++h) {
      const long g = h / (H / HKV);
      oracle_attn_probs(Q, K, B, T, Tk, H, HKV, D, scale, causal, window, b, h, P,
                        LSE + row_index(&s, b, h, 0));
#pragma omp parallel for schedule(dynamic, 16)
      for (long i = 0; i < T; ++i) {
        double* oi = O + q_index(&s, b, i, h);
        for (int d = 0; d < D; ++d) oi[d] = 0.0;
        for (long j = 0; j < Tk; ++j) {
          const double p = P[(size_t)i * Tk + j];
          if (p == 0.0) continue;
          const double* vj = V + kv_index(&s, b, j, g);
          for (int d = 0; d < D; ++d) oi[d] += p * vj[d];
        }
      }
    }
  }
  free(P);
  return ORACLE_OK;
}

/* ----------------------------------------------------------------- backward */

/*
 * dQ, dK, dV (and Delta, if not NULL) for every (b, h).  Per KV head g the
 * rep query heads of its group are visited in order and their dK / dV
 * contributions summed.  Materialises P and dS (Tq x Tk each) per head.
 */
int oracle_attn_bwd(const double* Q, const double* K, const double* V,
                    const double* dO,
                    int B, int T, int Tk, int H, int HKV, int D,
                    double scale, int causal, int window,
                    double* dQ, double* dK, double* dV, double* Delta) {
  shape_t s = {B, T, H, HKV, D, scale, causal, window, Tk};
  if (!check_shape(&s)) return ORACLE_EINVAL;
  const int rep = H / HKV;
  double* P = (double*)malloc(sizeof(double) * (size_t)T * Tk);
  double* dS = (double*)malloc(sizeof(double) * (size_t)T * Tk);
  if (!P || !dS) {
    free(P);
    free(dS);
    return ORACLE_ENOMEM;
  }
  for (int b = 0; b < B; ++b) {
    for (int g = 0; g < HKV; ++g) {
      for (long j = 0; j < Tk; ++j) {
        memset(dK + kv_index(&s, b, j, g), 0, sizeof(double) * D);
        memset(dV + kv_index(&s, b, j, g), 0, sizeof(double) * D);
      }
      for (int r = 0; r < rep; ++r) {
        const int h = g * rep + r;
        oracle_attn_probs(Q, K, B, T, Tk, H, HKV, D, scale, causal, window, b, h, P, NULL);
        /* rows: dP, Delta, dS, dQ */
#pragma omp parallel for schedule(dynamic, 16)
        for (long i = 0; i < T; ++i) {
          const double* Pi = P + (size_t)i * Tk;
          double* dSi = dS + (size_t)i * Tk;
          dp_row(&s, V, dO, b, h, i, dSi); /* dSi holds dP_i for now */
          double delta = 0.0;
          for (long j = 0; j < Tk; ++j) delta += Pi[j] * dSi[j];
          if (Delta) Delta[row_index(&s, b, h, i)] = delta;
          for (long j = 0; j < Tk; ++j) dSi[j] = Pi[j] * (dSi[j] - delta);
          double* dqi = dQ + q_index(&s, b, i, h);
          for (int d = 0; d < D; ++d) dqi[d] = 0.0;
          for (long j = 0; j < Tk; ++j) {
            if (dSi[j] == 0.0) continue;
            const double* kj = K + kv_index(&s, b, j, g);
            for (int d = 0; d < D; ++d) dqi[d] += dSi[j] * kj[d];
          }
          for (int d = 0; d < D; ++d) dqi[d] *= scale;
        }
        /* columns: dK_j += scale * dS^T Q, dV_j += P^T dO (one thread per j) */
#pragma omp parallel for schedule(dynamic, 16)
        for (long j = 0; j < Tk; ++j) {
          double* dkj = dK + kv_index(&s, b, j, g);
          double* dvj = dV + kv_index(&s, b, j, g);
          for (long i = 0; i < T; ++i) {
            const double p = P[(size_t)i * Tk + j];
            const double ds = dS[(size_t)i * Tk + j];
            const double* qi = Q + q_index(&s, b, i, h);
            const double* doi = dO + q_index(&s, b, i, h);
            if (ds != 0.0)
              for (int d = 0; d < D; ++d) dkj[d] += scale * ds * qi[d];
            if (p != 0.0)
              for (int d = 0; d < D; ++d) dvj[d] += p * doi[d];
          }
        }
      }
    }
  }
  free(P);
  free(dS);
  return ORACLE_OK;
}

/* ------------------------------------------- sampled rows (full-size checks) */

/*
 * O and LSE of selected query rows of one (b, h): O_rows[n*D + d], LSE_rows[n].
 * Same definition as oracle_attn_fwd, evaluated only on the listed rows, so
 * that outputs of a large problem can be checked one by one.
 */
int oracle_attn_fwd_rows(const double* Q, const double* K, const double* V,
                         int B, int T, int Tk, int H, int HKV, int D,
                         double scale, int causal, int window,
                         int b, int h, const int* rows, int nrows,
                         double* O_rows, double* LSE_rows) {
  shape_t s = {B, T, H, HKV, D, scale, causal, window, Tk};
  if (!check_shape(&s) || b < 0 || b >= B || h < 0 || h >= H) return ORACLE_EINVAL;
  for (int n = 0; n < nrows; ++n)
    if (rows[n] < 0 || rows[n] >= T) return ORACLE_EINVAL;
  const long g = h / (H / HKV);
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double* P = (double*)malloc(sizeof(double) * (size_t)Tk);
    if (!P) {
#pragma omp atomic write
      status = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int n = 0; n < nrows; ++n) {
        const long i = rows[n];
        score_row(&s, Q, K, b, h, i, P);
        LSE_rows[n] = softmax_row(P, Tk);
        double* oi = O_rows + (size_t)n * D;
        for (int d = 0; d < D; ++d) oi[d] = 0.0;
        for (long j = 0; j < Tk; ++j) {
          if (P[j] == 0.0) continue;
          const double* vj = V + kv_index(&s, b, j, g);
          for (int d = 0; d < D; ++d) oi[d] += P[j] * vj[d];
        }
      }
      free(P);
    }
  }
  return status;
}

/* dQ (and Delta) of selected query rows of one (b, h). */
int oracle_attn_dq_rows(const double* Q, const double* K, const double* V,
                        const double* dO,
                        int B, int T, int Tk, int H, int HKV, int D,
                        double scale, int causal, int window,
                        int b, int h, const int* rows, int nrows,
                        double* dQ_rows, double* Delta_rows) {
  shape_t s = {B, T, H, HKV, D, scale, causal, window, Tk};
  if (!check_shape(&s) || b < 0 || b >= B || h < 0 || h >= H) return ORACLE_EINVAL;
  for (int n = 0; n < nrows; ++n)
    if (rows[n] < 0 || rows[n] >= T) return ORACLE_EINVAL;
  const long g = h / (H / HKV);
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double* P = (double*)malloc(sizeof(double) * (size_t)Tk);
    double* dP = (double*)malloc(sizeof(double) * (size_t)Tk);
    if (!P || !dP) {
#pragma omp atomic write
      status = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int n = 0; n < nrows; ++n) {
        const long i = rows[n];
        score_row(&s, Q, K, b, h, i, P);
        softmax_row(P, Tk);
        dp_row(&s, V, dO, b, h, i, dP);
        double delta = 0.0;
        for (long j = 0; j < Tk; ++j) delta += P[j] * dP[j];
        if (Delta_rows) Delta_rows[n] = delta;
        double* dqi = dQ_rows + (size_t)n * D;
        for (int d = 0; d < D; ++d) dqi[d] = 0.0;
        for (long j = 0; j < Tk; ++j) {
          const double ds = P[j] * (dP[j] - delta);
          if (ds == 0.0) continue;
          const double* kj = K + kv_index(&s, b, j, g);
          for (int d = 0; d < D; ++d) dqi[d] += ds * kj[d];
        }
        for (int d = 0; d < D; ++d) dqi[d] *= scale;
      }
    }
    free(P);
    free(dP);
  }
  return status;
}

/*
 * dK and dV of selected key rows j of one (b, g).  Every query row i of every
 * head of the group that sees any selected j is evaluated in full (its P_i,
 * dP_i and Delta_i), and its contribution added to the selected rows.
 */
int oracle_attn_dkdv_rows(const double* Q, const double* K, const double* V,
                          const double* dO,
                          int B, int T, int Tk, int H, int HKV, int D,
                          double scale, int causal, int window,
                          int b, int g, const int* cols, int ncols,
                          double* dK_rows, double* dV_rows) {
  shape_t s = {B, T, H, HKV, D, scale, causal, window, Tk};
  if (!check_shape(&s) || b < 0 || b >= B || g < 0 || g >= HKV) return ORACLE_EINVAL;
  for (int n = 0; n < ncols; ++n)
    if (cols[n] < 0 || cols[n] >= Tk) return ORACLE_EINVAL;
  const int rep = H / HKV;
  memset(dK_rows, 0, sizeof(double) * (size_t)ncols * D);
  memset(dV_rows, 0, sizeof(double) * (size_t)ncols * D);
  /* which query rows see at least one selected key */
  char* need = (char*)calloc((size_t)T, 1);
  if (!need) return ORACLE_ENOMEM;
  for (int n = 0; n < ncols; ++n)
    for (long i = 0; i < T; ++i)
      if (visible(&s, i, cols[n])) need[i] = 1;
  int status = ORACLE_OK;
  /* Parallel over selected columns would re-evaluate rows; instead evaluate
     each needed row once per head (in parallel) and store its P / dS values
     at the selected columns, then reduce in row order per column. */
  double* Psel = (double*)malloc(sizeof(double) * (size_t)T * ncols);
  double* dSsel = (double*)malloc(sizeof(double) * (size_t)T * ncols);
  if (!Psel || !dSsel) {
    free(need);
    free(Psel);
    free(dSsel);
    return ORACLE_ENOMEM;
  }
  for (int r = 0; r < rep; ++r) {
    const int h = g * rep + r;
#pragma omp parallel
    {
      double* P = (double*)malloc(sizeof(double) * (size_t)Tk);
      double* dP = (double*)malloc(sizeof(double) * (size_t)Tk);
      if (!P || !dP) {
#pragma omp atomic write
        status = ORACLE_ENOMEM;
      } else {
#pragma omp for schedule(dynamic, 1)
        for (long i = 0; i < T; ++i) {
          if (!need[i]) continue;
          score_row(&s, Q, K, b, h, i, P);
          softmax_row(P, Tk);
          dp_row(&s, V, dO, b, h, i, dP);
          double delta = 0.0;
          for (long j = 0; j < Tk; ++j) delta += P[j] * dP[j];
          for (int n = 0; n < ncols; ++n) {
            const long j = cols[n];
            Psel[(size_t)i * ncols + n] = P[j];
            dSsel[(size_t)i * ncols + n] = P[j] * (dP[j] - delta);
          }
        }
      }
      free(P);
      free(dP);
    }
    if (status != ORACLE_OK) break;
#pragma omp parallel for schedule(dynamic, 1)
    for (int n = 0; n < ncols; ++n) {
      double* dkj = dK_rows + (size_t)n * D;
      double* dvj = dV_rows + (size_t)n * D;
      for (long i = 0; i < T; ++i) {
        if (!need[i]) continue;
        const double p = Psel[(size_t)i * ncols + n];
        const double ds = dSsel[(size_t)i * ncols + n];
        const double* qi = Q + q_index(&s, b, i, h);
        const double* doi = dO + q_index(&s, b, i, h);
        if (ds != 0.0)
          for (int d = 0; d < D; ++d) dkj[d] += scale * ds * qi[d];
        if (p != 0.0)
          for (int d = 0; d < D; ++d) dvj[d] += p * doi[d];
      }
    }
  }
  free(need);
  free(Psel);
  free(dSsel);
  return status;
}

/* ------------------------------------------------ block-offset (triu) scheme */

/*
 * The Graphcore page (flash_attention_qkv_packed.cpp, getTriuOffsetSequence
 * and its docstring examples) splits the causal mask into blocks of
 * numRows x numCols and keeps only the distinct diagonal-crossing blocks.
 * Block (i, j) crosses the diagonal with offset k = i*numRows - j*numCols + 1:
 * inside it, element (r, c) is masked iff c - r >= k.  The page walks these
 * offsets starting from 1: each step down one block row adds numRows; when the
 * offset passes numCols - 1 the walk moves one block column right, subtracting
 * numRows + numCols; offsets below 2 - numRows (blocks the diagonal misses,
 * which need no mask) are skipped, and the walk stops when it returns to 1.
 *
 * Writes at most `cap` offsets into `out` and returns how many the walk
 * produced (which may exceed cap), or -1 for invalid sizes.
 */
int oracle_triu_offsets(int numRows, int numCols, int* out, int cap) {
  if (numRows < 1 || numCols < 1) return -1;
  int count = 0;
  int k = 1;
  const long guard = 4L * (numRows + numCols) * (numRows + numCols) + 16;
  long steps = 0;
  if (count < cap) out[count] = k;
  ++count;
  for (;;) {
    k += numRows;
    if (k > numCols - 1) k -= numRows + numCols;
    if (k == 1) break;
    if (k >= 2 - numRows) {
      if (count < cap) out[count] = k;
      ++count;
    }
    if (++steps > guard) return -1; /* the walk always returns to 1; defensive */
  }
  return count;
}

/* ------------------------------------------------------------------------
 * Pre-attention prologue: RMS-norm of every query and key head vector, then
 * the rotary mix with per-position factors, as the modded-nanogpt page
 * qkv_rope.py defines it (module docstring and `_qk_norm_rope_forward_kernel`,
 * read without its "paired heads" and "key offset" options; the fp8 packing
 * of its backward kernel is left out).  Input: the packed projection
 * qk[t][c][d], t < tokens, heads c < hq are queries and hq <= c < hq + hk are
 * keys, d < D (D even); factors f1[t][d], f2[t][d].
 *
 *   ms   = (1/D) sum_d x_d^2 ;  rstd = 1 / sqrt(ms + eps),  eps = 2^-23
 *   n_d  = rstd x_d
 *   y_d  = f1[t][d] n_d + f2[t][d] n_{d xor 1}      (partner: the other lane
 *                                                     of the pair (2i, 2i+1))
 *
 * Queries go to q[t][c][d], keys to k[t][c - hq][d].  The backward takes the
 * gradients g of q and k and returns the gradient of qk: by the chain rule
 * through y (dL/dn_e = f1_e g_e + f2_{e xor 1} g_{e xor 1}) and through the
 * RMS-norm,
 *
 *   gn_e = f1[t][e] g_e + f2[t][e xor 1] g_{e xor 1}
 *   dx_e = rstd (gn_e - n_e (1/D) sum_d gn_d n_d)
 * ------------------------------------------------------------------------ */
static const double kQkEps = 1.1920928955078125e-7;

static double qk_rstd(const double* x, int D) {
  double ms = 0.0;
  for (int d = 0; d < D; ++d) ms += x[d] * x[d];
  ms /= D;
  return 1.0 / sqrt(ms + kQkEps);
}

int oracle_qk_norm_rope_fwd(const double* qk, const double* f1, const double* f2, double* q, double* k,
                            int tokens, int hq, int hk, int D) {
  if (tokens < 1 || hq < 1 || hk < 1 || D < 2 || D % 2) return 1;
  const int heads = hq + hk;
#pragma omp parallel for schedule(static)
  for (long t = 0; t < tokens; ++t) {
    for (int c = 0; c < heads; ++c) {
      const double* x = qk + ((size_t)t * heads + c) * D;
      double* y = c < hq ? q + ((size_t)t * hq + c) * D : k + ((size_t)t * hk + (c - hq)) * D;
      const double rstd = qk_rstd(x, D);
      for (int d = 0; d < D; ++d)
        y[d] = f1[(size_t)t * D + d] * (x[d] * rstd) + f2[(size_t)t * D + d] * (x[d ^ 1] * rstd);
    }
  }
  return 0;
}

int oracle_qk_norm_rope_bwd(const double* dq, const double* dk, const double* qk, const double* f1,
                            const double* f2, double* dqk, int tokens, int hq, int hk, int D) {
  if (tokens < 1 || hq < 1 || hk < 1 || D < 2 || D % 2) return 1;
  const int heads = hq + hk;
#pragma omp parallel for schedule(static)
  for (long t = 0; t < tokens; ++t) {
    double* gn = (double*)malloc(sizeof(double) * (size_t)D);
    for (int c = 0; c < heads; ++c) {
      const double* x = qk + ((size_t)t * heads + c) * D;
      const double* g = c < hq ? dq + ((size_t)t * hq + c) * D : dk + ((size_t)t * hk + (c - hq)) * D;
      double* dx = dqk + ((size_t)t * heads + c) * D;
      const double rstd = qk_rstd(x, D);
      double corr = 0.0;
      for (int e = 0; e < D; ++e) {
        gn[e] = f1[(size_t)t * D + e] * g[e] + f2[(size_t)t * D + (e ^ 1)] * g[e ^ 1];
        corr += gn[e] * (x[e] * rstd);
      }
      corr /= D;
      for (int e = 0; e < D; ++e) dx[e] = rstd * (gn[e] - (x[e] * rstd) * corr);
    }
    free(gn);
  }
  return 0;
}

/* --------------------------------------------------------------------------
 * Prologue options: paired heads and key offset (the same page's
 * `_qk_norm_rope_forward_kernel`, PAIRED and KEY_OFFSET branches, and the
 * norm/rotary part of `_qkv_norm_rope_pack_fp8_backward_kernel`).  Here the
 * projection has equally many query and key heads: qk[t][c][d] with
 * c < heads a query head and heads <= c < 2*heads a key head, logical head
 * h = c mod heads.  The two options are not combined (the page asserts so).
 *
 * Paired heads (heads even): factor rows are 2*D wide, head h rotates with
 * half (h mod 2) of its token's row, and the output of (t, h) goes to output
 * token 2t + h div (heads/2), output head h mod (heads/2); q and k are then
 * [2*tokens][heads/2][D].
 *
 * Key offset (rot even, 0 <= rot <= D): for a key head of token t > 0 the
 * stationary dims d >= rot of the output are the previous token's
 * normalised values of the same head, unrotated:  y_d = rstd' x'_d  with x'
 * = qk[t-1][c].  Token 0 and all query heads are unchanged.
 *
 * Backward: the exact gradient of this forward.  With key offset, n_e of a
 * key row at a stationary dim e >= rot reaches only the next token's output
 * (and, for token 0, its own rotated output), so
 *   gn_e = [t == 0] (f1_e g_e + f2_{e^1} g_{e^1}) + [t + 1 < tokens] g'_e
 * with g' the gradient of token t+1's key output; the page's kernel writes
 * g_e instead of the bracketed rotation term, which is the same value when
 * the stationary dims' factors are the identity (f1 = 1, f2 = 0).
 * ------------------------------------------------------------------------ */

static size_t qk_out_index(int t, int h, int heads, int D, int paired) {
  if (paired) {
    const int half = heads / 2;
    return ((size_t)(2 * t + h / half) * half + (h % half)) * D;
  }
  return ((size_t)t * heads + h) * D;
}

int oracle_qk_norm_rope_fwd_opt(const double* qk, const double* f1, const double* f2, double* q, double* k,
                                int tokens, int heads, int D, int rot, int paired, int key_offset) {
  if (tokens < 1 || heads < 1 || D < 2 || D % 2 || (paired && key_offset)) return 1;
  if (paired && heads % 2) return 1;
  if (key_offset && (rot < 0 || rot > D || rot % 2)) return 1;
  const int F = paired ? 2 * D : D;
#pragma omp parallel for schedule(static)
  for (long t = 0; t < tokens; ++t) {
    for (int c = 0; c < 2 * heads; ++c) {
      const int h = c % heads;
      const int is_key = c >= heads;
      const double* x = qk + ((size_t)t * 2 * heads + c) * D;
      const double rstd = qk_rstd(x, D);
      const double* a = f1 + (size_t)t * F + (paired ? (h % 2) * D : 0);
      const double* b = f2 + (size_t)t * F + (paired ? (h % 2) * D : 0);
      double* y = (is_key ? k : q) + qk_out_index((int)t, h, heads, D, paired);
      for (int d = 0; d < D; ++d) y[d] = a[d] * (x[d] * rstd) + b[d] * (x[d ^ 1] * rstd);
      if (key_offset && is_key && t > 0) {
        const double* xp = qk + ((size_t)(t - 1) * 2 * heads + c) * D;
        const double rp = qk_rstd(xp, D);
        for (int d = rot; d < D; ++d) y[d] = xp[d] * rp;
      }
    }
  }
  return 0;
}

int oracle_qk_norm_rope_bwd_opt(const double* dq, const double* dk, const double* qk, const double* f1,
                                const double* f2, double* dqk, int tokens, int heads, int D, int rot, int paired,
                                int key_offset) {
  if (tokens < 1 || heads < 1 || D < 2 || D % 2 || (paired && key_offset)) return 1;
  if (paired && heads % 2) return 1;
  if (key_offset && (rot < 0 || rot > D || rot % 2)) return 1;
  const int F = paired ? 2 * D : D;
  int status = 0;
#pragma omp parallel
  {
    double* gn = (double*)malloc(sizeof(double) * (size_t)D);
    if (!gn) {
#pragma omp atomic write
      status = 2;
    } else {
#pragma omp for schedule(static)
      for (long t = 0; t < tokens; ++t) {
        for (int c = 0; c < 2 * heads; ++c) {
          const int h = c % heads;
          const int is_key = c >= heads;
          const double* x = qk + ((size_t)t * 2 * heads + c) * D;
          const double* g = (is_key ? dk : dq) + qk_out_index((int)t, h, heads, D, paired);
          const double* a = f1 + (size_t)t * F + (paired ? (h % 2) * D : 0);
          const double* b = f2 + (size_t)t * F + (paired ? (h % 2) * D : 0);
          const int shifted = key_offset && is_key;
          for (int e = 0; e < D; ++e) {
            const int own = !shifted || t == 0 || e < rot;  /* does this row's own output use n_e? */
            gn[e] = own ? a[e] * g[e] + b[e ^ 1] * g[e ^ 1] : 0.0;
            if (shifted && e >= rot && t + 1 < tokens)
              gn[e] += dk[qk_out_index((int)t + 1, h, heads, D, paired) + e];
          }
          const double rstd = qk_rstd(x, D);
          double corr = 0.0;
          for (int e = 0; e < D; ++e) corr += gn[e] * (x[e] * rstd);
          corr /= D;
          double* dx = dqk + ((size_t)t * 2 * heads + c) * D;
          for (int e = 0; e < D; ++e) dx[e] = rstd * (gn[e] - (x[e] * rstd) * corr);
        }
      }
      free(gn);
    }
  }
  return status;
}
