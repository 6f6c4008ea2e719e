/*
 * oracle.c -- plain fp64 CPU attention: the reference the CUDA kernels are
 * checked against.  TEST INFRASTRUCTURE ONLY: nothing on the product path
 * loads or calls this library; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg do.
 *
 * What it computes (scaled dot-product attention, "Fused Kernel Compiler"
 * page, subsection FlashAttention Integration, equation
 * Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V):
 *
 *   s_ij  = scale * <q_i, k_j>                       (full score row, fp64)
 *   s_ij  = -inf where the causal mask hides key j   (j > i + Nk - Nq)
 *   m_i   = max_j s_ij                               (pass 1)
 *   l_i   = sum_j exp(s_ij - m_i)                    (pass 2)
 *   o_i   = sum_j exp(s_ij - m_i) v_j / l_i
 *   lse_i = m_i + log(l_i)                           (natural log)
 *
 * This is the "direct implementation" that writes every score before the
 * softmax ("Kernel Fusion, Softmax, and Attention" page, attention
 * paragraph): the score row of each query is materialised in full, and the
 * softmax is the two-pass safe form, with no running (online) update.  The
 * fused kernels reach the same numbers up to rounding order.
 *
 * Readings where the pages are silent:
 *   - causal mask aligned bottom-right: query i sees keys j <= i + Nk - Nq;
 *   - a query that sees no key gets o = 0 and lse = -inf;
 *   - lse uses the natural logarithm;
 *   - layouts: q,k,v,out [B, H, N, d] row-major; GQA maps query head hq to
 *     key/value head hq / (Hq / Hkv);
 *   - paged cache [num_blocks, Hkv, block_size, d]; logical token t of
 *     sequence s lives in physical block block_table[s][t / block_size],
 *     slot t % block_size ("Optimizing LLM Inference ..." page, section
 *     Paged Attention and Dynamic KV Cache Management); ctx_len counts the
 *     current token, which is already in the cache.
 *
 * Inputs are bf16 bit patterns (uint16), widened exactly to fp64.
 *
 * Also here: the residual add + RMS normalisation that sits next to
 * attention in every layer (oracle_add_rms_norm_f64, at the end).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t h) {
  union {
    uint32_t u;
    float f;
  } c;
  c.u = ((uint32_t)h) << 16;
  return (double)c.f;
}

/* One query row against n_keys keys whose rows are reached through
 * krow(j) / vrow(j) pointers.  Keys j >= n_visible are masked (-inf).
 * `s` is scratch of n_keys doubles; `qd` the query row in fp64. */
static void attend_row(const double* qd, const uint16_t* const* krows,
                       const uint16_t* const* vrows, long n_keys, long n_visible, int d,
                       double scale, double* s, double* o, double* lse) {
  long j;
  int t;
  /* full score row */
  for (j = 0; j < n_keys; ++j) {
    if (j >= n_visible) {
      s[j] = -INFINITY;
      continue;
    }
    double acc = 0.0;
    const uint16_t* kr = krows[j];
    for (t = 0; t < d; ++t) acc += qd[t] * bf16_to_f64(kr[t]);
    s[j] = scale * acc;
  }
  /* pass 1: row maximum */
  double m = -INFINITY;
  for (j = 0; j < n_keys; ++j)
    if (s[j] > m) m = s[j];
  for (t = 0; t < d; ++t) o[t] = 0.0;
  if (m == -INFINITY) { /* no visible key */
    *lse = -INFINITY;
    return;
  }
  /* pass 2: normaliser and weighted sum of values */
  double l = 0.0;
  for (j = 0; j < n_keys; ++j) {
    if (s[j] == -INFINITY) continue;
    double p = exp(s[j] - m);
    l += p;
    const uint16_t* vr = vrows[j];
    for (t = 0; t < d; ++t) o[t] += p * bf16_to_f64(vr[t]);
  }
  for (t = 0; t < d; ++t) o[t] /= l;
  *lse = m + log(l);
}

/* Number of keys query row i may see under the mask. */
static long visible_keys(long i, long Nq, long Nk, int causal) {
  if (!causal) return Nk;
  long lim = i + (Nk - Nq) + 1;
  if (lim < 0) lim = 0;
  if (lim > Nk) lim = Nk;
  return lim;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Attention for a list of query rows.  rows[3*r + {0,1,2}] = (b, hq, i).
 * out: [n_rows, d] fp64, lse: [n_rows] fp64.  Returns 0, or -1 on bad
 * arguments / allocation failure. */
int oracle_attn_rows_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int64_t* rows, long n_rows, int B, int Hq, int Hkv, long Nq,
                         long Nk, int d, double scale, int causal, double* out, double* lse) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || d < 1) return -1;
  const int group = Hq / Hkv;
  int bad = 0;
  long r;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)d);
    const uint16_t** kp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(Nk > 0 ? Nk : 1));
    const uint16_t** vp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(Nk > 0 ? Nk : 1));
    if (!s || !qd || !kp || !vp) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (r = 0; r < n_rows; ++r) {
        const long b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Nq) {
#pragma omp atomic write
          bad = 1;
          continue;
        }
        const long kvh = h / group;
        const uint16_t* qr = q + ((b * Hq + h) * Nq + i) * (long)d;
        const uint16_t* kb = k + (b * Hkv + kvh) * Nk * (long)d;
        const uint16_t* vb = v + (b * Hkv + kvh) * Nk * (long)d;
        int t;
        long j;
        for (t = 0; t < d; ++t) qd[t] = bf16_to_f64(qr[t]);
        for (j = 0; j < Nk; ++j) {
          kp[j] = kb + j * d;
          vp[j] = vb + j * d;
        }
        attend_row(qd, kp, vp, Nk, visible_keys(i, Nq, Nk, causal), d, scale, s, out + r * d,
                   lse + r);
      }
    }
    free(s);
    free(qd);
    free(kp);
    free(vp);
  }
  return bad ? -1 : 0;
}

/* Full prefill attention: out [B, Hq, Nq, d] fp64, lse [B, Hq, Nq] fp64. */
int oracle_attn_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Hq,
                    int Hkv, long Nq, long Nk, int d, double scale, int causal, double* out,
                    double* lse) {
  const long n_rows = (long)B * Hq * Nq;
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * 3 * (size_t)(n_rows > 0 ? n_rows : 1));
  if (!rows) return -1;
  long r = 0;
  for (long b = 0; b < B; ++b)
    for (long h = 0; h < Hq; ++h)
      for (long i = 0; i < Nq; ++i, ++r) {
        rows[3 * r] = b;
        rows[3 * r + 1] = h;
        rows[3 * r + 2] = i;
      }
  int rc = oracle_attn_rows_f64(q, k, v, rows, n_rows, B, Hq, Hkv, Nq, Nk, d, scale, causal,
                                out, lse);
  free(rows);
  return rc;
}

/* One-token decode over a block-paged cache.  q, out: [num_seqs, Hq, d];
 * lse: [num_seqs, Hq].  Every cached token t < ctx_lens[s] is visible. */
int oracle_decode_paged_f64(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* block_table, const int32_t* ctx_lens, int num_seqs,
                            int Hq, int Hkv, int d, int block_size, long num_blocks,
                            int max_blocks_per_seq, double scale, double* out, double* lse) {
  if (num_seqs < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || block_size < 1) return -1;
  const int group = Hq / Hkv;
  long max_ctx = (long)max_blocks_per_seq * block_size;
  int bad = 0;
  long w;
  const long n_work = (long)num_seqs * Hq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)d);
    const uint16_t** kp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    const uint16_t** vp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!s || !qd || !kp || !vp) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (w = 0; w < n_work; ++w) {
        const long sq = w / Hq, h = w % Hq, kvh = h / group;
        const long n = ctx_lens[sq];
        if (n < 0 || n > max_ctx) {
#pragma omp atomic write
          bad = 1;
          continue;
        }
        long t;
        int c;
        int fault = 0;
        for (t = 0; t < n; ++t) {
          const long phys = block_table[sq * (long)max_blocks_per_seq + t / block_size];
          if (phys < 0 || phys >= num_blocks) {
            fault = 1;
            break;
          }
          const long off = ((phys * Hkv + kvh) * block_size + t % block_size) * (long)d;
          kp[t] = k_cache + off;
          vp[t] = v_cache + off;
        }
        if (fault) {
#pragma omp atomic write
          bad = 1;
          continue;
        }
        const uint16_t* qr = q + (sq * Hq + h) * (long)d;
        for (c = 0; c < d; ++c) qd[c] = bf16_to_f64(qr[c]);
        attend_row(qd, kp, vp, n, n, d, scale, s, out + w * d, lse + w);
      }
    }
    free(s);
    free(qd);
    free(kp);
    free(vp);
  }
  return bad ? -1 : 0;
}

/* Two-pass safe softmax of one row (the form the oracle uses). */
void oracle_softmax_f64(const double* x, long n, double* y) {
  double m = -INFINITY, l = 0.0;
  long j;
  for (j = 0; j < n; ++j)
    if (x[j] > m) m = x[j];
  for (j = 0; j < n; ++j) l += exp(x[j] - m);
  for (j = 0; j < n; ++j) y[j] = exp(x[j] - m) / l;
}

/* Running (online) softmax of one row, the single-sweep recurrence of
 * Milakov & Gimelshein (cited on the "Fused Kernel Compiler" page,
 * FlashAttention Integration, item 3): keep the running maximum m_j and the
 * running normaliser d_j = d_{j-1} * exp(m_{j-1} - m_j) + exp(x_j - m_j);
 * then y_i = exp(x_i - m_n) / d_n.  Used only to pin the two-pass form. */
void oracle_online_softmax_f64(const double* x, long n, double* y) {
  double m = -INFINITY, dsum = 0.0;
  long j;
  for (j = 0; j < n; ++j) {
    double m_new = x[j] > m ? x[j] : m;
    dsum = (m == -INFINITY ? 0.0 : dsum * exp(m - m_new)) + exp(x[j] - m_new);
    m = m_new;
  }
  for (j = 0; j < n; ++j) y[j] = exp(x[j] - m) / dsum;
}

/* Residual add + RMS normalisation of n_rows rows of `hidden` values each
 * ("Inference Engineering VII.07: Kernel and Operator Fusion" page,
 * section 4, the unfused form and the steps of the fused kernel; section 5,
 * why the kernel returns the new residual as well):
 *
 *   h_i   = x_i + r_i                        the new residual
 *   ms    = (1 / hidden) * sum_i h_i^2       mean of squares over the row
 *   out_i = h_i / sqrt(ms + eps) * w_i
 *
 * x, r: [n_rows, hidden], w: [hidden], bf16 bit patterns widened exactly to
 * fp64; out, h_out: [n_rows, hidden] fp64.  Nothing is rounded.  Returns
 * nonzero for a bad argument. */
int oracle_add_rms_norm_f64(const uint16_t* x, const uint16_t* r, const uint16_t* w, long n_rows,
                            long hidden, double eps, double* out, double* h_out) {
  if (n_rows < 0 || hidden < 1 || !(eps >= 0.0)) return 1;
#pragma omp parallel for schedule(static)
  for (long row = 0; row < n_rows; ++row) {
    const uint16_t* xr = x + row * hidden;
    const uint16_t* rr = r + row * hidden;
    double* hr = h_out + row * hidden;
    double ss = 0.0;
    for (long i = 0; i < hidden; ++i) {
      hr[i] = bf16_to_f64(xr[i]) + bf16_to_f64(rr[i]);
      ss += hr[i] * hr[i];
    }
    const double ms = ss / (double)hidden;
    const double denom = sqrt(ms + eps);
    double* o = out + row * hidden;
    for (long i = 0; i < hidden; ++i) o[i] = hr[i] / denom * bf16_to_f64(w[i]);
  }
  return 0;
}

/* Rotary position embedding of the new tokens' queries and keys, then the
 * store of the rotated key and the value into the block-paged cache
 * ("Inference Engineering VII.07: Kernel and Operator Fusion" page,
 * section 2, catalogue item "rope + cache write: RoPE then KV store";
 * "Fused Kernel Compiler" page, table of fusion patterns, "RoPE embedding:
 * sin, cos, rotate"; the cache layout of the "Optimizing LLM Inference ..."
 * page, section Paged Attention and Dynamic KV Cache Management).
 *
 * Readings (the pages name the operation only): pairs (i, i + d/2) of each
 * head vector are rotated by theta_i = pos * base^(-2 i / d),
 *   y_i       = x_i cos theta_i - x_(i+d/2) sin theta_i
 *   y_(i+d/2) = x_(i+d/2) cos theta_i + x_i sin theta_i,
 * for i in [0, d/2); token t of sequence seq_ids[t] at position
 * positions[t] goes to physical block block_table[seq][pos / 16], slot
 * pos % 16.
 *
 * q [T, Hq, d], k, v [T, Hkv, d] bf16 bits; q_out [T, Hq, d], k_out
 * [T, Hkv, d] fp64 (v is stored unchanged); slot_out [T]: block * 16 +
 * slot, or -1 when the position or the block lies outside the table or the
 * cache (nothing is stored then).  Returns nonzero for a bad argument. */
static void rope_vec(const uint16_t* x, int d, long pos, double base, double* y) {
  const int half = d / 2;
  for (int i = 0; i < half; ++i) {
    const double ang = (double)pos * pow(base, -2.0 * (double)i / (double)d);
    const double c = cos(ang), s = sin(ang);
    const double a = bf16_to_f64(x[i]), b = bf16_to_f64(x[i + half]);
    y[i] = a * c - b * s;
    y[i + half] = b * c + a * s;
  }
}

int oracle_rope_cache_write_f64(const uint16_t* q, const uint16_t* k, const int32_t* seq_ids,
                                const int32_t* positions, const int32_t* block_table, int T,
                                int Hq, int Hkv, int d, int num_seqs, int num_blocks,
                                int max_blocks_per_seq, double base, double* q_out, double* k_out,
                                long* slot_out) {
  if (T < 0 || Hq < 1 || Hkv < 1 || d < 2 || d % 2 != 0 || num_blocks < 0 || max_blocks_per_seq < 0 ||
      !(base > 0.0))
    return 1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const long pos = positions[t];
    const int seq = seq_ids[t];
    for (int h = 0; h < Hq; ++h)
      rope_vec(q + ((long)t * Hq + h) * d, d, pos, base, q_out + ((long)t * Hq + h) * d);
    for (int h = 0; h < Hkv; ++h)
      rope_vec(k + ((long)t * Hkv + h) * d, d, pos, base, k_out + ((long)t * Hkv + h) * d);
    long slot = -1;
    if (seq >= 0 && seq < num_seqs && pos >= 0 && pos / 16 < max_blocks_per_seq) {
      const long blk = block_table[(long)seq * max_blocks_per_seq + pos / 16];
      if (blk >= 0 && blk < num_blocks) slot = blk * 16 + pos % 16;
    }
    slot_out[t] = slot;
  }
  return 0;
}

/* Gradients of scaled dot-product attention with respect to Q, K and V,
 * given the gradient dO of the output ("Kernel Fusion, Softmax, and
 * Attention" page: training runs a different schedule of the same
 * attention equation; the chain rule through O = P V and P = softmax(S)):
 *
 *   P_ij  = exp(s_ij - lse_i)           the forward's probabilities
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = <dO_i, v_j>
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_i dS_ij q_i
 *
 * with the forward's mask, and dK, dV of a key/value head summed over the
 * query heads that read it.  q, dout [B, Hq, Nq, d], k, v [B, Hkv, Nk, d]
 * bf16 bits; dq [B, Hq, Nq, d], dk, dv [B, Hkv, Nk, d] fp64.  The full
 * probability row of each query is formed in fp64; a row that sees no key
 * contributes nothing.  Returns nonzero for a bad argument. */
int oracle_attn_bwd_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                        int B, int Hq, int Hkv, long Nq, long Nk, int d, double scale, int causal,
                        double* dq, double* dk, double* dv) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || d < 1) return 1;
  const int G = Hq / Hkv;
  long bk;
#pragma omp parallel for schedule(dynamic)
  for (bk = 0; bk < (long)B * Hkv; ++bk) {
    const long b = bk / Hkv, hk = bk % Hkv;
    const uint16_t* kh = k + (size_t)bk * Nk * d;
    const uint16_t* vh = v + (size_t)bk * Nk * d;
    double* dkh = dk + (size_t)bk * Nk * d;
    double* dvh = dv + (size_t)bk * Nk * d;
    for (size_t e = 0; e < (size_t)Nk * d; ++e) dkh[e] = dvh[e] = 0.0;
    double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double* dp = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)d);
    double* gd = (double*)malloc(sizeof(double) * (size_t)d);
    for (int g = 0; g < G; ++g) {
      const long hq = hk * G + g;
      const size_t head = (size_t)(b * Hq + hq) * Nq * d;
      for (long i = 0; i < Nq; ++i) {
        const long n_vis = visible_keys(i, Nq, Nk, causal);
        double* dqi = dq + head + (size_t)i * d;
        for (int t = 0; t < d; ++t) {
          qd[t] = bf16_to_f64(q[head + (size_t)i * d + t]);
          gd[t] = bf16_to_f64(dout[head + (size_t)i * d + t]);
          dqi[t] = 0.0;
        }
        if (n_vis <= 0) continue;
        double m = -INFINITY;
        for (long j = 0; j < n_vis; ++j) {
          double acc = 0.0;
          for (int t = 0; t < d; ++t) acc += qd[t] * bf16_to_f64(kh[(size_t)j * d + t]);
          s[j] = scale * acc;
          if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (long j = 0; j < n_vis; ++j) l += exp(s[j] - m);
        const double lse = m + log(l);
        double D = 0.0;
        for (long j = 0; j < n_vis; ++j) {
          s[j] = exp(s[j] - lse); /* now P_ij */
          double acc = 0.0;
          for (int t = 0; t < d; ++t) acc += gd[t] * bf16_to_f64(vh[(size_t)j * d + t]);
          dp[j] = acc;
          D += s[j] * acc;
        }
        for (long j = 0; j < n_vis; ++j) {
          const double pij = s[j];
          const double ds = pij * (dp[j] - D);
          for (int t = 0; t < d; ++t) {
            dqi[t] += scale * ds * bf16_to_f64(kh[(size_t)j * d + t]);
            dkh[(size_t)j * d + t] += scale * ds * qd[t];
            dvh[(size_t)j * d + t] += pij * gd[t];
          }
        }
      }
    }
    free(s);
    free(dp);
    free(qd);
    free(gd);
  }
  return 0;
}
