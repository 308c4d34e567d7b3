/*
 * asv_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously-correct CPU statement of the logit-space
 * verification step, in double precision.  Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * Sources (web pages; sections named as on the page):
 *   [ASYM]   "AsymSpec: Context-Asymmetric Speculative Decoding for Agentic LLMs"
 *            (reading notes): sec. 4.1 (contrastive delta-fusion), sec. 4.2 (CDA gate).
 *   [RAPID]  "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
 *            Decoding" (paper notes): Key design 2 (retrieval-augmented target
 *            distribution), 3 (tail-distribution protection), 4 (adjusted
 *            residual sampling); "Workflow" paragraph (rejection sampling with the
 *            augmented target).
 *   [SCI]    "E2-SCI: Elastic Edge-Cloud Speculative Decoding via Credit Inertia"
 *            (paper notes): Key design 3 (online adaptive verification: JSD test,
 *            EWMA of the acceptance rate, clamped threshold).
 *   [PHILOX] J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
 *            numbers: as easy as 1, 2, 3", SC'11 -- the Philox4x32-10 generator.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - JSD uses natural logs and weights 1/2 (the stated bound ln 2 fixes both).
 *   - The CDA accept test is the printed strict inequality, taken in the log domain.
 *   - The delta-fusion token is also emitted at the bonus row when all K drafts pass.
 *   - argmax ties go to the lowest index.  The delta-fusion score t + beta*(a - b)
 *     is taken exactly (double); a row whose winner another entry could displace
 *     under the rounding of a single-precision evaluation of the same score is
 *     marked as a near tie, counted by the parity tests instead of graded.
 *   - RAPID: probability-domain tail mask taken before protection; tail entries
 *     keep p exactly and the head is rescaled so the protected target sums to 1;
 *     accept iff u*q(d) < p'(d); residual max(p - p', p - q, 0) drawn by an
 *     exponential race over Philox uniforms.
 *   - SCI: the window's threshold comes from the credit state left by earlier
 *     windows; a draft is rejected when its JSD exceeds the threshold.
 *
 * Parity pins are in tests/test_oracle_*.py.  Element types: 0 = fp32, 1 = bf16
 * (uint16 bit patterns); both are widened to double exactly.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1

/* Per-request flags.  Bits 0 and 1 mirror conditions the library reports; the
 * rest mark requests whose outcome hinges on a comparison closer than the
 * stated tolerance, which parity tests count instead of grading. */
#define OR_NONFINITE 1u
#define OR_BAD_DRAFT 2u
#define OR_NEAR_MARGIN 4u
#define OR_NEAR_TAIL 8u
#define OR_NEAR_RACE 16u
#define OR_NEAR_TIE 32u

static float widen_f(const void* base, int dtype, size_t i) {
  if (dtype == OR_F32) return ((const float*)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

static double widen(const void* base, int dtype, size_t i) { return (double)widen_f(base, dtype, i); }

/* NaN or +inf anywhere in the row, or a row that is -inf everywhere (it has no
 * softmax).  A single -inf is a legal logit: probability 0. */
static int row_nonfinite(const void* x, int dtype, size_t off, int V) {
  int all_ninf = 1;
  for (int k = 0; k < V; ++k) {
    double v = widen(x, dtype, off + (size_t)k);
    if (isnan(v) || (isinf(v) && v > 0)) return 1;
    if (!(isinf(v) && v < 0)) all_ninf = 0;
  }
  return all_ninf;
}

/* Any NaN or infinity (probabilities must be finite). */
static int row_any_nonfinite(const float* x, size_t off, int V) {
  for (int k = 0; k < V; ++k)
    if (!isfinite(x[off + (size_t)k])) return 1;
  return 0;
}

/* log sum_k exp(scale * x_k), shifted by the maximum.  scale = 1/T for a
 * temperature T.  Returns -inf for a row that is all -inf. */
double oracle_lse(const void* x, int dtype, size_t off, int V, double scale) {
  double m = -INFINITY;
  for (int k = 0; k < V; ++k) {
    double v = scale * widen(x, dtype, off + (size_t)k);
    if (v > m) m = v;
  }
  if (isinf(m) && m < 0) return -INFINITY;
  double s = 0.0;
  for (int k = 0; k < V; ++k) s += exp(scale * widen(x, dtype, off + (size_t)k) - m);
  return m + log(s);
}

/* D = JSD(softmax x || softmax y) = 1/2 KL(P||M) + 1/2 KL(Q||M), M = (P+Q)/2,
 * natural log, 0 ln 0 = 0.  [ASYM] sec. 4.2. */
double oracle_jsd(const void* x, const void* y, int dtype, size_t offx, size_t offy, int V) {
  double Lx = oracle_lse(x, dtype, offx, V, 1.0);
  double Ly = oracle_lse(y, dtype, offy, V, 1.0);
  double D = 0.0;
  for (int k = 0; k < V; ++k) {
    double p = exp(widen(x, dtype, offx + (size_t)k) - Lx);
    double q = exp(widen(y, dtype, offy + (size_t)k) - Ly);
    double m = 0.5 * (p + q);
    if (p > 0.0) D += 0.5 * p * log(p / m);
    if (q > 0.0) D += 0.5 * q * log(q / m);
  }
  return D;
}

/* The context-gain signal of the delta-fusion score ([ASYM] sec. 5, mechanism
 * ablation): 0 -> delta = a - b (the method), 1 -> delta = a (raw enhanced
 * logits), 2 -> delta = t - b (two-model difference). */
static double delta_of(const void* a, const void* b, const void* t, int dtype, size_t i, int delta_source) {
  if (delta_source == 1) return widen(a, dtype, i);
  if (delta_source == 2) return widen(t, dtype, i) - widen(b, dtype, i);
  return widen(a, dtype, i) - widen(b, dtype, i);
}

/* 1 when delta and the score t + beta * delta are single-precision numbers and the
 * double evaluation of the score is exact (so every correctly rounded evaluation,
 * in any precision down to single, gives the same value): delta is checked by a
 * round trip through float; beta * delta is then exact in double (two 24-bit
 * significands); the sum's rounding error comes from Knuth's TwoSum. */
static int score_is_f32(double t, double beta, double d) {
  if ((double)(float)d != d) return 0;
  double p = beta * d;
  double s = t + p;
  double bp = s - t;
  double err = (t - (s - bp)) + (p - bp);
  return err == 0.0 && (double)(float)s == s;
}

/* The delta-fusion token, [ASYM] sec. 4.1: d' = argmax_k (t_k + beta * delta_k),
 * taken exactly: the stored values widen to double without rounding, their
 * difference and beta * delta are exact in double, and the sum carries a
 * rounding of order 1e-16 relative at most.  Lowest index among equal scores;
 * an entry whose score is NaN or -inf (a token the fused scores make impossible)
 * is never chosen; if no entry qualifies the result is 0.
 *
 * *near (may be NULL) is set when the decision is within rounding distance of
 * another entry k for a single-precision evaluation of the same score (delta
 * rounded once, then one rounded fused multiply-add, each within 2^-24 relative):
 *   0 < s_w - s_k <= 2^-22 * (|s_w| + |s_k| + |beta| * (|delta_w| + |delta_k|)),
 * four times the bound on the two scores' rounding errors; or s_k == s_w with
 * one of the two deltas or scores not a single-precision number (the rounding
 * could then order them either way). */
int oracle_fused_argmax_exact(const void* a, const void* b, const void* t, int dtype, size_t off, int V, double beta,
                              int delta_source, int* near) {
  int best = -1;
  double bv = -INFINITY;
  for (int k = 0; k < V; ++k) {
    size_t i = off + (size_t)k;
    double s = widen(t, dtype, i) + beta * delta_of(a, b, t, dtype, i, delta_source);
    if (s > bv) {
      bv = s;
      best = k;
    }
  }
  if (near) *near = 0;
  if (best < 0) return 0;
  if (near) {
    size_t iw = off + (size_t)best;
    double dw = delta_of(a, b, t, dtype, iw, delta_source);
    int exact_w = score_is_f32(widen(t, dtype, iw), beta, dw);
    for (int k = 0; k < V; ++k) {
      if (k == best) continue;
      size_t i = off + (size_t)k;
      double dk = delta_of(a, b, t, dtype, i, delta_source);
      double tk = widen(t, dtype, i);
      double sk = tk + beta * dk;
      if (!(sk > -INFINITY)) continue; /* NaN or -inf: never chosen */
      double gap = bv - sk;
      if (gap == 0.0) {
        if (!(exact_w && score_is_f32(tk, beta, dk))) *near = 1;
      } else if (gap <= ldexp(1.0, -22) * (fabs(bv) + fabs(sk) + fabs(beta) * (fabs(dw) + fabs(dk)))) {
        *near = 1;
      }
    }
  }
  return best;
}

/* What a single-precision evaluation of the same score picks: delta as one
 * rounded fp32 operation (none for delta = a), then one fused multiply-add,
 * lowest index among equal values, NaN/-inf never chosen (0 if none qualifies).
 * The verification does not use it: the tests count the rows where it differs
 * from the exact argmax (every such row must be a near tie). */
int oracle_fused_argmax_fp32(const void* a, const void* b, const void* t, int dtype, size_t off, int V, float beta,
                             int delta_source) {
  int best = -1;
  float bv = -INFINITY;
  for (int k = 0; k < V; ++k) {
    float ak = widen_f(a, dtype, off + (size_t)k);
    float bk = widen_f(b, dtype, off + (size_t)k);
    float tk = widen_f(t, dtype, off + (size_t)k);
    float d = delta_source == 1 ? ak : (delta_source == 2 ? tk - bk : ak - bk);
    float s = fmaf(beta, d, tk);
    if (s > bv) {
      bv = s;
      best = k;
    }
  }
  return best < 0 ? 0 : best;
}

/*
 * AsymSpec verification over a batch [B, K+1, V].  [ASYM] sec. 4.1-4.2.
 *
 * Per row i of request r:
 *   lse of a, b, t;  D_i = JSD(softmax a_i || softmax b_i);
 *   c_i = argmax(t_i + beta*(a_i - b_i)) (exact score, lowest index; near_i marks a
 *         winner within single-precision rounding of another entry);
 * per draft row i < K with d = draft_ids[r][i]:
 *   accept iff  softmax(t_i)[d] > gamma * exp(-D_i) * softmax(b_i)[d],
 *   i.e. margin_i = (t_d - lse_t) - ln gamma + D_i - (b_d - lse_b) > 0;
 * n = first rejected i (else K); tokens = d_0..d_{n-1}, c_n, then -1.
 *
 * Outputs (any may be NULL except accept_len/tokens):
 *   out_D [B,K+1], out_lse [B,K+1,3] (a,b,t), out_margin [B,K], out_argmax [B,K+1],
 *   out_near [B,K+1] (near_i), out_flags [B].  A request with a non-finite row or an
 *   out-of-range draft id gets accept_len 0 and tokens all -1.  A request whose emitted
 *   position n has a near tie is flagged OR_NEAR_TIE.
 */
void oracle_asymspec_verify_src(const void* a, const void* b, const void* t, int dtype,
                                const int32_t* draft_ids, int B, int K, int V, float beta, float gamma,
                                int delta_source, int32_t* out_accept_len, int32_t* out_tokens, double* out_D,
                                double* out_lse, double* out_margin, int32_t* out_argmax, int32_t* out_near,
                                uint32_t* out_flags) {
  const double ln_gamma = log((double)gamma);
  for (int r = 0; r < B; ++r) {
    uint32_t flags = 0;
    int n = K;
    double* margin = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    int32_t* cbest = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K + 1));
    int* cnear = (int*)malloc(sizeof(int) * (size_t)(K + 1));
    for (int i = 0; i < K; ++i) {
      int d = draft_ids[(size_t)r * K + i];
      if (d < 0 || d >= V) flags |= OR_BAD_DRAFT;
    }
    for (int i = 0; i <= K; ++i) {
      size_t off = ((size_t)r * (K + 1) + i) * (size_t)V;
      if (row_nonfinite(a, dtype, off, V) || row_nonfinite(b, dtype, off, V) || row_nonfinite(t, dtype, off, V))
        flags |= OR_NONFINITE;
      double La = oracle_lse(a, dtype, off, V, 1.0);
      double Lb = oracle_lse(b, dtype, off, V, 1.0);
      double Lt = oracle_lse(t, dtype, off, V, 1.0);
      double D = oracle_jsd(a, b, dtype, off, off, V);
      int c = oracle_fused_argmax_exact(a, b, t, dtype, off, V, (double)beta, delta_source, &cnear[i]);
      cbest[i] = c;
      if (out_near) out_near[(size_t)r * (K + 1) + i] = cnear[i];
      size_t ri = (size_t)r * (K + 1) + i;
      if (out_D) out_D[ri] = D;
      if (out_lse) {
        out_lse[ri * 3 + 0] = La;
        out_lse[ri * 3 + 1] = Lb;
        out_lse[ri * 3 + 2] = Lt;
      }
      if (out_argmax) out_argmax[ri] = c;
      if (i < K) {
        int d = draft_ids[(size_t)r * K + i];
        double m = NAN;
        if (d >= 0 && d < V) {
          double lpt = widen(t, dtype, off + (size_t)d) - Lt;
          double lpb = widen(b, dtype, off + (size_t)d) - Lb;
          m = lpt - ln_gamma + D - lpb;
        }
        margin[i] = m;
        if (out_margin) out_margin[(size_t)r * K + i] = m;
      }
    }
    if (flags & (OR_NONFINITE | OR_BAD_DRAFT)) {
      out_accept_len[r] = 0;
      for (int i = 0; i <= K; ++i) out_tokens[(size_t)r * (K + 1) + i] = -1;
    } else {
      n = K;
      for (int i = 0; i < K; ++i) {
        if (fabs(margin[i]) < 1e-6) flags |= OR_NEAR_MARGIN;
        if (!(margin[i] > 0.0)) {
          n = i;
          break;
        }
      }
      out_accept_len[r] = n;
      if (cnear[n]) flags |= OR_NEAR_TIE;
      for (int i = 0; i <= K; ++i) {
        int32_t tok = -1;
        if (i < n) tok = draft_ids[(size_t)r * K + i];
        else if (i == n) tok = cbest[n];
        out_tokens[(size_t)r * (K + 1) + i] = tok;
      }
    }
    if (out_flags) out_flags[r] = flags;
    free(margin);
    free(cbest);
    free(cnear);
  }
}

void oracle_asymspec_verify(const void* a, const void* b, const void* t, int dtype, const int32_t* draft_ids, int B,
                            int K, int V, float beta, float gamma, int32_t* out_accept_len, int32_t* out_tokens,
                            double* out_D, double* out_lse, double* out_margin, int32_t* out_argmax,
                            int32_t* out_near, uint32_t* out_flags) {
  oracle_asymspec_verify_src(a, b, t, dtype, draft_ids, B, K, V, beta, gamma, 0, out_accept_len, out_tokens, out_D,
                             out_lse, out_margin, out_argmax, out_near, out_flags);
}

/* ------------------------------------------------------------------ Philox */

/* Philox4x32 with 10 rounds.  [PHILOX] sec. 5: each round multiplies words 0
 * and 2 by the two round multipliers, mixes the high halves with the other
 * words and the key, and the key is advanced by the Weyl constants between
 * rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* Uniform in (0,1) from one 32-bit word: the top 23 bits plus one half, scaled
 * by 2^-23.  Exactly representable in fp32, never 0 or 1. */
double oracle_uniform_from_word(uint32_t w) { return ((double)(w >> 9) + 0.5) * (1.0 / 8388608.0); }

/* Counter layout shared (by specification, not by code) with the library:
 *   key = (seed low 32 bits, seed high 32 bits)
 *   ctr = (word_index / 4, row i, request r, stream + 4 * offset)
 * and the uniform is word (word_index % 4) of the block.  Streams: 0 accept
 * test, 1 residual draw, 2 bonus draw. */
double oracle_rapid_uniform(uint64_t seed, uint32_t offset, uint32_t stream, uint32_t req, uint32_t row,
                            uint32_t word) {
  uint32_t ctr[4] = {word >> 2, row, req, stream + 4u * offset};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return oracle_uniform_from_word(out[word & 3u]);
}

/*
 * One RAPID row.  [RAPID] Key design 2-3.
 *   p    = softmax(z / T)
 *   zhat = z + eta * T * (q - p)
 *   phat = softmax(zhat / T)
 *   tail = { k : phat_k < tail_frac * max_j phat_j }
 *   tail_mode 0: prot_k = p_k on the tail; on the head phat_k * (1 - sum_tail p) / sum_head phat.
 *   tail_mode 1 (the other reading: substitute p on the tail, then renormalise every entry):
 *     w_k = p_k on the tail, phat_k on the head; prot_k = w_k / sum_j w_j.
 * Arrays p, zhat, phat, prot are length V (any may be NULL).  Returns the
 * number of tail entries; *near is set when some phat_k lies within a relative
 * 1e-5 of the tail boundary (the library decides the mask in fp32).
 */
int oracle_rapid_row_mode(const float* z, const float* q, int V, double T, double eta, double tail_frac,
                          int tail_mode, double* p_out, double* zhat_out, double* phat_out, double* prot_out,
                          int* near) {
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* zh = (double*)malloc(sizeof(double) * (size_t)V);
  double* ph = (double*)malloc(sizeof(double) * (size_t)V);
  double Lz = oracle_lse(z, OR_F32, 0, V, 1.0 / T);
  for (int k = 0; k < V; ++k) p[k] = exp((double)z[k] / T - Lz);
  for (int k = 0; k < V; ++k) zh[k] = (double)z[k] + eta * T * ((double)q[k] - p[k]);
  double m = -INFINITY;
  for (int k = 0; k < V; ++k)
    if (zh[k] / T > m) m = zh[k] / T;
  double s = 0.0;
  for (int k = 0; k < V; ++k) s += exp(zh[k] / T - m);
  double Lh = m + log(s);
  double pmax = 0.0;
  for (int k = 0; k < V; ++k) {
    ph[k] = exp(zh[k] / T - Lh);
    if (ph[k] > pmax) pmax = ph[k];
  }
  double thr = tail_frac * pmax;
  double tail_p = 0.0, head_ph = 0.0;
  int ntail = 0, nr = 0;
  for (int k = 0; k < V; ++k) {
    if (fabs(ph[k] - thr) <= 1e-5 * thr) nr = 1;
    if (ph[k] < thr) {
      tail_p += p[k];
      ++ntail;
    } else {
      head_ph += ph[k];
    }
  }
  double scale = (1.0 - tail_p) / head_ph;
  double wsum = 0.0;  /* tail_mode 1: the sum of the substituted weights */
  for (int k = 0; k < V; ++k) wsum += (ph[k] < thr) ? p[k] : ph[k];
  for (int k = 0; k < V; ++k) {
    if (p_out) p_out[k] = p[k];
    if (zhat_out) zhat_out[k] = zh[k];
    if (phat_out) phat_out[k] = ph[k];
    if (prot_out) {
      if (tail_mode == 0) prot_out[k] = (ph[k] < thr) ? p[k] : ph[k] * scale;
      else prot_out[k] = ((ph[k] < thr) ? p[k] : ph[k]) / wsum;
    }
  }
  if (near) *near = nr;
  free(p);
  free(zh);
  free(ph);
  return ntail;
}

int oracle_rapid_row(const float* z, const float* q, int V, double T, double eta, double tail_frac, double* p_out,
                     double* zhat_out, double* phat_out, double* prot_out, int* near) {
  return oracle_rapid_row_mode(z, q, V, T, eta, tail_frac, 0, p_out, zhat_out, phat_out, prot_out, near);
}

/* Exponential race: argmin_k E_k / w_k over w_k > 0, E_k = -ln u_k with u_k the
 * Philox uniform for (stream, req, row, word k).  The winner is distributed as
 * w / sum(w).  Lowest index on ties; -1 when every weight is 0.  *near is set
 * when the two smallest keys are within a relative 1e-5. */
int oracle_race(const double* w, int V, uint64_t seed, uint32_t offset, uint32_t stream, uint32_t req,
                uint32_t row, int* near) {
  int best = -1;
  double k1 = INFINITY, k2 = INFINITY;
  for (int k = 0; k < V; ++k) {
    if (!(w[k] > 0.0)) continue;
    double u = oracle_rapid_uniform(seed, offset, stream, req, row, (uint32_t)k);
    double key = -log(u) / w[k];
    if (key < k1) {
      k2 = k1;
      k1 = key;
      best = k;
    } else if (key < k2) {
      k2 = key;
    }
  }
  if (near) *near = (best >= 0 && isfinite(k2) && (k2 - k1) <= 1e-5 * k1) ? 1 : 0;
  return best;
}

/*
 * RAPID verification over [B, G+1, V] fp32 target logits z and drafter
 * probabilities q.  [RAPID] Workflow + Key designs 2-4.
 *   accept draft i iff u_i * q_i(d_i) < prot_i(d_i), u_i the stream-0 uniform of row i;
 *   n = first rejection (else G);
 *   if n < G: token n ~ norm(max(p_n - prot_n, p_n - q_n, 0)) (stream 1; a draw
 *             from p_n if that residual is all zero);
 *   else:     token G ~ prot_G (stream 2).
 */
void oracle_rapid_verify_mode(const float* z, const float* q, const int32_t* draft_ids, int B, int G, int V,
                              double T, double eta, double tail_frac, int tail_mode, uint64_t seed, uint32_t offset,
                              int32_t* out_accept_len, int32_t* out_tokens, uint32_t* out_flags) {
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* prot = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  for (int b = 0; b < B; ++b) {
    uint32_t flags = 0;
    for (int i = 0; i < G; ++i) {
      int d = draft_ids[(size_t)b * G + i];
      if (d < 0 || d >= V) flags |= OR_BAD_DRAFT;
    }
    for (int i = 0; i <= G; ++i) {
      size_t off = ((size_t)b * (G + 1) + i) * (size_t)V;
      if (row_nonfinite(z, OR_F32, off, V) || row_any_nonfinite(q, off, V)) flags |= OR_NONFINITE;
    }
    if (flags) {
      out_accept_len[b] = 0;
      for (int i = 0; i <= G; ++i) out_tokens[(size_t)b * (G + 1) + i] = -1;
      if (out_flags) out_flags[b] = flags;
      continue;
    }
    int n = G, near = 0;
    for (int i = 0; i < G; ++i) {
      size_t off = ((size_t)b * (G + 1) + i) * (size_t)V;
      oracle_rapid_row_mode(z + off, q + off, V, T, eta, tail_frac, tail_mode, NULL, NULL, NULL, prot, &near);
      if (near) flags |= OR_NEAR_TAIL;
      int d = draft_ids[(size_t)b * G + i];
      double u = oracle_rapid_uniform(seed, offset, 0u, (uint32_t)b, (uint32_t)i, 0u);
      double lhs = u * (double)q[off + (size_t)d];
      double rhs = prot[d];
      if (fabs(lhs - rhs) <= 1e-5 * fabs(rhs)) flags |= OR_NEAR_MARGIN;
      if (!(lhs < rhs)) {
        n = i;
        break;
      }
    }
    size_t off = ((size_t)b * (G + 1) + n) * (size_t)V;
    oracle_rapid_row_mode(z + off, q + off, V, T, eta, tail_frac, tail_mode, p, NULL, NULL, prot, &near);
    if (near) flags |= OR_NEAR_TAIL;
    int tok, rn = 0;
    if (n < G) {
      for (int k = 0; k < V; ++k) {
        double v = p[k] - prot[k];
        double w = p[k] - (double)q[off + (size_t)k];
        double m = v > w ? v : w;
        r[k] = m > 0.0 ? m : 0.0;
      }
      tok = oracle_race(r, V, seed, offset, 1u, (uint32_t)b, (uint32_t)n, &rn);
      if (tok < 0) tok = oracle_race(p, V, seed, offset, 1u, (uint32_t)b, (uint32_t)n, &rn);
    } else {
      tok = oracle_race(prot, V, seed, offset, 2u, (uint32_t)b, (uint32_t)G, &rn);
    }
    if (rn) flags |= OR_NEAR_RACE;
    out_accept_len[b] = n;
    for (int i = 0; i <= G; ++i) {
      int32_t v = -1;
      if (i < n) v = draft_ids[(size_t)b * G + i];
      else if (i == n) v = tok;
      out_tokens[(size_t)b * (G + 1) + i] = v;
    }
    if (out_flags) out_flags[b] = flags;
  }
  free(p);
  free(prot);
  free(r);
}

void oracle_rapid_verify(const float* z, const float* q, const int32_t* draft_ids, int B, int G, int V, double T,
                         double eta, double tail_frac, uint64_t seed, uint32_t offset, int32_t* out_accept_len,
                         int32_t* out_tokens, uint32_t* out_flags) {
  oracle_rapid_verify_mode(z, q, draft_ids, B, G, V, T, eta, tail_frac, 0, seed, offset, out_accept_len, out_tokens,
                           out_flags);
}

/* ------------------------------------------------------------------ E2-SCI */

/* T = max(T_min, min(T_base + alpha*omega*(r_hat - tau_credit), T_max)).  [SCI] Key design 3. */
double oracle_sci_threshold(double r_hat, double T_base, double alpha_omega, double tau_credit, double T_min,
                            double T_max) {
  double T = T_base + alpha_omega * (r_hat - tau_credit);
  if (T > T_max) T = T_max;
  if (T < T_min) T = T_min;
  return T;
}

/* r_hat <- (1 - beta) * r_hat + beta * p_acc.  [SCI] Key design 3. */
double oracle_sci_ewma(double r_hat, double p_acc, double beta) { return (1.0 - beta) * r_hat + beta * p_acc; }

/*
 * E2-SCI stabilisers ([SCI] Key design 3 names hysteresis, a minimum refresh interval and a
 * fallback to a conservative threshold when the accuracy under the predicted threshold drops
 * below delta; it gives no constants).  One window's threshold from the candidate T_cand and the
 * request's state (T_applied, age = windows since the applied threshold last changed, set,
 * fallback pending):
 *   first window (not set)            -> T_cand
 *   fallback pending                  -> fallback_T
 *   age >= min_refresh and |T_cand - T_applied| > hysteresis -> T_cand
 *   otherwise                         -> T_applied (age grows by one)
 * A change sets age to 1.  After the window, fallback is pending for the next one iff the
 * window's acceptance rate n / K is below fallback_acc.  With hysteresis 0, min_refresh 1 and
 * fallback_acc 0 every window uses T_cand.
 */
typedef struct {
  double T_applied;
  int32_t age;
  uint32_t flags; /* 1: a threshold has been applied; 2: fallback pending */
} oracle_sci_state;

double oracle_sci_stab_threshold(const oracle_sci_state* st, double T_cand, double hysteresis, int min_refresh,
                                 double fallback_T, int32_t* new_age) {
  if (!(st->flags & 1u)) {
    *new_age = 1;
    return T_cand;
  }
  if (st->flags & 2u) {
    *new_age = 1;
    return fallback_T;
  }
  if (st->age >= min_refresh && fabs(T_cand - st->T_applied) > hysteresis) {
    *new_age = 1;
    return T_cand;
  }
  *new_age = st->age + 1;
  return st->T_applied;
}

/*
 * One E2-SCI verification window per request over [B, K+1, V] draft and
 * target logits.  [SCI] Key design 3.
 *   T = threshold(r_hat[r]) (through the stabilisers when `state` is given);
 *   J_i = JSD(softmax draft_i || softmax target_i);
 *   draft i is accepted while J_i <= T (rejected when J_i > T); n = accepted prefix;
 *   tokens = d_0..d_{n-1}, argmax(target_n) (lowest index);
 *   p_acc = n / K;  r_hat[r] <- ewma(r_hat[r], p_acc)   (in place; state updated likewise).
 * out_jsd [B,K+1] and out_T [B] are optional.  A flagged request keeps its r_hat and state.
 */
void oracle_sci_verify_stab(const void* draft, const void* target, int dtype, const int32_t* draft_ids, int B,
                            int K, int V, double T_base, double alpha_omega, double tau_credit, double T_min,
                            double T_max, double ewma_beta, double hysteresis, int min_refresh, double fallback_acc,
                            double fallback_T, oracle_sci_state* state, double* r_hat, int32_t* out_accept_len,
                            int32_t* out_tokens, double* out_jsd, double* out_T, uint32_t* out_flags) {
  double* J = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  for (int r = 0; r < B; ++r) {
    uint32_t flags = 0;
    double T = oracle_sci_threshold(r_hat[r], T_base, alpha_omega, tau_credit, T_min, T_max);
    int32_t age = 0;
    if (state) T = oracle_sci_stab_threshold(&state[r], T, hysteresis, min_refresh, fallback_T, &age);
    if (out_T) out_T[r] = T;
    for (int i = 0; i < K; ++i) {
      int d = draft_ids[(size_t)r * K + i];
      if (d < 0 || d >= V) flags |= OR_BAD_DRAFT;
    }
    for (int i = 0; i <= K; ++i) {
      size_t off = ((size_t)r * (K + 1) + i) * (size_t)V;
      if (row_nonfinite(draft, dtype, off, V) || row_nonfinite(target, dtype, off, V)) flags |= OR_NONFINITE;
      J[i] = oracle_jsd(draft, target, dtype, off, off, V);
      if (out_jsd) out_jsd[(size_t)r * (K + 1) + i] = J[i];
    }
    if (flags & (OR_NONFINITE | OR_BAD_DRAFT)) {
      out_accept_len[r] = 0;
      for (int i = 0; i <= K; ++i) out_tokens[(size_t)r * (K + 1) + i] = -1;
      if (out_flags) out_flags[r] = flags;
      continue; /* the credit state is left unchanged */
    }
    int n = K;
    for (int i = 0; i < K; ++i) {
      if (fabs(J[i] - T) < 1e-6) flags |= OR_NEAR_MARGIN;
      if (J[i] > T) {
        n = i;
        break;
      }
    }
    size_t offn = ((size_t)r * (K + 1) + n) * (size_t)V;
    int c = -1;
    float bv = -INFINITY;
    for (int k = 0; k < V; ++k) {
      float v = widen_f(target, dtype, offn + (size_t)k);
      if (v > bv) {
        bv = v;
        c = k;
      }
    }
    if (c < 0) c = 0;
    out_accept_len[r] = n;
    for (int i = 0; i <= K; ++i) {
      int32_t v = -1;
      if (i < n) v = draft_ids[(size_t)r * K + i];
      else if (i == n) v = c;
      out_tokens[(size_t)r * (K + 1) + i] = v;
    }
    const double p_acc = K > 0 ? (double)n / (double)K : 0.0;
    r_hat[r] = oracle_sci_ewma(r_hat[r], p_acc, ewma_beta);
    if (state) {
      state[r].T_applied = T;
      state[r].age = age;
      state[r].flags = 1u | (p_acc < fallback_acc ? 2u : 0u);
    }
    if (out_flags) out_flags[r] = flags;
  }
  free(J);
}

void oracle_sci_verify(const void* draft, const void* target, int dtype, const int32_t* draft_ids, int B, int K,
                       int V, double T_base, double alpha_omega, double tau_credit, double T_min, double T_max,
                       double ewma_beta, double* r_hat, int32_t* out_accept_len, int32_t* out_tokens,
                       double* out_jsd, double* out_T, uint32_t* out_flags) {
  oracle_sci_verify_stab(draft, target, dtype, draft_ids, B, K, V, T_base, alpha_omega, tau_credit, T_min, T_max,
                         ewma_beta, 0.0, 1, 0.0, 0.0, NULL, r_hat, out_accept_len, out_tokens, out_jsd, out_T,
                         out_flags);
}
