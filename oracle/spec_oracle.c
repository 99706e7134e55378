/*
 * spec_oracle.c -- plain, slow CPU oracle for the token-level hot path of speculative
 * decoding (draft proposal, target verification, confidence and prefix scheduling).
 *
 * TEST INFRASTRUCTURE ONLY. The product library never links, loads or calls this file.
 * Only the tests, __graft_entry__.smoke() and the CPU-baseline leg of bench.py use it.
 * It shares no code, header, table or helper with the CUDA library: it defines its own
 * constants, its own bf16 decode and its own loops.
 *
 * What it restates, and where the pages define it:
 *   - Draft distribution of the semi-autoregressive Markov head:
 *       "[DeepSeek-6] DSpark", section 3 (p_k(v | x0, x<k) = softmax_v(U_k(v) + B_k(..., v)))
 *       and section 4 "Markov Head" (B(x_{k-1}, .) = W1[x_{k-1}] W2, default rank 256).
 *     Section 3 also makes the anchor the first predicted position ("anchor + gamma-1 masks"
 *     yields gamma logit rows), so draft position k reads base-logit row k-1 and the bias of
 *     position 1 is conditioned on the anchor x0.
 *   - MTP/NextN greedy proposal: "Module deepseek_v4_mtp", Forward (draft = argmax(logits)).
 *   - Verify window [bonus, d1..d_gamma] and greedy longest-prefix acceptance plus one target
 *     token: "DeepSeek-V4 MTP/NextN 怎样逐步生成候选", sections 三 and 四, and DSpark section 1
 *     (accept the longest legal prefix, then emit one bonus token).
 *   - Lossless rejection sampling: named in DSpark sections 3 and 9, never printed there.
 *     This file follows the standard speculative-sampling rule: accept x_k with probability
 *     min(1, p_t(x_k)/p_d(x_k)); at the first rejection draw from norm(max(0, p_t - p_d));
 *     if every proposed token is accepted draw the bonus from p_t of the next row.
 *   - TV soft label c*_k = 1 - 1/2 ||p_d,k - p_t,k||_1: DSpark section 5.
 *   - Prefix survival a_{r,j} = prod_{i<=j} c_{r,i}, B = sum(1 + l_r),
 *     tau = sum(1 + sum_{j<=l_r} a_{r,j}), Theta = tau * SPS(B), queue all (r, j) by a_{r,j}
 *     descending: DSpark section 6.
 *
 * Readings where the pages are silent:
 *   R1  Markov bias arithmetic. With fp32 weights the bias is the canonical fp32 chain
 *       acc = fmaf(W1[x][i], W2[v][i], acc) for i = 0..r-1 ascending, and the logit is the
 *       fp32 sum U + acc. With bf16 weights every product is exact and the sum is taken in
 *       fp64. W2 is stored [V, r]: row v holds the r weights that project onto token v
 *       (the weight layout of a bias-free linear layer r -> V).
 *   R2  Temperature. One T scales draft and target logits alike, after the bias is added;
 *       invT is the fp32 number 1.0f/T. T == 0 (or no uniforms) means greedy argmax, and the
 *       reported draft log-probabilities are then those of the unscaled softmax.
 *   R3  Argmax ties go to the lowest token id.
 *   R4  Inverse-CDF sampling with u in [0,1): the smallest v whose cumulative probability
 *       (ascending token id) exceeds u; if rounding leaves none, the largest v with p(v) > 0.
 *   R5  Target row i scores the token after window position i: draft x_k is checked
 *       against row k-1, and row l is the bonus row when all l proposed tokens survive.
 *   R6  Acceptance test: accept iff u * p_d(x) < p_t(x) (strict), i.e. u < min(1, p_t/p_d).
 *   R7  Scheduler: candidates ordered by (a desc, r asc, j asc); tau is carried in fixed
 *       point q = round-half-even(a * 2^32) so that S_K is an exact integer;
 *       Theta(K) = double(R * 2^32 + S_K) * SPS[R + K]; K ranges over
 *       [0, min(R*gamma, Bmax - R)]; K* is the smallest K reaching the maximum; l_r is the
 *       number of selected candidates of request r.
 *   R11 Grammar-masked drafting: an optional per-request bitmask of ceil(V/32) words (bit
 *       v%32 of word v/32 set = token v may be proposed) restricts the draft distribution of
 *       every position to the allowed tokens (their logits are -inf otherwise); argmax,
 *       sampling, log p_d and (m, log Z), the residual and the TV label all use that
 *       restricted p_d. The target distribution is never masked.
 *
 * Arithmetic is fp64 except where R1 fixes fp32. Requests are independent in every function
 * but the scheduler; OpenMP spreads requests over host threads and nothing else.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype and status codes: same numeric values as the public header of the CUDA library,
 * restated here so that the two share no header. */
#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG (-1)
#define ORACLE_ERR_UNSUPPORTED_DTYPE (-2)
#define ORACLE_ERR_NO_MEMORY (-7)

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- element access */

static float bf16_bits_to_float(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* Element i of an f32 or bf16 array, as the exact fp32 value it encodes. */
static float elem(const void* base, int dtype, size_t i) {
  if (dtype == ORACLE_BF16) return bf16_bits_to_float(((const uint16_t*)base)[i]);
  return ((const float*)base)[i];
}

static int dtype_ok(int d) { return d == ORACLE_F32 || d == ORACLE_BF16; }

/* ---------------------------------------------------------------- building blocks */

/* Softmax of z[0..n) in fp64 (DSpark section 3): p(v) = exp(z(v) - m) / sum_u exp(z(u) - m).
 * Writes p and returns m and log Z (Z = sum exp(z - m)). */
void oracle_softmax(const double* z, int n, double* p, double* m_out, double* logz_out) {
  double m = z[0];
  for (int v = 1; v < n; ++v)
    if (z[v] > m) m = z[v];
  double Z = 0.0;
  for (int v = 0; v < n; ++v) {
    p[v] = exp(z[v] - m);
    Z += p[v];
  }
  for (int v = 0; v < n; ++v) p[v] /= Z;
  if (m_out) *m_out = m;
  if (logz_out) *logz_out = log(Z);
}

/* Argmax with ties to the lowest index (reading R3). If gap_out is given it receives the
 * distance from the maximum to the best other value (0 on an exact tie). */
int oracle_argmax(const double* s, int n, double* gap_out) {
  int best = 0;
  for (int v = 1; v < n; ++v)
    if (s[v] > s[best]) best = v;
  if (gap_out) {
    double second = -INFINITY;
    for (int v = 0; v < n; ++v)
      if (v != best && s[v] > second) second = s[v];
    *gap_out = (n > 1) ? s[best] - second : INFINITY;
  }
  return best;
}

/* Inverse-CDF draw from a normalised distribution p[0..n) with u in [0,1) (reading R4).
 * margin_out receives min(u - C(v-1), C(v) - u) for the returned v, the distance from u to
 * the nearer of the two cumulative sums that bracket it (0 if rounding left no crossing). */
int oracle_sample(const double* p, int n, double u, double* margin_out) {
  double c = 0.0;
  int last_positive = -1;
  for (int v = 0; v < n; ++v) {
    double before = c;
    c += p[v];
    if (p[v] > 0.0) last_positive = v;
    if (c > u) {
      if (margin_out) *margin_out = fmin(u - before, c - u);
      return v;
    }
  }
  if (margin_out) *margin_out = 0.0;
  return last_positive;
}

/* Acceptance test of rejection sampling (reading R6): accept the proposed token x iff
 * u * p_d(x) < p_t(x). Over u ~ U[0,1) this accepts with probability min(1, p_t/p_d). */
int oracle_accept_test(double u, double pd_x, double pt_x) { return u * pd_x < pt_x; }

/* The acceptance probability that oracle_accept_test realises: min(1, p_t/p_d). */
double oracle_accept_prob(double pd_x, double pt_x) {
  double ratio = pt_x / pd_x;
  return ratio < 1.0 ? ratio : 1.0;
}

/* Residual distribution after a rejection: q = norm(max(0, p_t - p_d)). Returns the
 * normaliser sum max(0, p_t - p_d) (0 when p_t == p_d, then q is left all zero). */
double oracle_residual(const double* pt, const double* pd, int n, double* q) {
  double Zq = 0.0;
  for (int v = 0; v < n; ++v) {
    double d = pt[v] - pd[v];
    q[v] = d > 0.0 ? d : 0.0;
    Zq += q[v];
  }
  if (Zq > 0.0)
    for (int v = 0; v < n; ++v) q[v] /= Zq;
  return Zq;
}

/* ---------------------------------------------------------------- logits */

typedef struct {
  const void* U; /* draft base logits [R, gamma, V] */
  int u_dtype;
  const void* W1; /* Markov embedding [V, rank] */
  const void* W2; /* Markov projection [V, rank] (row v projects onto token v) */
  int w_dtype;
  int rank;
  int gamma, V;
  const uint32_t* mask; /* allowed draft tokens [R, ceil(V/32)] (bit v%32 of word v/32), or NULL */
} DraftSide;

/* Pre-temperature draft scores s(v) of request r at draft position k (1-based) given the
 * previous token prev (DSpark sections 3-4, readings R1 and the anchor-first layout). A
 * disallowed token of a masked request scores -inf (grammar-masked drafting, "Module
 * deepseek_v4_mtp", Forward: the draft argmax is grammar-masked; reading R11). */
static void draft_scores(const DraftSide* d, int r, int k, int32_t prev, double* s) {
  const size_t row = ((size_t)r * d->gamma + (size_t)(k - 1)) * (size_t)d->V;
  const int rk = d->rank;
  for (int v = 0; v < d->V; ++v) {
    const float u = elem(d->U, d->u_dtype, row + (size_t)v);
    if (rk == 0) {
      s[v] = (double)u;
    } else if (d->w_dtype == ORACLE_F32) {
      const float* w1 = (const float*)d->W1 + (size_t)prev * rk;
      const float* w2 = (const float*)d->W2 + (size_t)v * rk;
      float acc = 0.0f;
      for (int i = 0; i < rk; ++i) acc = fmaf(w1[i], w2[i], acc);
      float sum = u + acc;
      s[v] = (double)sum;
    } else {
      double b = 0.0;
      for (int i = 0; i < rk; ++i)
        b += (double)elem(d->W1, ORACLE_BF16, (size_t)prev * rk + (size_t)i) *
             (double)elem(d->W2, ORACLE_BF16, (size_t)v * rk + (size_t)i);
      s[v] = (double)u + b;
    }
  }
  if (d->mask) {
    const uint32_t* mrow = d->mask + (size_t)r * (size_t)((d->V + 31) / 32);
    for (int v = 0; v < d->V; ++v)
      if (!((mrow[v / 32] >> (v % 32)) & 1u)) s[v] = -INFINITY;
  }
}

/* p_d at draft position k of request r after previous token prev, at inverse temperature
 * invT. Exposed for the exact-enumeration pin. */
int oracle_draft_probs(const void* U, int u_dtype, const void* W1, const void* W2, int w_dtype,
                       int rank, int R, int gamma, int V, int r, int k, int32_t prev,
                       float temperature, double* p_out, double* m_out, double* logz_out,
                       const uint32_t* mask) {
  if (!U || !p_out || r < 0 || r >= R || k < 1 || k > gamma || V < 1 || rank < 0)
    return ORACLE_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || prev < 0 || prev >= V)) return ORACLE_ERR_INVALID_ARG;
  DraftSide d = {U, u_dtype, W1, W2, w_dtype, rank, gamma, V, mask};
  double* s = (double*)malloc(sizeof(double) * (size_t)V);
  if (!s) return ORACLE_ERR_NO_MEMORY;
  draft_scores(&d, r, k, prev, s);
  const double invT = temperature > 0.0f ? (double)(1.0f / temperature) : 1.0;
  for (int v = 0; v < V; ++v) s[v] *= invT;
  oracle_softmax(s, V, p_out, m_out, logz_out);
  free(s);
  return ORACLE_OK;
}

/* p_t of target row i of request r (rows laid out [R, rows_per_req, V]). */
static void target_probs_row(const void* target, int t_dtype, int rows_per_req, int V, int r,
                             int i, double invT, double* z, double* p, double* m,
                             double* logz) {
  const size_t row = ((size_t)r * rows_per_req + (size_t)i) * (size_t)V;
  for (int v = 0; v < V; ++v) z[v] = (double)elem(target, t_dtype, row + (size_t)v) * invT;
  oracle_softmax(z, V, p, m, logz);
}

int oracle_target_probs(const void* target, int t_dtype, int R, int rows_per_req, int V, int r,
                        int i, float temperature, double* p_out) {
  if (!target || !p_out || r < 0 || r >= R || i < 0 || i >= rows_per_req || V < 1)
    return ORACLE_ERR_INVALID_ARG;
  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  if (!z) return ORACLE_ERR_NO_MEMORY;
  const double invT = temperature > 0.0f ? (double)(1.0f / temperature) : 1.0;
  target_probs_row(target, t_dtype, rows_per_req, V, r, i, invT, z, p_out, NULL, NULL);
  free(z);
  return ORACLE_OK;
}

/* ---------------------------------------------------------------- 1. draft proposal */

/*
 * Draft proposal for gamma serial positions (DSpark sections 3-4; rank == 0 is the plain
 * MTP/NextN argmax of "Module deepseek_v4_mtp"):
 *   for k = 1..gamma:  s = U[r, k-1, :] + W1[x_{k-1}] W2   (x_0 = anchor)
 *                      x_k = argmax s                       (greedy)
 *                      x_k = inverse-CDF(softmax(s * invT), u_draft[r, k-1])  (sampling)
 * Outputs per (r, k): the token, log p_d(x_k), the softmax stats (m, log Z) of s * invT, and
 * the decision margin (CDF margin when sampling; top-two score gap when greedy).
 */
int oracle_markov_propose(const void* U, int u_dtype, const void* W1, const void* W2,
                          int w_dtype, int rank, const int32_t* anchors, const float* u_draft,
                          float temperature, int R, int gamma, int V, int32_t* draft_tokens,
                          double* draft_logp, double* draft_stats, double* margin,
                          const uint32_t* mask) {
  if (R < 0 || gamma < 0 || V < 1 || rank < 0 || !dtype_ok(u_dtype))
    return R < 0 || gamma < 0 || V < 1 || rank < 0 ? ORACLE_ERR_INVALID_ARG
                                                  : ORACLE_ERR_UNSUPPORTED_DTYPE;
  if (R == 0 || gamma == 0) return ORACLE_OK;
  if (!U || !draft_tokens || !(temperature >= 0.0f)) return ORACLE_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || !anchors || !dtype_ok(w_dtype)))
    return ORACLE_ERR_INVALID_ARG;
  const int greedy = (u_draft == NULL) || (temperature == 0.0f);
  const double invT = greedy ? 1.0 : (double)(1.0f / temperature);
  DraftSide d = {U, u_dtype, W1, W2, w_dtype, rank, gamma, V, mask};
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < R; ++r) {
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s || !p) {
      status = ORACLE_ERR_NO_MEMORY;
      free(s);
      free(p);
      continue;
    }
    int32_t prev = anchors ? anchors[r] : 0;
    for (int k = 1; k <= gamma; ++k) {
      if (rank > 0 && (prev < 0 || prev >= V)) {
        status = ORACLE_ERR_INVALID_ARG;
        break;
      }
      draft_scores(&d, r, k, prev, s);
      int x;
      double mrg;
      if (greedy) {
        x = oracle_argmax(s, V, &mrg);
      } else {
        for (int v = 0; v < V; ++v) s[v] *= invT;
      }
      double m, logz;
      oracle_softmax(s, V, p, &m, &logz);
      if (!greedy) x = oracle_sample(p, V, (double)u_draft[(size_t)r * gamma + (k - 1)], &mrg);
      const size_t o = (size_t)r * gamma + (size_t)(k - 1);
      draft_tokens[o] = x;
      if (draft_logp) draft_logp[o] = s[x] - m - logz;
      if (draft_stats) {
        draft_stats[2 * o] = m;
        draft_stats[2 * o + 1] = logz;
      }
      if (margin) margin[o] = mrg;
      prev = x;
    }
    free(s);
    free(p);
  }
  return status;
}

/* ---------------------------------------------------------------- 2a. greedy verify */

/*
 * Greedy verification of the window [x_0, x_1..x_gamma] ("DeepSeek-V4 MTP/NextN 怎样逐步生成
 * 候选", sections 三-四; DSpark section 1): n = the largest i <= l such that x_j equals the
 * target argmax of row j-1 for every j <= i; the emitted block is x_1..x_n followed by the
 * target argmax of row n. out_tokens [R, gamma+1] is padded with -1.
 */
int oracle_verify_greedy(const void* target, int t_dtype, const int32_t* draft_tokens,
                         const int32_t* lengths, int R, int gamma, int V, int32_t* accept_len,
                         int32_t* out_tokens, int32_t* next_anchor) {
  if (R < 0 || gamma < 0 || V < 1) return ORACLE_ERR_INVALID_ARG;
  if (!dtype_ok(t_dtype)) return ORACLE_ERR_UNSUPPORTED_DTYPE;
  if (R == 0) return ORACLE_OK;
  if (!target || (gamma > 0 && !draft_tokens) || !accept_len) return ORACLE_ERR_INVALID_ARG;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < R; ++r) {
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s) {
      status = ORACLE_ERR_NO_MEMORY;
      continue;
    }
    const int l = lengths ? lengths[r] : gamma;
    if (l < 0 || l > gamma) {
      status = ORACLE_ERR_INVALID_ARG;
      free(s);
      continue;
    }
    int n = 0;
    int y = -1;
    for (int i = 0; i <= l; ++i) {
      const size_t row = ((size_t)r * (gamma + 1) + (size_t)i) * (size_t)V;
      for (int v = 0; v < V; ++v) s[v] = (double)elem(target, t_dtype, row + (size_t)v);
      y = oracle_argmax(s, V, NULL);
      if (i == l || draft_tokens[(size_t)r * gamma + i] != y) break;
      n = i + 1;
    }
    accept_len[r] = n;
    if (out_tokens) {
      int32_t* o = out_tokens + (size_t)r * (gamma + 1);
      for (int j = 0; j <= gamma; ++j) o[j] = -1;
      for (int j = 0; j < n; ++j) o[j] = draft_tokens[(size_t)r * gamma + j];
      o[n] = y;
    }
    if (next_anchor) next_anchor[r] = y;
    free(s);
  }
  return status;
}

/* ---------------------------------------------------------------- 2b. rejection verify */

/*
 * Lossless rejection-sampling verification (named in DSpark sections 3 and 9; rule as in the
 * header comment, readings R5 and R6). For k = 1..l: p_d = draft distribution of position k
 * after x_{k-1}, p_t = target row k-1; accept x_k iff oracle_accept_test(u_accept[r,k-1]).
 * At the first rejection k = n+1 draw the output token from norm(max(0, p_t(row n) -
 * p_d(position n+1))) with u_resid[r]; if all l survive draw it from p_t(row l).
 * Diagnostics: accept_margin[r,k-1] = |u - p_t/p_d| for every tested position (NaN where
 * untested), resid_margin[r] = the CDF margin of the final draw.
 */
int oracle_verify_rejection(const void* target, const void* U, int l_dtype, const void* W1,
                            const void* W2, int w_dtype, int rank, const int32_t* anchors,
                            const int32_t* draft_tokens, const float* u_accept,
                            const float* u_resid, float temperature, const int32_t* lengths,
                            int R, int gamma, int V, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* next_anchor, double* accept_margin, double* resid_margin,
                            const uint32_t* mask) {
  if (R < 0 || gamma < 0 || V < 1 || rank < 0) return ORACLE_ERR_INVALID_ARG;
  if (!dtype_ok(l_dtype)) return ORACLE_ERR_UNSUPPORTED_DTYPE;
  if (R == 0) return ORACLE_OK;
  if (!target || !U || !u_resid || !accept_len || !(temperature > 0.0f))
    return ORACLE_ERR_INVALID_ARG;
  if (gamma > 0 && (!draft_tokens || !u_accept)) return ORACLE_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || !anchors || !dtype_ok(w_dtype))) return ORACLE_ERR_INVALID_ARG;
  const double invT = (double)(1.0f / temperature);
  DraftSide d = {U, l_dtype, W1, W2, w_dtype, rank, gamma, V, mask};
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < R; ++r) {
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    double* pd = (double*)malloc(sizeof(double) * (size_t)V);
    double* pt = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s || !pd || !pt || !q) {
      status = ORACLE_ERR_NO_MEMORY;
      free(s); free(pd); free(pt); free(q);
      continue;
    }
    const int l = lengths ? lengths[r] : gamma;
    if (l < 0 || l > gamma) {
      status = ORACLE_ERR_INVALID_ARG;
      free(s); free(pd); free(pt); free(q);
      continue;
    }
    if (accept_margin)
      for (int k = 0; k < gamma; ++k) accept_margin[(size_t)r * gamma + k] = NAN;
    int32_t prev = anchors ? anchors[r] : 0;
    int n = 0, rejected = 0;
    for (int k = 1; k <= l; ++k) {
      const int32_t x = draft_tokens[(size_t)r * gamma + (k - 1)];
      draft_scores(&d, r, k, prev, s);
      for (int v = 0; v < V; ++v) s[v] *= invT;
      oracle_softmax(s, V, pd, NULL, NULL);
      target_probs_row(target, l_dtype, gamma + 1, V, r, k - 1, invT, s, pt, NULL, NULL);
      const double u = (double)u_accept[(size_t)r * gamma + (k - 1)];
      if (accept_margin) accept_margin[(size_t)r * gamma + (k - 1)] = fabs(u - pt[x] / pd[x]);
      if (!oracle_accept_test(u, pd[x], pt[x])) {
        rejected = 1;
        break;
      }
      n = k;
      prev = x;
    }
    double mrg;
    int y;
    if (rejected) {
      /* pd holds position n+1 and pt holds row n (both computed in the last iteration). */
      oracle_residual(pt, pd, V, q);
      y = oracle_sample(q, V, (double)u_resid[r], &mrg);
    } else {
      target_probs_row(target, l_dtype, gamma + 1, V, r, l, invT, s, pt, NULL, NULL);
      y = oracle_sample(pt, V, (double)u_resid[r], &mrg);
    }
    accept_len[r] = n;
    if (out_tokens) {
      int32_t* o = out_tokens + (size_t)r * (gamma + 1);
      for (int j = 0; j <= gamma; ++j) o[j] = -1;
      for (int j = 0; j < n; ++j) o[j] = draft_tokens[(size_t)r * gamma + j];
      o[n] = y;
    }
    if (next_anchor) next_anchor[r] = y;
    if (resid_margin) resid_margin[r] = mrg;
    free(s); free(pd); free(pt); free(q);
  }
  return status;
}

/* ---------------------------------------------------------------- 3a. TV confidence */

/*
 * TV soft labels and prefix survival (DSpark sections 5-6):
 *   c*_k = 1 - 1/2 sum_v |p_d,k(v) - p_t,k-1(v)|, evaluated as sum_v min(p_d,k(v), p_t,k-1(v))
 *   (equal in exact arithmetic), with p_d,k conditioned on the proposed prefix and p_t,k-1 the
 *   aligned target row (reading R5); a_{r,j} = prod_{i<=j} c*_{r,i}, both in fp64.
 */
int oracle_tv_confidence(const void* U, const void* target, int l_dtype, const void* W1,
                         const void* W2, int w_dtype, int rank, const int32_t* anchors,
                         const int32_t* draft_tokens, float temperature, int R, int gamma,
                         int V, double* conf, double* survival, const uint32_t* mask) {
  if (R < 0 || gamma < 0 || V < 1 || rank < 0) return ORACLE_ERR_INVALID_ARG;
  if (!dtype_ok(l_dtype)) return ORACLE_ERR_UNSUPPORTED_DTYPE;
  if (R == 0 || gamma == 0) return ORACLE_OK;
  if (!U || !target || !draft_tokens || !conf || !(temperature > 0.0f))
    return ORACLE_ERR_INVALID_ARG;
  if (rank > 0 && (!W1 || !W2 || !anchors || !dtype_ok(w_dtype))) return ORACLE_ERR_INVALID_ARG;
  const double invT = (double)(1.0f / temperature);
  DraftSide d = {U, l_dtype, W1, W2, w_dtype, rank, gamma, V, mask};
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < R; ++r) {
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    double* pd = (double*)malloc(sizeof(double) * (size_t)V);
    double* pt = (double*)malloc(sizeof(double) * (size_t)V);
    if (!s || !pd || !pt) {
      status = ORACLE_ERR_NO_MEMORY;
      free(s); free(pd); free(pt);
      continue;
    }
    int32_t prev = anchors ? anchors[r] : 0;
    double a = 1.0;
    for (int k = 1; k <= gamma; ++k) {
      draft_scores(&d, r, k, prev, s);
      for (int v = 0; v < V; ++v) s[v] *= invT;
      oracle_softmax(s, V, pd, NULL, NULL);
      target_probs_row(target, l_dtype, gamma + 1, V, r, k - 1, invT, s, pt, NULL, NULL);
      double c = 0.0;
      for (int v = 0; v < V; ++v) c += pd[v] < pt[v] ? pd[v] : pt[v];
      a *= c;
      conf[(size_t)r * gamma + (k - 1)] = c;
      if (survival) survival[(size_t)r * gamma + (k - 1)] = a;
      prev = draft_tokens[(size_t)r * gamma + (k - 1)];
    }
    free(s); free(pd); free(pt);
  }
  return status;
}

/* ---------------------------------------------------------------- 3b. prefix scheduler */

typedef struct {
  float a;
  int r, j;
} Candidate;

/* Order (a desc, r asc, j asc) of reading R7. */
static int candidate_cmp(const void* pa, const void* pb) {
  const Candidate* x = (const Candidate*)pa;
  const Candidate* y = (const Candidate*)pb;
  if (x->a != y->a) return x->a > y->a ? -1 : 1;
  if (x->r != y->r) return x->r < y->r ? -1 : 1;
  return (x->j > y->j) - (x->j < y->j);
}

/*
 * Hardware-aware prefix scheduler (DSpark section 6): choose l_r maximising
 * Theta = tau * SPS(B), B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r} a_{r,j}), by
 * queueing every candidate (r, j) in decreasing survival and scanning the queue length K.
 * Exactness per reading R7. survival [R, gamma] must hold finite values in [0, 1];
 * sps[B] for B = 0..Bmax.
 */
/*
 * Prefix scheduler (DSpark section 6). With capacity < 0 the batch size B = R + K is the
 * Theta-maximising one (smallest K on ties). With capacity >= 0 it is the dynamic top-K of
 * DSpark section 7: the capacity B comes from confidences of an earlier step, and the current
 * candidates are taken in the same queue order up to K = min(capacity - R, R*gamma, Bmax - R)
 * (clamped at 0); theta_out is Theta at that K.
 */
static int schedule_impl(const float* survival, const double* sps, int Bmax, int R, int gamma,
                         int capacity, int32_t* lengths, int32_t* B_out, double* theta_out) {
  if (R < 0 || gamma < 0 || Bmax < R || !sps) return ORACLE_ERR_INVALID_ARG;
  if (R > 0 && (!lengths || (gamma > 0 && !survival))) return ORACLE_ERR_INVALID_ARG;
  const size_t n = (size_t)R * (size_t)gamma;
  for (size_t i = 0; i < n; ++i)
    if (!(survival[i] >= 0.0f && survival[i] <= 1.0f)) return ORACLE_ERR_INVALID_ARG;
  for (int b = 0; b <= Bmax; ++b)
    if (!(sps[b] >= 0.0 && sps[b] < INFINITY)) return ORACLE_ERR_INVALID_ARG;

  Candidate* c = (Candidate*)malloc(sizeof(Candidate) * (n ? n : 1));
  if (!c) return ORACLE_ERR_NO_MEMORY;
  for (int r = 0; r < R; ++r)
    for (int j = 1; j <= gamma; ++j) {
      Candidate* e = &c[(size_t)r * gamma + (j - 1)];
      e->a = survival[(size_t)r * gamma + (j - 1)];
      e->r = r;
      e->j = j;
    }
  qsort(c, n, sizeof(Candidate), candidate_cmp);

  const double two32 = 4294967296.0;
  size_t Kmax = n;
  if ((size_t)(Bmax - R) < Kmax) Kmax = (size_t)(Bmax - R);
  const uint64_t base = (uint64_t)R << 32; /* the "1 +" of every request, in fixed point */
  uint64_t S = 0;
  size_t best_K = 0;
  double best = (double)base * sps[R];
  if (capacity >= 0) { /* fixed capacity: take the first K candidates of the queue */
    const long long want = (long long)capacity - R;
    best_K = want <= 0 ? 0 : ((size_t)want < Kmax ? (size_t)want : Kmax);
    for (size_t K = 1; K <= best_K; ++K) S += (uint64_t)nearbyint((double)c[K - 1].a * two32);
    best = (double)(base + S) * sps[R + best_K];
  } else {
    for (size_t K = 1; K <= Kmax; ++K) {
      S += (uint64_t)nearbyint((double)c[K - 1].a * two32);
      const double theta = (double)(base + S) * sps[R + K];
      if (theta > best) {
        best = theta;
        best_K = K;
      }
    }
  }
  for (int r = 0; r < R; ++r) lengths[r] = 0;
  for (size_t K = 0; K < best_K; ++K) lengths[c[K].r] += 1;
  if (B_out) *B_out = (int32_t)(R + best_K);
  if (theta_out) *theta_out = best / two32; /* tau * SPS(B) in natural units */
  free(c);
  return ORACLE_OK;
}

int oracle_schedule_prefix(const float* survival, const double* sps, int Bmax, int R, int gamma,
                           int32_t* lengths, int32_t* B_out, double* theta_out) {
  return schedule_impl(survival, sps, Bmax, R, gamma, -1, lengths, B_out, theta_out);
}

int oracle_schedule_topk(const float* survival, const double* sps, int Bmax, int R, int gamma,
                         int capacity, int32_t* lengths, int32_t* B_out, double* theta_out) {
  if (capacity < 0) return ORACLE_ERR_INVALID_ARG;
  return schedule_impl(survival, sps, Bmax, R, gamma, capacity, lengths, B_out, theta_out);
}

/*
 * Flattened verify batch (DSpark section 7: tokens of all requests flattened into independent
 * rows, the sequence structure carried by a marker tensor). Request r's 1 + l_r target rows
 * (positions 0..l_r) are packed rows offsets[r] .. offsets[r] + l_r, with offsets[0] = 0 and
 * offsets[r+1] = offsets[r] + 1 + l_r; row_req / row_pos name the request and position of every
 * packed row, -1 for the R*(gamma+1) - offsets[R] rows past the batch.
 */
int oracle_flat_layout(const int32_t* lengths, int R, int gamma, int32_t* offsets,
                       int32_t* row_req, int32_t* row_pos) {
  if (R < 0 || gamma < 0) return ORACLE_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r)
    if (lengths[r] < 0 || lengths[r] > gamma) return ORACLE_ERR_INVALID_ARG;
  long long b = 0;
  offsets[0] = 0;
  for (int r = 0; r < R; ++r) {
    for (int i = 0; i <= lengths[r]; ++i, ++b) {
      row_req[b] = r;
      row_pos[b] = i;
    }
    offsets[r + 1] = (int32_t)b;
  }
  for (long long c = (long long)R * (gamma + 1); b < c; ++b) row_req[b] = row_pos[b] = -1;
  return ORACLE_OK;
}
