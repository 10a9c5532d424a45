/*
 * sdcp_oracle.c - plain, slow CPU oracle of the SDCP verifier's acceptance step.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py (its
 * cpu_baseline leg and its reference arm) load this library.  It shares no code, header
 * or constant with the CUDA path; it is written straight from the definitions below, in
 * fp64, one session after another, with a full sort wherever a filter needs an order.
 *
 * Definitions followed (IETF draft-li-mlc-inference-acceleration-00, "Speculative
 * Decoding Coordination Protocol (SDCP) for Distributed Inference with Multi-Level
 * Caches"):
 *   Section 4.1 (sampling profile): p is the model's next-token distribution after
 *     temperature, top-k and top-p, in that order; temperature 0 selects the most
 *     probable token, ties to the smallest token id.
 *   Section 6.3 ("Preconditions of the rule"): under a rule that needs q, q[i](x[i])
 *     must be non-zero at every position, checked before any random value is drawn.
 *   Section 6.4, Rule 1 (greedy): accept x[i] iff it is argmax p[i] (smallest id on
 *     ties), stop at the first mismatch, then emit argmax p[a+1].
 *   Section 6.4, Rule 2 (speculative sampling): draw r in [0,1), accept iff
 *     r < min(1, p[i](x[i]) / q[i](x[i])); at the first rejection emit a draw from the
 *     normalised residual max(0, p[i] - q[i]); if all M are accepted, a draw from p[M+1].
 *   Section 5.2 (verdict): accepted = a with 0 <= a <= M; emitted tokens.
 *   Table 2: problem types sdcp-bad-proposal, sdcp-limit, sdcp-q-unavailable.
 * Second, informal statement of Rule 2: "Inference: KV Cache, Batching, Speculative
 * Decoding", section "The acceptance rule" (accept loop, residual at the first failure,
 * bonus token after a loop without failure).
 *
 * Readings where the pages leave a step open (each one is listed in the design notes):
 *   - positions are 0-based in the random counter; the rows of session b are the
 *     ragged layout of the C ABI;
 *   - the profile is applied to the draft logits as well, giving q;
 *   - the top-k order is (logit descending, id ascending) on the raw logits;
 *   - top-p keeps the minimal prefix of that order, over the renormalised top-k
 *     distribution, whose cumulative probability is >= top_p_milli/1000 (at least one
 *     token; the crossing token included); top_p_milli = 1000 keeps everything;
 *   - q[i](x[i]) = 0 means: x[i] is outside the kept set or its logit is -inf (a
 *     structural zero, decided without rounding);
 *   - the additional token is the smallest id j whose cumulative weight (ids ascending)
 *     exceeds u * W; if rounding leaves none, the largest j with positive weight; a
 *     residual whose total weight is 0 falls back to p itself;
 *   - random values: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 *     numbers: as easy as 1, 2, 3", SC'11), key = (low, high) 32 bits of the seed,
 *     counter = (position, purpose, round, session_tag), u = first 53 output bits / 2^53;
 *   - NaN, +inf or an all -inf row: no distribution exists; the session is refused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------------- */
/* Interface (mirrors the C ABI's memory layouts; written here again on purpose).      */
/* ---------------------------------------------------------------------------------- */
enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_BAD_PROPOSAL = 1, ORC_LIMIT = 2, ORC_BAD_PARAMS = 3,
       ORC_Q_UNAVAILABLE = 4 };
enum { ORC_MMAX = 64 };
/* A private-use acceptance rule (the draft's registry keeps 192-255 for private use, Section
   10.2): the relaxed rule of "Inference: KV Cache, Batching, Speculative Decoding", section
   on variants of the acceptance rule ("accept if the token is in the target's top-k").
   Acceptance test: x[i] lies in the kept set of p[i] (the target distribution after the
   session's sampling profile; top_k = k gives "in the target's top-k") with a finite logit.
   Additional token: a draw from p[a] (purpose 1), whether at the first rejection or after
   all M (argmax at temperature 0).  A proposal carries tokens only (no q).  It does not
   preserve the target distribution and needs no trust in a drafter's q. */
enum { ORC_RULE_RELAXED = 192 };

typedef struct {
  uint32_t rule_id, temperature_milli, top_k, top_p_milli;
  uint64_t seed;
  uint32_t round, session_tag;
} orc_params;

typedef struct {
  double lmax;        /* largest raw logit */
  double log_s;       /* log sum over the kept set of exp(z_j - z_max) */
  int32_t argmax;     /* smallest id of the largest logit */
  int32_t kept;       /* size of the kept set */
  int32_t k1;         /* size of the top-k set */
  int32_t invalid;    /* 1: NaN, +inf or no finite logit */
  double topp_cum_before; /* cumulative top-p mass before the crossing token (or -1) */
  double topp_cum_at;     /* cumulative top-p mass including the crossing token (or -1) */
  double topp_target;     /* top_p_milli / 1000 (or -1 when top-p is off) */
} orc_row_info;

/* Per-session record of every decision, so that a disagreement can be classified. */
typedef struct {
  int32_t status, a, n_out, extra_mode; /* extra_mode: 0 none, 1 argmax, 2 residual, 3 bonus, 4 residual fell back to p, 5 draw from p at a rejection (relaxed rule) */
  int32_t extra_token, extra_pos, m, pad;
  double u1, W, c_lo, c_hi;          /* draw: uniform, total weight, C_{j-1}, C_j */
  double u0[ORC_MMAX];               /* acceptance uniforms at evaluated positions */
  double ratio[ORC_MMAX];            /* min(1, p/q) at evaluated positions */
  double log_p[ORC_MMAX];            /* log p_i(x_i) */
  double log_q[ORC_MMAX];            /* log q_i(x_i) */
  double topp_margin;                /* smallest relative top-p crossing margin of the rows used */
} orc_detail;

/* ---------------------------------------------------------------------------------- */
/* Philox4x32-10 (Salmon et al., SC'11): ten rounds of the S-box                        */
/*   (c0,c1,c2,c3) -> (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0))   */
/* with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by the Weyl constants          */
/* (0x9E3779B9, 0xBB67AE85) between rounds.                                            */
/* ---------------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* U(seed, round, position, purpose, tag) in [0,1): first 53 bits of the output / 2^53. */
double oracle_uniform(uint64_t seed, uint32_t round, uint32_t position, uint32_t purpose,
                      uint32_t tag) {
  uint32_t ctr[4] = {position, purpose, round, tag};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  uint64_t bits53 = ((uint64_t)w[0] << 21) | (uint64_t)(w[1] >> 11);
  return (double)bits53 * (1.0 / 9007199254740992.0); /* 2^53 */
}

/* The draft's own derivation (Section 6.4, last paragraph): HMAC-SHA-256 keyed with the
   seed over the session identifier, round, 1-based position and purpose (in
   sdcp_oracle_commit.c). */
double oracle_hmac_uniform(uint64_t seed, const uint8_t session[16], uint32_t round, uint32_t i,
                           uint32_t purpose);

/* The verifier's random value for 0-based position `pos` and `purpose`: Philox when sid is
   NULL, else the HMAC derivation with the session's 16-octet identifier sid and the
   1-based position pos + 1. */
static double verifier_uniform(const orc_params* p, const uint8_t* sid, uint32_t pos, uint32_t purpose) {
  if (sid) return oracle_hmac_uniform(p->seed, sid, p->round, pos + 1u, purpose);
  return oracle_uniform(p->seed, p->round, pos, purpose, p->session_tag);
}

/* ---------------------------------------------------------------------------------- */
/* Logit access: bf16 is the upper half of a binary32, so both widen to double exactly. */
/* ---------------------------------------------------------------------------------- */
static double logit_at(const void* row, int dtype, int64_t j) {
  if (dtype == ORC_F32) return (double)((const float*)row)[j];
  uint16_t h = ((const uint16_t*)row)[j];
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/*
 * Relative shift of the top-p target, 0 by default.  The top-p crossing is a decision
 * boundary: where the cumulative mass lies within rounding of P, keeping the crossing
 * token and leaving it out are both faithful to Section 4.1.  The parity tests set a shift
 * of -1e-5 or +1e-5 to form the two readings of such a row; nothing else changes it.
 */
static double g_topp_shift = 0.0;
void oracle_set_topp_shift(double rel) { g_topp_shift = rel; }

/* Sort support: ids ordered by (logit descending, id ascending). */
typedef struct { double l; int32_t id; } orc_pair;
static int cmp_desc(const void* a, const void* b) {
  const orc_pair* x = (const orc_pair*)a;
  const orc_pair* y = (const orc_pair*)b;
  if (x->l > y->l) return -1;
  if (x->l < y->l) return 1;
  return (x->id < y->id) ? -1 : (x->id > y->id);
}

/*
 * The sampling profile of Section 4.1 applied to one row of logits.
 * dist (optional, [V]): the fp64 distribution; kept (optional, [V]): 1 for kept ids.
 * force_k2 >= 1 (a test hook; -1 otherwise) places the top-p crossing at that many tokens
 * instead of where the cumulative mass first reaches P: the parity tests use it, for a row
 * whose crossing lies within rounding of P, to form the distribution of the crossing the
 * GPU chose (info still records the crossing of the definition).
 * Returns 0, or 1 when the row holds NaN, +inf or no finite logit.
 */
static int row_dist_impl(const void* row, int dtype, int64_t V, uint32_t temperature_milli,
                         uint32_t top_k, uint32_t top_p_milli, double* dist, uint8_t* kept,
                         orc_row_info* info, int64_t force_k2) {
  orc_row_info local;
  if (!info) info = &local;
  memset(info, 0, sizeof *info);
  if (V < 1) { info->invalid = 1; return 1; }
  info->topp_cum_before = info->topp_cum_at = info->topp_target = -1.0;
  if (dist) for (int64_t j = 0; j < V; ++j) dist[j] = 0.0;
  if (kept) memset(kept, 0, (size_t)V);

  /* Validity and argmax on the raw logits (ties to the smallest id). */
  double lmax = -INFINITY;
  int32_t amax = -1;
  for (int64_t j = 0; j < V; ++j) {
    double l = logit_at(row, dtype, j);
    if (isnan(l) || l == INFINITY) { info->invalid = 1; return 1; }
    if (l > lmax) { lmax = l; amax = (int32_t)j; }
  }
  if (amax < 0) { info->invalid = 1; return 1; } /* every logit is -inf */
  info->lmax = lmax;
  info->argmax = amax;

  if (temperature_milli == 0) { /* one-hot at the argmax */
    info->kept = 1; info->k1 = 1; info->log_s = 0.0;
    if (dist) dist[amax] = 1.0;
    if (kept) kept[amax] = 1;
    return 0;
  }
  double t = (double)temperature_milli / 1000.0;
  double zmax = lmax / t;

  int filter_k = (top_k != 0 && (int64_t)top_k < V);
  int filter_p = (top_p_milli < 1000);
  if (!filter_k && !filter_p) {
    /* Every token is kept: S = sum_j exp(z_j - z_max), ids ascending. */
    double s = 0.0;
    for (int64_t j = 0; j < V; ++j) s += exp(logit_at(row, dtype, j) / t - zmax);
    info->kept = (int32_t)V; info->k1 = (int32_t)V; info->log_s = log(s);
    if (dist) for (int64_t j = 0; j < V; ++j) dist[j] = exp(logit_at(row, dtype, j) / t - zmax) / s;
    if (kept) memset(kept, 1, (size_t)V);
    return 0;
  }

  /* Order every id by (logit descending, id ascending). */
  orc_pair* ord = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)V);
  for (int64_t j = 0; j < V; ++j) { ord[j].l = logit_at(row, dtype, j); ord[j].id = (int32_t)j; }
  qsort(ord, (size_t)V, sizeof(orc_pair), cmp_desc);

  /* top-k: the first min(k, V) of that order. */
  int64_t k1 = filter_k ? (int64_t)top_k : V;
  double* pi = (double*)malloc(sizeof(double) * (size_t)k1);
  double s1 = 0.0;
  for (int64_t r = 0; r < k1; ++r) { pi[r] = exp(ord[r].l / t - zmax); s1 += pi[r]; }
  for (int64_t r = 0; r < k1; ++r) pi[r] /= s1;

  /* top-p: minimal prefix of the same order whose cumulative probability >= P. */
  int64_t k2 = k1;
  if (filter_p) {
    double target = (double)top_p_milli / 1000.0 * (1.0 + g_topp_shift);
    double cum = 0.0, before = 0.0;
    k2 = k1;
    for (int64_t r = 0; r < k1; ++r) {
      before = cum;
      cum += pi[r];
      if (cum >= target) { k2 = r + 1; break; }
    }
    info->topp_cum_before = before;
    info->topp_cum_at = cum;
    info->topp_target = target;
    if (force_k2 >= 1) k2 = force_k2 < k1 ? force_k2 : k1;
  }

  /* Renormalise over the final kept set (same order of summation). */
  double s2 = 0.0;
  for (int64_t r = 0; r < k2; ++r) s2 += pi[r];
  info->kept = (int32_t)k2;
  info->k1 = (int32_t)k1;
  info->log_s = log(s1) + log(s2); /* sum over the kept set of exp(z - z_max) = s1 * s2 */
  for (int64_t r = 0; r < k2; ++r) {
    if (dist) dist[ord[r].id] = pi[r] / s2;
    if (kept) kept[ord[r].id] = 1;
  }
  free(pi);
  free(ord);
  return 0;
}

int oracle_row_dist(const void* row, int dtype, int64_t V, uint32_t temperature_milli,
                    uint32_t top_k, uint32_t top_p_milli, double* dist, uint8_t* kept,
                    orc_row_info* info) {
  return row_dist_impl(row, dtype, V, temperature_milli, top_k, top_p_milli, dist, kept, info, -1);
}

int oracle_row_dist_forced(const void* row, int dtype, int64_t V, uint32_t temperature_milli,
                           uint32_t top_k, uint32_t top_p_milli, double* dist, uint8_t* kept,
                           orc_row_info* info, int64_t force_k2) {
  return row_dist_impl(row, dtype, V, temperature_milli, top_k, top_p_milli, dist, kept, info,
                       force_k2);
}

/*
 * Statistics of every scored row of a ragged batch, in the row order of the C ABI's
 * row-statistics call: the total + B target rows, then the total draft rows.  Each row is
 * formed by oracle_row_dist under its session's profile; lpx[r] is the natural log of the
 * row's probability of its draft token (target row i < M and draft row i carry x[i]):
 * -inf outside the kept set, NaN for a row without a token or with one outside [0, V).
 * skipped[r] = 1 for rows of sessions whose offsets or top_p_milli make no distribution.
 * Rows are independent; nthreads > 1 forms them on OpenMP threads.
 */
int oracle_row_stats_batch(const void* T, const void* D, int dtype, int64_t V, int32_t B,
                           const int32_t* m_offsets, int64_t total, const int32_t* x,
                           const orc_params* params, orc_row_info* info, double* lpx,
                           int32_t* skipped, int nthreads) {
  if (B < 0 || V < 1 || total < 0 || (dtype != ORC_F32 && dtype != ORC_BF16)) return 1;
  const int64_t R_T = total + B, R = R_T + total;
  size_t esz = (dtype == ORC_F32) ? 4 : 2;
  /* session and draft token of every row */
  int32_t* sess = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
  int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
  for (int64_t r = 0; r < R; ++r) { sess[r] = -1; tok[r] = -1; }
  for (int32_t b = 0; b < B; ++b) {
    int64_t o0 = m_offsets[b], o1 = m_offsets[b + 1];
    if (o0 < 0 || o1 < o0 || o1 > total) continue;
    for (int64_t i = 0; i <= o1 - o0; ++i) {
      sess[o0 + b + i] = b;
      tok[o0 + b + i] = (i < o1 - o0) ? 1 : 0;
    }
    for (int64_t i = 0; i < o1 - o0; ++i) { sess[R_T + o0 + i] = b; tok[R_T + o0 + i] = 1; }
  }
#ifdef _OPENMP
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* dist = (double*)malloc(sizeof(double) * (size_t)V);
    uint8_t* kept = (uint8_t*)malloc((size_t)V);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < R; ++r) {
      memset(&info[r], 0, sizeof info[r]);
      lpx[r] = NAN;
      const int32_t b = sess[r];
      if (b < 0 || params[b].top_p_milli > 1000) { skipped[r] = 1; continue; }
      skipped[r] = 0;
      const int is_target = r < R_T;
      const char* row = is_target ? (const char*)T + (size_t)r * (size_t)V * esz
                                  : (const char*)D + (size_t)(r - R_T) * (size_t)V * esz;
      const orc_params* p = &params[b];
      if (oracle_row_dist(row, dtype, V, p->temperature_milli, p->top_k, p->top_p_milli, dist,
                          kept, &info[r]))
        continue;
      if (tok[r] == 1) {
        const int64_t xi = is_target ? (int64_t)x[r - b] : (int64_t)x[r - R_T];
        if (xi >= 0 && xi < V)
          lpx[r] = (kept[xi] && dist[xi] > 0.0) ? log(dist[xi]) : -INFINITY;
      }
    }
    free(dist);
    free(kept);
  }
  free(sess);
  free(tok);
  return 0;
}

/*
 * Cumulative weights of a draw (ids ascending): w = max(0, p - q) when q is given
 * (the residual of Rule 2), else w = p.  C[j] = w_0 + ... + w_j.  Returns W = C[V-1].
 */
double oracle_draw_cdf(const double* p, const double* q, int64_t V, double* C) {
  double c = 0.0;
  for (int64_t j = 0; j < V; ++j) {
    double w = q ? p[j] - q[j] : p[j];
    if (w < 0.0) w = 0.0;
    c += w;
    C[j] = c;
  }
  return c;
}

/* Inverse-CDF draw: smallest j with C[j] > u * W, else the largest j with w_j > 0. */
static int32_t draw_from(const double* p, const double* q, int64_t V, double u, double* C,
                         double* W_out, double* lo_out, double* hi_out) {
  double W = oracle_draw_cdf(p, q, V, C);
  *W_out = W;
  double target = u * W;
  for (int64_t j = 0; j < V; ++j) {
    if (C[j] > target) {
      *lo_out = (j > 0) ? C[j - 1] : 0.0;
      *hi_out = C[j];
      return (int32_t)j;
    }
  }
  for (int64_t j = V - 1; j >= 0; --j) {
    double prev = (j > 0) ? C[j - 1] : 0.0;
    if (C[j] > prev) { *lo_out = prev; *hi_out = C[j]; return (int32_t)j; }
  }
  *lo_out = *hi_out = 0.0;
  return -1;
}

/* The draw alone (exported for its tests): token for uniform u, weights from p (and q). */
int32_t oracle_draw(const double* p, const double* q, int64_t V, double u) {
  double* C = (double*)malloc(sizeof(double) * (size_t)V);
  double W, lo, hi;
  int32_t j = draw_from(p, q, V, u, C, &W, &lo, &hi);
  free(C);
  return j;
}

static double topp_margin_of(const orc_row_info* in) {
  if (in->topp_target < 0.0) return INFINITY;
  double m1 = fabs(in->topp_cum_at - in->topp_target);
  double m2 = fabs(in->topp_cum_before - in->topp_target);
  double m = m1 < m2 ? m1 : m2;
  return m / in->topp_target;
}

/* One session, Sections 6.3 and 6.4. */
static void verify_session(const void* T, const void* D, int dtype, int64_t V,
                           const int32_t* m_offsets, int64_t total_drafts, int32_t b,
                           const int32_t* x, const orc_params* prm, const uint8_t* sid,
                           const int32_t* force, int64_t R_T, const float* QR,
                           int32_t* accepted, int32_t* n_out,
                           int32_t* out_tokens, int32_t* status, orc_detail* det) {
  size_t esz = (dtype == ORC_F32) ? 4 : 2;
  orc_detail dl;
  if (!det) det = &dl;
  memset(det, 0, sizeof *det);
  det->extra_token = -1; det->extra_pos = -1; det->topp_margin = INFINITY;
  for (int i = 0; i < ORC_MMAX; ++i) det->u0[i] = det->ratio[i] = det->log_p[i] = det->log_q[i] = NAN;

  int64_t off0 = m_offsets[b], off1 = m_offsets[b + 1];
  int offsets_ok = (off0 >= 0 && off1 >= off0 && off1 <= total_drafts);
  int64_t M = off1 - off0;
  det->m = (int32_t)M;
  int st = ORC_OK;
  if (prm->rule_id != 1 && prm->rule_id != 2 && prm->rule_id != ORC_RULE_RELAXED) st = ORC_BAD_PARAMS;
  else if (prm->top_p_milli > 1000) st = ORC_BAD_PARAMS;
  else if (!offsets_ok) st = ORC_BAD_PARAMS;
  else if (M < 1 || M > ORC_MMAX) st = ORC_LIMIT;
  else if (prm->rule_id == 2 && D == NULL && QR == NULL) st = ORC_Q_UNAVAILABLE;
  else {
    for (int64_t i = 0; i < M; ++i)
      if (x[off0 + i] < 0 || x[off0 + i] >= V) { st = ORC_BAD_PROPOSAL; break; }
  }
  int rule2 = (prm->rule_id == 2);
  int relaxed = (prm->rule_id == ORC_RULE_RELAXED);
  uint32_t tm = prm->temperature_milli;
#define TROW(i) ((const char*)T + (size_t)(off0 + b + (i)) * (size_t)V * esz)
#define DROW(i) ((const char*)D + (size_t)(off0 + (i)) * (size_t)V * esz)
  /* forced top-p crossings (test hook), indexed like the C ABI's row statistics:
     target rows first, then the draft rows from R_T = total_drafts + B */
#define FT(i) (force ? (int64_t)force[off0 + b + (i)] : -1)
#define FD(i) (force ? (int64_t)force[R_T + off0 + (i)] : -1)

  /* Every scored row is formed before any draw: p for the M+1 target rows, q for the
     M draft rows (Rule 2).  Rule 1 needs only the argmax of the raw scores; the relaxed
     rule needs p's kept sets. */
  orc_row_info* pin = NULL; orc_row_info* qin = NULL;
  uint8_t** pk = NULL; uint8_t** qk = NULL;
  if (st == ORC_OK) {
    pin = (orc_row_info*)calloc((size_t)(M + 1), sizeof(orc_row_info));
    pk = (uint8_t**)calloc((size_t)(M + 1), sizeof(uint8_t*));
    for (int64_t i = 0; i <= M && st == ORC_OK; ++i) {
      if (rule2 || relaxed) {
        pk[i] = (uint8_t*)malloc((size_t)V);
        if (row_dist_impl(TROW(i), dtype, V, tm, prm->top_k, prm->top_p_milli, NULL,
                          pk[i], &pin[i], FT(i)))
          st = ORC_BAD_PARAMS;
      } else if (oracle_row_dist(TROW(i), dtype, V, 0, 0, 1000, NULL, NULL, &pin[i])) {
        st = ORC_BAD_PARAMS;
      }
      double mg = topp_margin_of(&pin[i]);
      if (mg < det->topp_margin) det->topp_margin = mg;
    }
    if (st == ORC_OK && rule2 && QR) {
      /* q given as rows of probabilities (Section 5.2 q_rows): used as given, no profile.
         A value that is not a probability (NaN, infinite, negative) at x: no distribution;
         q(x) = 0: the precondition fails (Section 6.3). */
      for (int64_t i = 0; i < M && st == ORC_OK; ++i) {
        double qx = (double)QR[(size_t)(off0 + i) * (size_t)V + (size_t)x[off0 + i]];
        if (isnan(qx) || isinf(qx) || qx < 0.0) st = ORC_BAD_PARAMS;
      }
      for (int64_t i = 0; i < M && st == ORC_OK; ++i)
        if (QR[(size_t)(off0 + i) * (size_t)V + (size_t)x[off0 + i]] == 0.0f) st = ORC_BAD_PROPOSAL;
    } else if (st == ORC_OK && rule2) {
      qin = (orc_row_info*)calloc((size_t)M, sizeof(orc_row_info));
      qk = (uint8_t**)calloc((size_t)M, sizeof(uint8_t*));
      for (int64_t i = 0; i < M && st == ORC_OK; ++i) {
        qk[i] = (uint8_t*)malloc((size_t)V);
        if (row_dist_impl(DROW(i), dtype, V, tm, prm->top_k, prm->top_p_milli, NULL,
                          qk[i], &qin[i], FD(i)))
          st = ORC_BAD_PARAMS;
        double mg = topp_margin_of(&qin[i]);
        if (mg < det->topp_margin) det->topp_margin = mg;
      }
      /* Precondition (Section 6.3): q_i(x_i) != 0 at every position, before any draw.
         A zero is structural: x outside the kept set of q, or a -inf logit. */
      for (int64_t i = 0; i < M && st == ORC_OK; ++i) {
        int32_t xi = x[off0 + i];
        if (!qk[i][xi] || logit_at(DROW(i), dtype, xi) == -INFINITY) st = ORC_BAD_PROPOSAL;
      }
    }
  }

  int64_t a = 0;
  int32_t extra = -1;
  if (st == ORC_OK && relaxed) {
    /* The relaxed rule: accept while x_i is in the kept set of p_i (finite logit); the
       additional token is a draw from p_a. */
    while (a < M && pk[a][x[off0 + a]] && logit_at(TROW(a), dtype, x[off0 + a]) != -INFINITY) ++a;
    double* pa = (double*)malloc(sizeof(double) * (size_t)V);
    double* C = (double*)malloc(sizeof(double) * (size_t)V);
    row_dist_impl(TROW(a), dtype, V, tm, prm->top_k, prm->top_p_milli, pa, NULL, NULL, FT(a));
    double u1 = verifier_uniform(prm, sid, (uint32_t)a, 1);
    det->u1 = u1;
    extra = draw_from(pa, NULL, V, u1, C, &det->W, &det->c_lo, &det->c_hi);
    det->extra_mode = (a < M) ? 5 : 3;
    free(pa); free(C);
  } else if (st == ORC_OK && !rule2) {
    /* Rule 1: accept while x_i is the argmax of target row i; emit argmax of row a. */
    while (a < M && x[off0 + a] == pin[a].argmax) ++a;
    extra = pin[a].argmax;
    det->extra_mode = 1;
  } else if (st == ORC_OK) {
    /* Rule 2, positions in order: accept iff u < min(1, p/q).  The ratio comes from
       log p - log q, so that no underflow of p or q decides it. */
    double t = (double)tm / 1000.0;
    for (a = 0; a < M; ++a) {
      int32_t xi = x[off0 + a];
      double lp, lq;
      if (QR) { /* q(x) as given */
        double lpx = logit_at(TROW(a), dtype, xi);
        if (tm == 0) lp = (xi == pin[a].argmax) ? 0.0 : -INFINITY;
        else lp = (pk[a][xi] && lpx != -INFINITY) ? lpx / t - pin[a].lmax / t - pin[a].log_s : -INFINITY;
        lq = log((double)QR[(size_t)(off0 + a) * (size_t)V + (size_t)xi]);
      } else if (tm == 0) { /* one-hot rows; q(x) = 1 by the precondition */
        lp = (xi == pin[a].argmax) ? 0.0 : -INFINITY;
        lq = 0.0;
      } else {
        double lpx = logit_at(TROW(a), dtype, xi);
        double lqx = logit_at(DROW(a), dtype, xi);
        lp = (pk[a][xi] && lpx != -INFINITY) ? lpx / t - pin[a].lmax / t - pin[a].log_s
                                             : -INFINITY;
        lq = lqx / t - qin[a].lmax / t - qin[a].log_s;
      }
      double ratio = (lp == -INFINITY) ? 0.0 : exp(lp - lq);
      if (ratio > 1.0) ratio = 1.0;
      double u = verifier_uniform(prm, sid, (uint32_t)a, 0);
      det->log_p[a] = lp; det->log_q[a] = lq; det->u0[a] = u; det->ratio[a] = ratio;
      if (!(u < ratio)) break; /* first rejection */
    }
    /* The additional token: residual at the first rejection, else the bonus from p_M. */
    double* pa = (double*)malloc(sizeof(double) * (size_t)V);
    double* qa = (a < M) ? (double*)malloc(sizeof(double) * (size_t)V) : NULL;
    double* C = (double*)malloc(sizeof(double) * (size_t)V);
    row_dist_impl(TROW(a), dtype, V, tm, prm->top_k, prm->top_p_milli, pa, NULL, NULL, FT(a));
    if (qa && QR) {
      for (int64_t j = 0; j < V; ++j) qa[j] = (double)QR[(size_t)(off0 + a) * (size_t)V + (size_t)j];
    } else if (qa) {
      row_dist_impl(DROW(a), dtype, V, tm, prm->top_k, prm->top_p_milli, qa, NULL, NULL, FD(a));
    }
    double u1 = verifier_uniform(prm, sid, (uint32_t)a, 1);
    det->u1 = u1;
    if (qa) {
      extra = draw_from(pa, qa, V, u1, C, &det->W, &det->c_lo, &det->c_hi);
      det->extra_mode = 2;
      if (!(det->W > 0.0)) { /* residual mass lost to rounding: draw from p itself */
        extra = draw_from(pa, NULL, V, u1, C, &det->W, &det->c_lo, &det->c_hi);
        det->extra_mode = 4;
      }
    } else {
      extra = draw_from(pa, NULL, V, u1, C, &det->W, &det->c_lo, &det->c_hi);
      det->extra_mode = 3;
    }
    free(pa); free(qa); free(C);
  }
#undef TROW
#undef DROW
#undef FT
#undef FD

  /* Outputs (Section 5.2): a accepted tokens, then the additional token. */
  status[b] = st;
  int64_t slot0 = off0 + b;
  if (st == ORC_OK) {
    accepted[b] = (int32_t)a;
    n_out[b] = (int32_t)(a + 1);
    for (int64_t j = 0; j < a; ++j) out_tokens[slot0 + j] = x[off0 + j];
    out_tokens[slot0 + a] = extra;
    for (int64_t j = a + 1; j <= M; ++j) out_tokens[slot0 + j] = -1;
  } else {
    accepted[b] = 0;
    n_out[b] = 0;
    if (offsets_ok)
      for (int64_t j = 0; j <= M; ++j) out_tokens[slot0 + j] = -1;
  }
  det->status = st;
  det->a = (int32_t)a;
  det->n_out = n_out[b];
  det->extra_token = extra;
  det->extra_pos = (int32_t)a;

  if (pk) { for (int64_t i = 0; i <= M; ++i) free(pk[i]); free(pk); }
  if (qk) { for (int64_t i = 0; i < M; ++i) free(qk[i]); free(qk); }
  free(pin); free(qin);
}

/*
 * The whole ragged batch; sessions are independent (Section 6.3 "Scoring" batches
 * proposals of many sessions), so nthreads > 1 runs them on OpenMP threads.
 * detail (optional, [B]) records every decision of every session.
 */
/* session_ids (optional, [B][16]) selects the HMAC derivation of the random values;
   force_kept (optional, [2 total + B], row order of the C ABI's row statistics) is the
   parity tests' hook that places top-p crossings (-1: where the definition puts them);
   q_rows (optional, [total][V] binary32) gives q as rows of probabilities (Section 5.2
   q_rows) instead of draft logits with the profile. */
int oracle_verify_batch_rng(const void* T, const void* D, int dtype, int64_t V, int32_t B,
                            const int32_t* m_offsets, int64_t total_drafts,
                            const int32_t* draft_tokens, const orc_params* params,
                            const uint8_t* session_ids, const int32_t* force_kept,
                            const float* q_rows, int32_t* accepted, int32_t* n_out,
                            int32_t* out_tokens, int32_t* status, orc_detail* detail,
                            int nthreads) {
  if (B < 0 || V < 1 || (dtype != ORC_F32 && dtype != ORC_BF16)) return 1;
  if (!T || !m_offsets || !draft_tokens || !params) return 1;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int32_t b = 0; b < B; ++b)
    verify_session(T, D, dtype, V, m_offsets, total_drafts, b, draft_tokens, &params[b],
                   session_ids ? session_ids + 16 * (size_t)b : NULL, force_kept,
                   total_drafts + B, q_rows, accepted, n_out, out_tokens, status,
                   detail ? &detail[b] : NULL);
  return 0;
}

/* The whole batch with Philox random values. */
int oracle_verify_batch(const void* T, const void* D, int dtype, int64_t V, int32_t B,
                        const int32_t* m_offsets, int64_t total_drafts,
                        const int32_t* draft_tokens, const orc_params* params,
                        int32_t* accepted, int32_t* n_out, int32_t* out_tokens,
                        int32_t* status, orc_detail* detail, int nthreads) {
  return oracle_verify_batch_rng(T, D, dtype, V, B, m_offsets, total_drafts, draft_tokens,
                                 params, NULL, NULL, NULL, accepted, n_out, out_tokens, status,
                                 detail, nthreads);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
