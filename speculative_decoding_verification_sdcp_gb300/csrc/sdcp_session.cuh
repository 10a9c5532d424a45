// sdcp_session.cuh - completion of one session of the acceptance step (SDCP draft
// draft-li-mlc-inference-acceleration-00: Section 6.3 "Preconditions of the rule",
// Section 6.4 Rules 1 and 2, and the verdict fields of Section 5.2) by a thread-block
// cluster of C CTAs (C = 1 .. 8).
//
// Verdict (one warp per CTA, the same in every CTA): the M acceptance tests from the row
// statistics (one lane per position, fp64 ratio, Philox uniform of purpose 0), the first
// rejection a by ballot; rank 0 writes every output slot that needs no draw.  Rule 2 then
// draws one token (purpose 1): from the residual max(0, p_a - q_a) when a < M, else from
// p_M, as the smallest id whose cumulative weight exceeds u * W.  Each CTA owns a slice of
// the row's 256-id segments and sums the weights of each segment (warps own contiguous
// runs of segments, read with batches of coalesced 16-byte loads); the slice totals are
// exchanged through distributed shared memory, the CTA whose slice holds u * W scans its
// segment sums, and one warp walks the segment that holds it.  Where a top-k / top-p cut
// falls inside one value, the id bound of its kept tokens is found first the same way
// (counts per segment, exchange, walk).
#pragma once

#include <type_traits>

#include "sdcp_device.cuh"
#include "sdcp_sha256.cuh"

namespace sdcp {

constexpr int kSegIds = 32 * kEpt;  // ids per segment: 8 per lane
constexpr int kSegCap = 2048;       // segment-group sums held in shared memory
constexpr int kTieCap = 64;         // tokens on a cut value held per warp (single-pass draw)
constexpr int kTieStages = 64;      // stages whose cut-value counts are kept (single-pass draw)
constexpr int kDrawHalf = 16384;    // bytes of p (and of q) per stage of the streamed draw
constexpr int kDrawStages = 2;      // stages of the streamed draw's ring
constexpr int kKeptW = 128;         // candidates (p's kept tokens) per warp: kept-set draw
constexpr int kQCutW = 32;          // q's cut-value ids per warp: kept-set draw
constexpr int kMaxCluster = 8;     // CTAs per session cluster at most
constexpr int kKeptSliceBytes = 65536;  // largest slice of p a CTA scans with plain loads
#define kNaN64 __longlong_as_double(0x7FF8000000000000ll)  // "the draw could not decide"

// A token whose keptness depends on its rank among the tokens of a cut value (p's or q's).
struct TieEntry {
  int id;
  float P, Q;  // its p and q weights were it kept
  int code;    // bit 0: on p's cut value; bit 1: on q's cut value; bits 8..: stage
  int lp, lq;  // its index among p's (q's) cut-value tokens of its stage and warp
};

// The kept-set draw's lists (per warp, in id order) and its per-CTA results.
struct KeptSmem {
  int id[kWarps][kKeptW];     // p's candidates: tokens at or above p's cut value
  float v[kWarps][kKeptW];    // their p logits
  float r[kWarps][kKeptW];    // their weights (first their q logits)
  float pre[kWarps][kKeptW];  // running weight sums before them, within the warp
  int qid[kWarps][kQCutW];    // q's cut-value tokens
  int n[kWarps], qn[kWarps], pc[kWarps], best[kWarps], last[kWarps];
  float wsum[kWarps], wbase[kWarps];
  int cta_ovf, cta_pc, cta_qc, tie_p, tie_q;
};

// Shared memory of one CTA of a session's cluster (the streamed draw's ring is dynamic).
struct SessSmem {
  uint64_t full[kDrawStages], empty[kDrawStages];
  float seg[kSegCap];  // per segment group of the CTA's slice: weight sums or tie counts
  union {
    TieEntry ties[kWarps][kTieCap];  // per warp, in id order within each stage
    KeptSmem kept;                   // the kept-set draw
  };
  int tie_n[kWarps];
  uint8_t plist[kWarps][kDrawHalf / kEpt / kWarps / 2];  // per warp: the stage's pieces to weigh
  int tsc_p[kTieStages][kWarps], tsc_q[kTieStages][kWarps];  // cut-value tokens per stage, warp
  int overflow;
  long long cta_np, cta_nq;  // cut-value tokens of the slice (read by the cluster)
  int cta_ovf;
  int tie_p_cand, tie_q_cand;  // id bounds found in this slice (read by the cluster)
  float fscr[2 * 32 + 4];
  long long lscr[2 * 32 + 4];
  double cta_sum;      // the slice's total weight (read by the cluster)
  long long cta_cnt;   // the slice's tie count (read by the cluster)
  double owner_base;
  long long owner_pre, owner_carry;
  long long result;    // a tie id found by this CTA (read by the cluster)
  int st, a, draw;
  uint32_t ring_uses;  // stages of the draw ring used so far (slot and barrier parity)
  // local copies of the cluster's per-CTA values (lane r of warp 0 reads rank r, so each
  // value crosses the cluster once per CTA, not once per thread)
  double cv_sum[kMaxCluster];
  long long cv_n0[kMaxCluster], cv_n1[kMaxCluster];
  int cv_ovf[kMaxCluster], cv_i0[kMaxCluster], cv_i1[kMaxCluster];
  long long cv_res;
  // the draw's target over the cluster, worked out by thread 0 alone (fp64 arithmetic runs at
  // a small fraction of the fp32 rate on this GPU, so it is kept off the other threads)
  double d_W, d_target, d_base;
  float d_tloc;
  int d_owner, d_bad;
  RowStat stash[2];  // the statistics of target row a and draft row a (from the verdict)
};

// Lanes r < C of warp 0: dst[r] = the value at src in the shared memory of cluster rank r.
// Between two cluster barriers: the first publishes src, the second orders dst before its
// readers (and keeps every CTA's src alive until the cluster has read it).
template <typename V>
__device__ __forceinline__ void cluster_copy(cg::cluster_group& cluster, V* src, V* dst) {
  if (threadIdx.x < cluster.num_blocks()) dst[threadIdx.x] = *cluster.map_shared_rank(src, threadIdx.x);
}

// Verdict of a session: status, accepted count, and whether Rule 2 still draws a token.
struct Verdict {
  int st, a;
  bool draw;
};

// The verifier's random value of session b for 0-based position pos and purpose (0: the
// acceptance test, 1: the additional token), by the call's generator: Philox with counter
// (pos, purpose, round, session_tag), or the draft's HMAC-SHA-256 derivation with the
// session's 16-octet identifier and the 1-based position pos + 1.
__device__ __forceinline__ double session_uniform(const SessIO& A, int32_t b, const sdcp_session_params& P,
                                                  uint32_t pos, uint32_t purpose) {
  if (A.rng == SDCP_RNG_HMAC_SHA256) {
    const uint8_t* s = A.session_ids + (size_t)16 * (size_t)b;
    uint32_t sid[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
      sid[w] = ((uint32_t)s[4 * w] << 24) | ((uint32_t)s[4 * w + 1] << 16) | ((uint32_t)s[4 * w + 2] << 8) |
               (uint32_t)s[4 * w + 3];
    return hmac_uniform(P.seed, sid, P.round, pos + 1u, purpose);
  }
  return verifier_uniform(P, pos, purpose);
}

// A row statistic as the other CTAs of the grid left it in L2 (never a stale L1 line).
__device__ __forceinline__ RowStat load_stat(const RowStat* p) {
  union { float4 v[2]; RowStat s; } u;
  u.v[0] = __ldcg(reinterpret_cast<const float4*>(p));
  u.v[1] = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  return u.s;
}

// ---------------------------------------------------------------------------------
// Verdict (one full warp; every lane returns the same value).  Writes status, accepted,
// n_out and every output slot except the drawn token, and leaves the statistics of target
// row a and draft row a in stash[0], stash[1] (the draw's rows; the warp has read them).
// ---------------------------------------------------------------------------------
static __device__ Verdict session_verdict(const SessIO& A, int32_t b, bool write, RowStat* stash) {
  const int lane = threadIdx.x & 31;
  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const bool offsets_ok = off0 >= 0 && off1 >= off0 && off1 <= A.total && A.m_offsets[0] == 0 &&
                          (int64_t)A.m_offsets[A.B] == A.total;
  const int64_t M = off1 - off0;
  const int64_t R_T = A.total + A.B;
  const int64_t V = A.V;
  const bool rule2 = (P.rule_id == 2u);
  const bool relaxed = (P.rule_id == SDCP_RULE_RELAXED_TOP_K);
  const uint32_t tm = P.temperature_milli;
  const float c = (tm == 0u) ? 0.f : profile_c(tm);
  int st = SDCP_S_OK;
  if ((P.rule_id != 1u && P.rule_id != 2u && !relaxed) || P.top_p_milli > 1000u) st = SDCP_S_BAD_PARAMS;
  else if (!offsets_ok) st = SDCP_S_BAD_PARAMS;
  else if (M < 1 || M > SDCP_MAX_M) st = SDCP_S_LIMIT;
  else if (rule2 && A.draft == nullptr && A.q_rows == nullptr) st = SDCP_S_Q_UNAVAILABLE;
  if (st == SDCP_S_OK && __ldcg(A.error) != 0u) st = SDCP_S_INTERNAL;
  int a = 0;
  int32_t xr[2] = {-1, -1};
  RowStat kp0{}, kp1{}, kq0{}, kq1{}, sl{};  // this lane's rows (positions lane, lane + 32)
  if (st == SDCP_S_OK) {
    bool range_bad = false, row_bad = false, q_zero = false;
    bool rej[2] = {false, false};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      if (i < M) {
        const int32_t x = A.tokens[off0 + i];
        xr[h] = x;
        if (x < 0 || (int64_t)x >= V) range_bad = true;
        const RowStat sp = load_stat(A.stats + off0 + b + i);
        if (h == 0) kp0 = sp; else kp1 = sp;
        if (sp.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
        if (rule2 && A.q_rows != nullptr) {
          // q as given (Section 5.2 q_rows): q(x) must be a probability, and not zero
          float qx = 0.f;
          if (x >= 0 && (int64_t)x < V) qx = __ldg(A.q_rows + (size_t)(off0 + i) * (size_t)V + (size_t)x);
          if (!(qx >= 0.f) || qx == INFINITY) row_bad = true;
          if (qx == 0.f) q_zero = true;
          if (tm == 0u) {
            rej[h] = (x != sp.argmax);
          } else {
            // p(x) / q(x) = 2^(dlx_p c) / S_p / q(x)
            float ratio = 0.f;
            if ((sp.flags & SDCP_ROW_X_KEPT) && qx > 0.f && qx < INFINITY)
              ratio = __fdiv_rn(ex2(sp.dlx * c) * __fdiv_rn(1.f, sp.s), qx);
            ratio = ratio > 1.f ? 1.f : ratio;
            const double u = session_uniform(A, b, P, (uint32_t)i, 0u);
            rej[h] = !(u < (double)ratio);
          }
        } else if (rule2) {
          const RowStat sq = load_stat(A.stats + R_T + off0 + i);
          if (h == 0) kq0 = sq; else kq1 = sq;
          if (sq.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
          if (!(sq.flags & SDCP_ROW_X_KEPT)) q_zero = true;
          if (tm == 0u) {
            rej[h] = (x != sp.argmax);
          } else {
            // p(x) / q(x) = 2^((dlx_p - dlx_q) c) * S_q / S_p, with the c of the row statistics
            float ratio = 0.f;
            if (sp.flags & SDCP_ROW_X_KEPT)
              ratio = ex2((sp.dlx - sq.dlx) * c) * __fdiv_rn(sq.s, sp.s);
            ratio = ratio > 1.f ? 1.f : ratio;
            const double u = session_uniform(A, b, P, (uint32_t)i, 0u);
            rej[h] = !(u < (double)ratio);
          }
        } else if (relaxed) {  // x must lie in p's kept set (a finite logit)
          rej[h] = !(sp.flags & SDCP_ROW_X_KEPT);
        } else {
          rej[h] = (x != sp.argmax);
        }
      }
    }
    if (lane == 0) {  // the bonus / last target row must be valid too
      sl = load_stat(A.stats + off0 + b + M);
      if (sl.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
    }
    if (__any_sync(0xFFFFFFFFu, range_bad)) st = SDCP_S_BAD_PROPOSAL;
    else if (__any_sync(0xFFFFFFFFu, row_bad)) st = SDCP_S_BAD_PARAMS;
    else if (rule2 && __any_sync(0xFFFFFFFFu, q_zero)) st = SDCP_S_BAD_PROPOSAL;
    const unsigned r0 = __ballot_sync(0xFFFFFFFFu, rej[0]);
    const unsigned r1 = __ballot_sync(0xFFFFFFFFu, rej[1]);
    a = r0 ? (__ffs(r0) - 1) : (r1 ? 32 + __ffs(r1) - 1 : (int)M);
    if (a > M) a = (int)M;
    // the rows of position a, from the lane that read them
    const int owner = (a < M) ? (a & 31) : 0;
    if (lane == owner) {
      stash[0] = (a == M) ? sl : ((a < 32) ? kp0 : kp1);
      stash[1] = (a < 32) ? kq0 : kq1;
    }
    __syncwarp();
  }
  const bool ok = (st == SDCP_S_OK);
  const bool draw = ok && (rule2 || relaxed) && tm != 0u;
  if (write && lane == 0) {
    A.status[b] = st;
    A.accepted[b] = ok ? a : 0;
    A.n_out[b] = ok ? a + 1 : 0;
  }
  if (write && offsets_ok) {
    const int64_t slot0 = off0 + b;
    int32_t extra = -1;
    if (ok && !draw) extra = stash[0].argmax;
#pragma unroll
    for (int h = 0; h < 3; ++h) {
      const int64_t j = lane + 32 * h;
      if (j > M) break;
      int32_t v = -1;
      if (ok) {
        if (j < a) v = xr[h < 2 ? h : 1];
        else if (j == a) {
          if (draw) continue;  // written by the draw
          v = extra;
        }
      }
      A.out_tokens[slot0 + j] = v;
    }
  }
  return Verdict{ok ? SDCP_S_OK : st, a, draw};
}

// ---------------------------------------------------------------------------------
// The draw.
// ---------------------------------------------------------------------------------

// Weight of token j: p_j = 2^((l_j - lmax) c) / S over the kept set, where c = log2(e) 1000/T
// (l_j - lmax is exact near the maximum, where the mass is, so the weights carry no shared
// rounding of a large exponent offset; 1/S is one correctly rounded division); kept = value
// above the cut value, or the cut value and id <= tie (values compare as floats: -0 and +0
// are one value, as their order keys are).
struct DrawRow {
  float c, lmax, inv_s;
  float thr;  // the cut value (-inf: no cut)
  int tie;    // INT_MAX: every token of the cut value is kept
};
__device__ __forceinline__ float row_weight(const DrawRow& r, float v) {
  return ex2((v - r.lmax) * r.c) * r.inv_s;
}
template <bool FILT>
__device__ __forceinline__ float draw_weight(const DrawRow& r, uint32_t bits, int j) {
  const float v = __uint_as_float(bits);
  const float e = row_weight(r, v);
  if (!FILT) return e;
  return (v > r.thr || (v == r.thr && j <= r.tie)) ? e : 0.f;
}

// Raw words of the 8 ids [j0, j0 + 8) of a row: bf16 one 16-byte vector, fp32 two.  Ids at
// or past `end` (and every id of a group that is not 16-byte aligned) are read one by one,
// those past `end` as `fill`.
template <typename T> struct Raw8 { static constexpr int W = (sizeof(T) == 2) ? 1 : 2; uint4 v[W]; };
// q's element type in a draw: the batch's logits type, or binary32 when q is given as rows of
// probabilities (QR: Section 5.2 q_rows, used as given)
template <typename T, bool QR> using QElem = typename std::conditional<QR, float, T>::type;

// fill: the bits read for ids at or past `end` (-inf for logits, +0 for q given as
// probabilities: both are probability 0).
template <typename T>
__device__ __forceinline__ void load_raw8(const T* row, bool aligned16, int end, int j0, Raw8<T>& r,
                                          uint32_t fill = 0xFF800000u) {
  if (aligned16 && j0 + kEpt <= end) {
#pragma unroll
    for (int w = 0; w < Raw8<T>::W; ++w) r.v[w] = __ldg(reinterpret_cast<const uint4*>(row + j0) + w);
  } else {
    uint32_t b[kEpt];
#pragma unroll
    for (int e = 0; e < kEpt; ++e) b[e] = (j0 + e < end) ? load_bits(row, j0 + e) : fill;
    if (sizeof(T) == 2) {
      r.v[0] = make_uint4((b[0] >> 16) | (b[1] & 0xFFFF0000u), (b[2] >> 16) | (b[3] & 0xFFFF0000u),
                          (b[4] >> 16) | (b[5] & 0xFFFF0000u), (b[6] >> 16) | (b[7] & 0xFFFF0000u));
    } else {
      r.v[0] = make_uint4(b[0], b[1], b[2], b[3]);
      r.v[Raw8<T>::W - 1] = make_uint4(b[4], b[5], b[6], b[7]);
    }
  }
}
template <typename T>
__device__ __forceinline__ void unpack_raw8(const Raw8<T>& r, uint32_t (&b)[kEpt]) {
  if (sizeof(T) == 2) {
    uint32_t t[8];
    Elem<__nv_bfloat16>::unpack(r.v[0], t);
#pragma unroll
    for (int e = 0; e < kEpt; ++e) b[e] = t[e];
  } else {
    b[0] = r.v[0].x; b[1] = r.v[0].y; b[2] = r.v[0].z; b[3] = r.v[0].w;
    b[4] = r.v[Raw8<T>::W - 1].x; b[5] = r.v[Raw8<T>::W - 1].y; b[6] = r.v[Raw8<T>::W - 1].z; b[7] = r.v[Raw8<T>::W - 1].w;
  }
}

// Whether some value of a piece is >= thr (bf16: packed maxima; -inf pads count as below).
template <typename T>
__device__ __forceinline__ bool piece_reaches(const Raw8<T>& r, float thr) {
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&r.v[0].x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&r.v[0].y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&r.v[0].z),
                                     *reinterpret_cast<const __nv_bfloat162*>(&r.v[0].w));
    const __nv_bfloat162 ab = __hmax2(a, b);
    const uint32_t m = *reinterpret_cast<const uint32_t*>(&ab);
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u)) >= thr;
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < Raw8<T>::W; ++w)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(r.v[w].x), __uint_as_float(r.v[w].y)),
                         fmaxf(__uint_as_float(r.v[w].z), __uint_as_float(r.v[w].w))));
    return m >= thr;
  }
}
// Whether some value of a piece equals v.
template <typename T>
__device__ __forceinline__ bool piece_holds(const Raw8<T>& r, float v) {
  uint32_t b[kEpt];
  unpack_raw8<T>(r, b);
  bool h = false;
#pragma unroll
  for (int e = 0; e < kEpt; ++e) h |= (__uint_as_float(b[e]) == v);
  return h;
}

// f(bits of p, bits of q, e) for the 8 elements of one lane piece, in id order, straight from
// the loaded words (no per-element arrays: they would not fit the register budget).
template <typename T, typename F>
__device__ __forceinline__ void for_each8(const Raw8<T>& rp, const Raw8<T>& rq, F f) {
  if constexpr (sizeof(T) == 2) {
    f(rp.v[0].x << 16, rq.v[0].x << 16, 0); f(rp.v[0].x & 0xFFFF0000u, rq.v[0].x & 0xFFFF0000u, 1);
    f(rp.v[0].y << 16, rq.v[0].y << 16, 2); f(rp.v[0].y & 0xFFFF0000u, rq.v[0].y & 0xFFFF0000u, 3);
    f(rp.v[0].z << 16, rq.v[0].z << 16, 4); f(rp.v[0].z & 0xFFFF0000u, rq.v[0].z & 0xFFFF0000u, 5);
    f(rp.v[0].w << 16, rq.v[0].w << 16, 6); f(rp.v[0].w & 0xFFFF0000u, rq.v[0].w & 0xFFFF0000u, 7);
  } else {
    f(rp.v[0].x, rq.v[0].x, 0); f(rp.v[0].y, rq.v[0].y, 1); f(rp.v[0].z, rq.v[0].z, 2); f(rp.v[0].w, rq.v[0].w, 3);
    f(rp.v[Raw8<T>::W - 1].x, rq.v[Raw8<T>::W - 1].x, 4); f(rp.v[Raw8<T>::W - 1].y, rq.v[Raw8<T>::W - 1].y, 5);
    f(rp.v[Raw8<T>::W - 1].z, rq.v[Raw8<T>::W - 1].z, 6); f(rp.v[Raw8<T>::W - 1].w, rq.v[Raw8<T>::W - 1].w, 7);
  }
}

// The segments of one CTA's slice of a row (ids are int: V <= SDCP_MAX_VOCAB): segments
// [s0, s1) of 256 ids, grouped G at a time into ngrp <= kSegCap groups; warp w owns groups
// [ngrp w / 8, ngrp (w + 1) / 8).
struct SegSlice {
  int nseg, s0, s1, G, ngrp;
  __device__ __forceinline__ SegSlice(int V, unsigned C, unsigned rank) {
    nseg = (V + kSegIds - 1) / kSegIds;
    // nseg <= 2^16 (V <= SDCP_MAX_VOCAB) and rank < C <= 8, so the products fit 32 bits (a
    // 64-bit division is a long emulated sequence on the GPU)
    s0 = (int)(((unsigned)nseg * rank) / C);
    s1 = (int)(((unsigned)nseg * (rank + 1u)) / C);
    const int n = s1 - s0;
    G = max(1, (n + kSegCap - 1) / kSegCap);
    ngrp = (n + G - 1) / G;
  }
  __device__ __forceinline__ void warp_range(int w, int nw, int& a, int& b) const {
    a = s0 + (ngrp * w / nw) * G;
    b = min(s0 + (ngrp * (w + 1) / nw) * G, s1);
  }
  __device__ __forceinline__ int grp_lo(int k) const { return s0 + k * G; }
  __device__ __forceinline__ int grp_hi(int k) const { return min(s0 + (k + 1) * G, s1); }
};

// Sum of the 8 weights of one lane piece, and the weights themselves.
template <typename T, bool FILT, bool QR = false>
__device__ __forceinline__ float piece_weights(const Raw8<T>& rp, const Raw8<QElem<T, QR>>& rq, bool residual,
                                               const DrawRow& pr, const DrawRow& qr, int j0,
                                               float (&w)[kEpt]) {
  uint32_t bp[kEpt], bq[kEpt];
  unpack_raw8<T>(rp, bp);
  if (residual) unpack_raw8<QElem<T, QR>>(rq, bq);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kEpt; ++e) {
    float x = draw_weight<FILT>(pr, bp[e], j0 + e);
    if (residual) x = fmaxf(x - (QR ? __uint_as_float(bq[e]) : draw_weight<FILT>(qr, bq[e], j0 + e)), 0.f);
    w[e] = x;
    s += x;
  }
  return s;
}

// This CTA's slice: sm.seg[k] = weight of segment group k (ids in order within a group).
template <typename T, bool FILT, bool QR = false>
__device__ void draw_pass(const SegSlice& sl, SessSmem& sm, const T* prow, const T* qrow, bool residual,
                          bool al_p, bool al_q, int V, const DrawRow& pr, const DrawRow& qr) {
  using QT = QElem<T, QR>;
  const QT* qsrc = reinterpret_cast<const QT*>(qrow);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int a, b;
  sl.warp_range(w, kWarps, a, b);
  constexpr int U = (sizeof(T) == 2) ? 4 : 2;  // segments whose loads are in flight together
  float gacc = 0.f;
  for (int k = a; k < b; k += U) {
    Raw8<T> rp[U];
    Raw8<QT> rq[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j0 = (k + u) * kSegIds + lane * kEpt;
      if (k + u < b) {
        load_raw8<T>(prow, al_p, V, j0, rp[u]);
        if (residual) load_raw8<QT>(qsrc, al_q, V, j0, rq[u], QR ? 0u : 0xFF800000u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = k + u;
      if (kk < b) {
        const int j0 = kk * kSegIds + lane * kEpt;
        float ls = 0.f;
        if constexpr (QR) {
          float wv[kEpt];
          ls = piece_weights<T, FILT, true>(rp[u], rq[u], residual, pr, qr, j0, wv);
        } else {
          for_each8<T>(rp[u], rq[u], [&](uint32_t bp, uint32_t bq, int e) {
            float x = draw_weight<FILT>(pr, bp, j0 + e);
            if (residual) x = fmaxf(x - draw_weight<FILT>(qr, bq, j0 + e), 0.f);
            ls += x;
          });
        }
        gacc += warp_reduce(ls, [](float x, float y) { return x + y; });
        if ((kk - sl.s0 + 1) % sl.G == 0 || kk + 1 == sl.s1) {
          if (lane == 0) sm.seg[(kk - sl.s0) / sl.G] = gacc;
          gacc = 0.f;
        }
      }
    }
  }
}

// One warp walks segments [k0, k1) from cumulative weight `carry`: the smallest id whose
// cumulative weight exceeds target, else (rounding) the largest id with positive weight seen.
// Weights and their sums within a segment are fp32; the running total across segments and
// the comparison with the target are fp64, so long rows keep the position of u * W.
template <typename T, bool FILT, bool QR = false>
__device__ int draw_walk(const T* prow, const T* qrow, bool residual, bool al_p, bool al_q, int V,
                         const DrawRow& pr, const DrawRow& qr, int k0, int k1, double carry,
                         double target) {
  const int lane = threadIdx.x & 31;
  int lastpos = -1;
  for (int k = k0; k < k1; ++k) {
    const int j0 = k * kSegIds + lane * kEpt;
    Raw8<T> rp;
    Raw8<QElem<T, QR>> rq;
    load_raw8<T>(prow, al_p, V, j0, rp);
    if (residual)
      load_raw8<QElem<T, QR>>(reinterpret_cast<const QElem<T, QR>*>(qrow), al_q, V, j0, rq, QR ? 0u : 0xFF800000u);
    float wv[kEpt];
    const float ls = piece_weights<T, FILT, QR>(rp, rq, residual, pr, qr, j0, wv);
    int lp = -1;
#pragma unroll
    for (int e = 0; e < kEpt; ++e) if (wv[e] > 0.f) lp = j0 + e;
    lastpos = max(lastpos, __reduce_max_sync(0xFFFFFFFFu, lp));
    float incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float tv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += tv;
    }
    // the lanes' intervals tile the segment: lane l covers [incl(l-1), incl(l)) past carry,
    // so a target never falls between two lanes, whatever the rounding of incl.  The target's
    // offset past carry is taken once in fp64 and rounded down to a float, dt: for a float x,
    // x <= dt exactly when x <= target - carry, and dt < x exactly when target - carry < x.
    float ex = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    if (lane == 0) ex = 0.f;
    const float dt = __double2float_rd(target - carry);
    int hit = INT_MAX;
    if (ls > 0.f && ex <= dt && dt < incl) {
      float cc = ex;
#pragma unroll
      for (int e = 0; e < kEpt; ++e) {
        cc += wv[e];
        if (hit == INT_MAX && wv[e] > 0.f && cc > dt) hit = j0 + e;
      }
      if (hit == INT_MAX) hit = lp;  // the lane's sum reached the target, its steps fell short
    }
    const int found = __reduce_min_sync(0xFFFFFFFFu, hit);
    if (found != INT_MAX && found >= 0) return found;
    carry += (double)__shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  return lastpos;
}


// ---------------------------------------------------------------------------------
// Locating the token: the slices' totals through distributed shared memory, the CTA
// whose slice holds u * W scans its segment sums, one warp walks the segment.
// ---------------------------------------------------------------------------------

// Returns W (the same in every CTA), or NaN when some CTA of the cluster flagged its pass
// as unusable (sm.overflow).  Tie ids come from the CTAs' candidates when `ties`.  Sums
// within a CTA's slice are fp32 (a scan of at most 2048 segment sums: about 20 roundings);
// the slices' totals, the target u * W and the owner's base are fp64.
template <typename T, bool FILT, bool QR = false>
__device__ double locate_and_walk(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                              const SegSlice& sl, const T* prow, const T* qrow, bool residual,
                                              bool al_p, bool al_q, int V, DrawRow pr, DrawRow qr,
                                              bool pp, bool qp, double u1, int32_t* out) {
  const int t = threadIdx.x, w = t >> 5, lane = t & 31;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const int gpt = (sl.ngrp + g.nthreads - 1) / g.nthreads;
  float loc = 0.f;
  for (int i = 0; i < gpt; ++i) {
    const int k = t * gpt + i;
    if (k < sl.ngrp) loc += sm.seg[k];
  }
  float Wc;
  const float pre = group_excl_scan(g, loc, sm.fscr, &Wc);
  if (t == 0) { sm.cta_sum = (double)Wc; sm.cta_ovf = sm.overflow; }
  cluster.sync();
  cluster_copy(cluster, &sm.cta_sum, sm.cv_sum);
  cluster_copy(cluster, &sm.tie_p_cand, sm.cv_i0);
  cluster_copy(cluster, &sm.tie_q_cand, sm.cv_i1);
  cluster_copy(cluster, &sm.cta_ovf, sm.cv_ovf);
  cluster.sync();  // every CTA has read the slice totals
  if (t == 0) {
    // the owner is the last slice with weight whose start is at or below the target (the
    // slices tile [0, W) by construction, whatever the rounding of their sums)
    double W = 0.0, acc = 0.0, obase = 0.0;
    int owner = -1, bad = 0;
    for (unsigned r = 0; r < C; ++r) { W += sm.cv_sum[r]; bad |= sm.cv_ovf[r]; }
    const double target = u1 * W;
    for (unsigned r = 0; r < C; ++r) {
      const double sr = sm.cv_sum[r];
      if (sr > 0.0 && acc <= target) { owner = (int)r; obase = acc; }
      acc += sr;
    }
    sm.d_W = W; sm.d_target = target; sm.d_base = obase; sm.d_owner = owner; sm.d_bad = bad;
    sm.d_tloc = (float)(target - obase);  // the target within the owner's slice
  }
  g.sync();
  int tp_id = INT_MAX, tq_id = INT_MAX;
  for (unsigned r = 0; r < C; ++r) {
    tp_id = min(tp_id, sm.cv_i0[r]);
    tq_id = min(tq_id, sm.cv_i1[r]);
  }
  const double W = sm.d_W;
  const int owner = sm.d_owner;
  if (sm.d_bad) return kNaN64;
  if (!(W > 0.0)) return W;
  if (owner != (int)rank) return W;
  // tie ids found by this pass (the lists); otherwise the caller's stand (found beforehand
  // by cut_tie_id, or INT_MAX: every token of the cut value kept)
  if (pp) pr.tie = tp_id;
  if (qp) qr.tie = tq_id;
  // the group: the last one with weight whose start is at or below the target (groups tile
  // the slice by construction; a target past the slice's rounded end takes its last group,
  // whose walk then ends on its last token with weight)
  long long cand = -1;
  float cbase = 0.f;
  {
    const float tloc = sm.d_tloc;  // the target within this slice
    float bsum = pre;
    for (int i = 0; i < gpt; ++i) {
      const int k = t * gpt + i;
      if (k >= sl.ngrp) break;
      const float sk = sm.seg[k];
      if (sk > 0.f && bsum <= tloc) { cand = k; cbase = bsum; }
      bsum += sk;
    }
  }
  const long long og = group_max_i64(g, cand, sm.lscr);
  if (og >= 0 && cand == og) sm.owner_base = sm.d_base + (double)cbase;
  g.sync();
  if (w == 0 && og >= 0) {
    const int tok = draw_walk<T, FILT, QR>(prow, qrow, residual, al_p, al_q, V, pr, qr, sl.grp_lo((int)og),
                                       sl.grp_hi((int)og), sm.owner_base, sm.d_target);
    if (lane == 0) *out = tok;
  }
  return W;
}

// ---------------------------------------------------------------------------------
// Tokens on a cut value (the single-pass draws): left out of the segment sums during the
// pass and held, with both weights, in a per-warp list in id order within each stage.
// ---------------------------------------------------------------------------------

// Clears the per-call state of the cut-value tokens (group).
__device__ __forceinline__ void ties_reset(const Group& g, SessSmem& sm) {
  for (int i = threadIdx.x; i < kTieStages * kWarps; i += g.nthreads) {
    (&sm.tsc_p[0][0])[i] = 0;
    (&sm.tsc_q[0][0])[i] = 0;
  }
  if (threadIdx.x == 0) { sm.overflow = 0; sm.tie_p_cand = INT_MAX; sm.tie_q_cand = INT_MAX; }
  if (threadIdx.x < kWarps) sm.tie_n[threadIdx.x] = 0;
}

// Appends the lane's cut-value tokens of one piece (amb; cp / cq: on p's / q's cut value),
// lanes in order, to the warp's list, and counts them for stage st.  Whole warp, only when
// some lane has such a token.
template <typename T>
__device__ void tie_append(SessSmem& sm, const Raw8<T>& rp, const Raw8<T>& rq, bool residual,
                                        const DrawRow& pr, const DrawRow& qr, int j0, uint32_t amb,
                                        uint32_t cp, uint32_t cq, int st, int& nt, bool& ovf) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = __popc(amb), cnp = __popc(cp), cnq = __popc(cq);
  int incl = c, ip = cnp, iq = cnq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a1 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    const int a2 = __shfl_up_sync(0xFFFFFFFFu, ip, o);
    const int a3 = __shfl_up_sync(0xFFFFFFFFu, iq, o);
    if (lane >= o) { incl += a1; ip += a2; iq += a3; }
  }
  const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  const int tp = __shfl_sync(0xFFFFFFFFu, ip, 31), tq = __shfl_sync(0xFFFFFFFFu, iq, 31);
  if (ovf || st >= kTieStages || nt + total > kTieCap) { ovf = true; return; }
  const int bp = sm.tsc_p[st][w], bq = sm.tsc_q[st][w];
  __syncwarp();
  int pos = nt + incl - c, lp = bp + ip - cnp, lq = bq + iq - cnq;
  for_each8<T>(rp, rq, [&](uint32_t xp, uint32_t xq, int e) {
    if ((amb >> e) & 1u) {
      const float vp = __uint_as_float(xp), vq = __uint_as_float(xq);
      const float P = (vp >= pr.thr) ? row_weight(pr, vp) : 0.f;
      const float Q = (residual && vq >= qr.thr) ? row_weight(qr, vq) : 0.f;
      const int ep = (cp >> e) & 1u, eq = (cq >> e) & 1u;
      sm.ties[w][pos] = TieEntry{j0 + e, P, Q, ep | (eq << 1) | (st << 8), lp, lq};
      ++pos;
      lp += ep;
      lq += eq;
    }
  });
  if (lane == 0) { sm.tsc_p[st][w] = bp + tp; sm.tsc_q[st][w] = bq + tq; }
  nt += total;
  __syncwarp();
}

// After the pass (group, every CTA of the cluster): the rank of a cut-value token is its
// index among the cluster's tokens of that cut value in id order (slices in rank order,
// then stages, then warps, then list order); the first thr_n are kept.  Their weights
// join the segment sums (each warp adds its own, in id order) and the id bound of the kept
// ones goes to sm.tie_*_cand.  Returns false when a list overflowed anywhere (uniform).
static __device__ bool resolve_ties(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                          const SegSlice& sl, int nstages, bool residual, int np_cut,
                                          int nq_cut) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  if (t == 0) {  // exclusive prefix per (stage, warp) within the slice
    int ap = 0, aq = 0;
    for (int s = 0; s < nstages && s < kTieStages; ++s)
      for (int i = 0; i < kWarps; ++i) {
        const int cp = sm.tsc_p[s][i], cq = sm.tsc_q[s][i];
        sm.tsc_p[s][i] = ap; sm.tsc_q[s][i] = aq;
        ap += cp; aq += cq;
      }
    sm.cta_np = ap; sm.cta_nq = aq; sm.cta_ovf = sm.overflow;
  }
  cluster.sync();
  cluster_copy(cluster, &sm.cta_np, sm.cv_n0);
  cluster_copy(cluster, &sm.cta_nq, sm.cv_n1);
  cluster_copy(cluster, &sm.cta_ovf, sm.cv_ovf);
  cluster.sync();  // every CTA has read the counts
  long long P0 = 0, Q0 = 0;
  int ovf_any = 0;
  for (unsigned r = 0; r < C; ++r) {
    if (r < rank) { P0 += sm.cv_n0[r]; Q0 += sm.cv_n1[r]; }
    ovf_any |= sm.cv_ovf[r];
  }
  if (ovf_any) return false;
  TieEntry* L = sm.ties[w];
  const int nt = sm.tie_n[w];
  for (int i = lane; i < nt; i += 32) {
    const TieEntry en = L[i];
    const int st = en.code >> 8, isp = en.code & 1, isq = (en.code >> 1) & 1;
    const long long rp = P0 + sm.tsc_p[st][w] + en.lp, rq = Q0 + sm.tsc_q[st][w] + en.lq;
    const bool kp = !isp || rp < np_cut, kq = !isq || rq < nq_cut;
    if (isp && rp == (long long)np_cut - 1) sm.tie_p_cand = en.id;
    if (isq && rq == (long long)nq_cut - 1) sm.tie_q_cand = en.id;
    const float P = kp ? en.P : 0.f, Q = kq ? en.Q : 0.f;
    L[i].P = residual ? fmaxf(P - Q, 0.f) : P;  // the token's weight
  }
  __syncwarp();
  if (lane == 0)  // into the segment sums, in id order
    for (int i = 0; i < nt; ++i) sm.seg[(L[i].id / kSegIds - sl.s0) / sl.G] += L[i].P;
  g.sync();
  return true;
}

// ---------------------------------------------------------------------------------
// The draw from global memory (any row alignment, any slice length).
// ---------------------------------------------------------------------------------

// Without cut-value tokens to rank: every token's weight is known during the pass.
template <typename T, bool FILT, bool QR = false>
__device__ double draw_token(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                         const T* prow, const T* qrow, bool residual, bool al_p,
                                         bool al_q, int V, const DrawRow& pr, const DrawRow& qr,
                                         double u1, int32_t* out) {
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  if (threadIdx.x == 0) { sm.overflow = 0; sm.tie_p_cand = INT_MAX; sm.tie_q_cand = INT_MAX; }
  draw_pass<T, FILT, QR>(sl, sm, prow, qrow, residual, al_p, al_q, V, pr, qr);
  g.sync();
  return locate_and_walk<T, FILT, QR>(cluster, g, sm, sl, prow, qrow, residual, al_p, al_q, V, pr, qr,
                                      false, false, u1, out);
}

// A cut inside a value (p's, q's or both), in one pass; NaN when a list overflowed.
template <typename T>
__device__ double draw_token_ties(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                              const T* prow, const T* qrow, bool residual, bool al_p,
                                              bool al_q, int V, const DrawRow& pr, const DrawRow& qr,
                                              int np_cut, int nq_cut, double u1, int32_t* out) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  const bool pp = np_cut != INT_MAX, qp = residual && nq_cut != INT_MAX;
  ties_reset(g, sm);
  g.sync();
  {
    int a, b;
    sl.warp_range(w, kWarps, a, b);
    constexpr int U = 2;
    float gacc = 0.f;
    int nt = 0;
    bool ovf = false;
    for (int k = a; k < b; k += U) {
      Raw8<T> rp[U], rq[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j0 = (k + u) * kSegIds + lane * kEpt;
        if (k + u < b) {
          load_raw8<T>(prow, al_p, V, j0, rp[u]);
          if (residual) load_raw8<T>(qrow, al_q, V, j0, rq[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int kk = k + u;
        if (kk >= b) continue;
        const int j0 = kk * kSegIds + lane * kEpt;
        uint32_t amb = 0u, cp = 0u, cq = 0u;
        float ls = 0.f;
        for_each8<T>(rp[u], rq[u], [&](uint32_t bp, uint32_t bq, int e) {
          const float vp = __uint_as_float(bp), vq = __uint_as_float(bq);
          const bool tp = pp && vp == pr.thr, tq = qp && vq == qr.thr;
          float x = (vp >= pr.thr) ? row_weight(pr, vp) : 0.f;
          if (residual) x = fmaxf(x - ((vq >= qr.thr) ? row_weight(qr, vq) : 0.f), 0.f);
          const bool am = tp || tq;  // on a cut value: weighed after the pass
          amb |= (am ? 1u : 0u) << e;
          cp |= (tp ? 1u : 0u) << e;
          cq |= (tq ? 1u : 0u) << e;
          ls += am ? 0.f : x;
        });
        gacc += warp_reduce(ls, [](float x, float y) { return x + y; });
        if ((kk - sl.s0 + 1) % sl.G == 0 || kk + 1 == sl.s1) {
          if (lane == 0) sm.seg[(kk - sl.s0) / sl.G] = gacc;
          gacc = 0.f;
        }
        if (__any_sync(0xFFFFFFFFu, amb != 0u))
          tie_append<T>(sm, rp[u], rq[u], residual, pr, qr, j0, amb, cp, cq, 0, nt, ovf);
      }
    }
    if (lane == 0) {
      sm.tie_n[w] = nt;
      if (ovf) sm.overflow = 1;
    }
  }
  g.sync();
  if (!resolve_ties(cluster, g, sm, sl, 1, residual, np_cut, nq_cut)) return kNaN64;
  return locate_and_walk<T, true>(cluster, g, sm, sl, prow, qrow, residual, al_p, al_q, V, pr, qr, pp, qp,
                                  u1, out);
}

// ---------------------------------------------------------------------------------
// The streamed draw: thread 0 copies the CTA's slice of p (and q) into a two-stage ring
// of shared memory with bulk copies (TMA) that complete on mbarriers, 16 KB of each row
// per stage; each warp reduces its segments of a stage from shared memory and hands the
// stage back.  Needs 16-byte aligned rows, V a multiple of 8, one segment per group (a
// slice of at most 2048 segments) and, with cut-value tokens, at most kTieStages stages.
// Returns W, or NaN when it could not decide (a list overflowed, a wait gave up): the
// caller then draws from global memory.
// ---------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ bool stream_ok(int V, unsigned C, unsigned rank, bool al, bool ties) {
  const SegSlice sl(V, C, rank);
  constexpr int S = kDrawHalf / (int)sizeof(T);
  const int n = min(sl.s1 * kSegIds, V) - sl.s0 * kSegIds;
  return al && (V % 8) == 0 && sl.G == 1 && (!ties || (n + S - 1) / S <= kTieStages);
}

template <typename T, bool FILT, bool TIES>
__device__ double draw_stream(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                          unsigned char* ring, const T* prow, const T* qrow, bool residual,
                                          int V, const DrawRow& pr, const DrawRow& qr, int np_cut,
                                          int nq_cut, double u1, int32_t* out) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  constexpr int S = kDrawHalf / (int)sizeof(T);  // ids per stage
  constexpr int SPW = S / kSegIds / kWarps;       // segments of a warp per stage
  static_assert(SPW >= 1 && SPW * kWarps * kSegIds == S, "stage layout");
  static_assert(SPW * 32 <= (int)sizeof(sm.plist[0]), "piece list");
  const int lo = sl.s0 * kSegIds, hi = min(sl.s1 * kSegIds, V);
  const int nst = (hi > lo) ? (hi - lo + S - 1) / S : 0;
  const bool pp = TIES && np_cut != INT_MAX, qp = TIES && residual && nq_cut != INT_MAX;
  const uint32_t use0 = sm.ring_uses;
  (void)pp; (void)qp;
  if (TIES) ties_reset(g, sm);
  else if (t == 0) { sm.overflow = 0; sm.tie_p_cand = INT_MAX; sm.tie_q_cand = INT_MAX; }
  g.sync();  // every thread has read ring_uses
  bool fail = false;
  int issued = 0;  // thread 0: stages whose copies were issued (always a prefix 0 .. issued-1)
  auto issue = [&](int s) {  // thread 0: stage s of the slice into its slot
    const uint32_t u = use0 + (uint32_t)s;
    const int slot = (int)(u % kDrawStages);
    if (fail) return;
    if (u >= kDrawStages && !mbar_wait_for(&sm.empty[slot], ((u / kDrawStages) - 1) & 1u, nullptr)) {
      fail = true;
      return;
    }
    issued = s + 1;
    const int n = min(S, hi - (lo + s * S));
    const uint32_t bytes = (uint32_t)n * sizeof(T);
    unsigned char* dst = ring + (size_t)slot * 2 * kDrawHalf;
    mbar_arrive_expect_tx(&sm.full[slot], residual ? 2 * bytes : bytes);
    bulk_copy_g2s(dst, prow + lo + s * S, bytes, &sm.full[slot]);
    if (residual) bulk_copy_g2s(dst + kDrawHalf, qrow + lo + s * S, bytes, &sm.full[slot]);
  };
  if (t == 0)
    for (int s = 0; s < nst && s < kDrawStages; ++s) issue(s);
  int nt = 0;
  bool ovf = false;
  for (int s = 0; s < nst; ++s) {
    const uint32_t u = use0 + (uint32_t)s;
    const int slot = (int)(u % kDrawStages);
    if (!mbar_wait_for(&sm.full[slot], (u / kDrawStages) & 1u, nullptr)) fail = true;
    const unsigned char* src = ring + (size_t)slot * 2 * kDrawHalf;
    const int stage_lo = lo + s * S;
    // the lane's piece (8 ids) of segment sis of the stage; ids past the slice read as -inf
    auto load_piece = [&](int sis, int pl, Raw8<T>& rp, Raw8<T>& rq) {
      const int j0 = stage_lo + sis * kSegIds + pl * kEpt;
      const uint4* pv = reinterpret_cast<const uint4*>(src + (size_t)(sis * kSegIds + pl * kEpt) * sizeof(T));
#pragma unroll
      for (int q = 0; q < Raw8<T>::W; ++q) rp.v[q] = pv[q];
      if (residual) {
        const uint4* qv = reinterpret_cast<const uint4*>(src + kDrawHalf + (size_t)(sis * kSegIds + pl * kEpt) * sizeof(T));
#pragma unroll
        for (int q = 0; q < Raw8<T>::W; ++q) rq.v[q] = qv[q];
      }
      if (j0 + kEpt > hi) {  // the row's last segment
        uint32_t* a = reinterpret_cast<uint32_t*>(rp.v);
        uint32_t* bq = reinterpret_cast<uint32_t*>(rq.v);
#pragma unroll
        for (int e = 0; e < kEpt; ++e) {
          if (j0 + e >= hi) {
            if (sizeof(T) == 2) {
              a[e >> 1] = (e & 1) ? ((a[e >> 1] & 0x0000FFFFu) | 0xFF800000u) : ((a[e >> 1] & 0xFFFF0000u) | 0xFF80u);
              bq[e >> 1] = (e & 1) ? ((bq[e >> 1] & 0x0000FFFFu) | 0xFF800000u) : ((bq[e >> 1] & 0xFFFF0000u) | 0xFF80u);
            } else {
              a[e] = 0xFF800000u;
              bq[e] = 0xFF800000u;
            }
          }
        }
      }
      return j0;
    };
    // the weights of one piece: ls (tokens off the cut values), amb / cp / cq (on them)
    auto weigh = [&](const Raw8<T>& rp, const Raw8<T>& rq, int j0, float& ls, uint32_t& amb, uint32_t& cp,
                     uint32_t& cq) {
      for_each8<T>(rp, rq, [&](uint32_t bp, uint32_t bqq, int e) {
        if (!TIES) {
          float x = draw_weight<FILT>(pr, bp, j0 + e);
          if (residual) x = fmaxf(x - draw_weight<FILT>(qr, bqq, j0 + e), 0.f);
          ls += x;
        } else {
          const float vp = __uint_as_float(bp), vq = __uint_as_float(bqq);
          const bool tp = pp && vp == pr.thr, tq = qp && vq == qr.thr;
          float x = (vp >= pr.thr) ? row_weight(pr, vp) : 0.f;
          if (residual) x = fmaxf(x - ((vq >= qr.thr) ? row_weight(qr, vq) : 0.f), 0.f);
          const bool am = tp || tq;
          amb |= (am ? 1u : 0u) << e;
          cp |= (tp ? 1u : 0u) << e;
          cq |= (tq ? 1u : 0u) << e;
          ls += am ? 0.f : x;
        }
      });
    };
    if constexpr (!FILT) {
#pragma unroll 1
      for (int i = 0; i < SPW; ++i) {
        const int sis = w * SPW + i;  // segment in the stage
        const int seg_lo = stage_lo + sis * kSegIds;
        if (seg_lo >= hi) continue;  // past the slice (warp-uniform)
        Raw8<T> rp, rq;
        const int j0 = load_piece(sis, lane, rp, rq);
        uint32_t amb = 0u, cp = 0u, cq = 0u;
        float ls = 0.f;
        weigh(rp, rq, j0, ls, amb, cp, cq);
        const float ssum = warp_reduce(ls, [](float x, float y) { return x + y; });
        if (lane == 0) sm.seg[(seg_lo - lo) / kSegIds] = ssum;
      }
    } else {
      // p has a cut: a piece whose p values all lie below p's cut value weighs nothing (p is
      // 0 there, so is the residual), and holds no cut-value token of p.  Only the pieces
      // that reach p's cut value, or hold a token on q's cut value (whose ranks the ties
      // need), are weighed: listed per warp in id order, then taken one per lane.
      uint32_t mk = 0u;
#pragma unroll
      for (int i = 0; i < SPW; ++i) {
        const int sis = w * SPW + i;
        if (stage_lo + sis * kSegIds >= hi) continue;  // warp-uniform
        Raw8<T> rp, rq;
        (void)load_piece(sis, lane, rp, rq);
        bool m = piece_reaches<T>(rp, pr.thr);
        if (TIES && qp) m = m || piece_holds<T>(rq, qr.thr);
        mk |= (m ? 1u : 0u) << i;
      }
      uint8_t* list = sm.plist[w];
      int H = 0;
#pragma unroll
      for (int i = 0; i < SPW; ++i) {
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, (mk >> i) & 1u);
        if ((mk >> i) & 1u) list[H + __popc(bal & ((1u << lane) - 1u))] = (uint8_t)(i * 32 + lane);
        H += __popc(bal);
      }
      __syncwarp();
      float segsum[SPW];
#pragma unroll
      for (int i = 0; i < SPW; ++i) segsum[i] = 0.f;
      for (int e0 = 0; e0 < H; e0 += 32) {
        const int e = e0 + lane;
        Raw8<T> rp, rq;
        uint32_t amb = 0u, cp = 0u, cq = 0u;
        float ls = 0.f;
        int pi = -1, j0 = 0;
        if (e < H) {
          pi = list[e];
          j0 = load_piece(w * SPW + (pi >> 5), pi & 31, rp, rq);
          weigh(rp, rq, j0, ls, amb, cp, cq);
        }
#pragma unroll
        for (int i = 0; i < SPW; ++i) segsum[i] += (pi >= 0 && (pi >> 5) == i) ? ls : 0.f;
        if (TIES && __any_sync(0xFFFFFFFFu, amb != 0u))
          tie_append<T>(sm, rp, rq, residual, pr, qr, j0, amb, cp, cq, s, nt, ovf);
      }
      __syncwarp();  // the list is free for the next stage
#pragma unroll
      for (int i = 0; i < SPW; ++i) {
        const int seg_lo = stage_lo + (w * SPW + i) * kSegIds;
        const float ssum = warp_reduce(segsum[i], [](float x, float y) { return x + y; });
        if (lane == 0 && seg_lo < hi) sm.seg[(seg_lo - lo) / kSegIds] = ssum;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
    if (t == 0 && s + kDrawStages < nst) issue(s + kDrawStages);
  }
  if (TIES && lane == 0) sm.tie_n[w] = nt;
  if (lane == 0 && (ovf || fail)) sm.overflow = 1;
  if (t == 0 && fail) {  // a wait gave up: the copies already issued land first (bounded)
    for (int s = max(0, issued - kDrawStages); s < issued; ++s) {
      const uint32_t u = use0 + (uint32_t)s;
      (void)mbar_wait_for(&sm.full[u % kDrawStages], (u / kDrawStages) & 1u, nullptr);
    }
  }
  if (t == 0) sm.ring_uses = use0 + (uint32_t)nst;
  g.sync();
  if (TIES && !resolve_ties(cluster, g, sm, sl, nst, residual, np_cut, nq_cut)) return kNaN64;
  const bool al_p = ((uintptr_t)prow & 15u) == 0, al_q = ((uintptr_t)qrow & 15u) == 0;
  return locate_and_walk<T, FILT || TIES>(cluster, g, sm, sl, prow, qrow, residual, al_p, al_q, V, pr, qr,
                                          pp, qp, u1, out);
}

// Id of the n-th token (1-based, id order) with value `val` over the cluster (every CTA
// gets it); INT_MAX if none.
template <typename T>
__device__ int cut_tie_id(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                       const T* row, bool al, int V, float val, int n) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  int a, b;
  sl.warp_range(w, kWarps, a, b);
  constexpr int U = (sizeof(T) == 2) ? 4 : 2;
  int gacc = 0;
  for (int k = a; k < b; k += U) {
    Raw8<T> r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (k + u < b) load_raw8<T>(row, al, V, (k + u) * kSegIds + lane * kEpt, r[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = k + u;
      if (kk < b) {
        uint32_t bb[kEpt];
        unpack_raw8<T>(r[u], bb);
        int c = 0;
#pragma unroll
        for (int e = 0; e < kEpt; ++e) c += (__uint_as_float(bb[e]) == val) ? 1 : 0;
        gacc += __reduce_add_sync(0xFFFFFFFFu, (unsigned)c);
        if ((kk - sl.s0 + 1) % sl.G == 0 || kk + 1 == sl.s1) {
          if (lane == 0) sm.seg[(kk - sl.s0) / sl.G] = (float)gacc;  // counts <= 2^24: exact
          gacc = 0;
        }
      }
    }
  }
  g.sync();
  const int gpt = (sl.ngrp + g.nthreads - 1) / g.nthreads;
  long long loc = 0;
  for (int i = 0; i < gpt; ++i) {
    const int k = t * gpt + i;
    if (k < sl.ngrp) loc += (long long)sm.seg[k];
  }
  if (t == 0) sm.result = LLONG_MAX;  // ordered before the owner's write by the scan's barriers
  long long tot;
  const long long pre = group_excl_scan_ll(g, loc, sm.lscr, &tot);
  if (t == 0) sm.cta_cnt = tot;
  cluster.sync();
  cluster_copy(cluster, &sm.cta_cnt, sm.cv_n0);
  g.sync();  // the copies, before their readers (sm.cta_cnt is not written again in this call)
  long long base = 0, acc = 0;
  int owner = -1;
  for (unsigned r = 0; r < C; ++r) {
    const long long cr = sm.cv_n0[r];
    if (r == rank) base = acc;
    if (owner < 0 && acc < n && n <= acc + cr) owner = (int)r;
    acc += cr;
  }
  if (owner == (int)rank) {
    if (base + pre < n && n <= base + pre + loc) {  // this thread's groups hold it
      long long bb = base + pre;
      for (int i = 0; i < gpt; ++i) {
        const int k = t * gpt + i;
        const long long c = (long long)sm.seg[k];
        if (bb < n && n <= bb + c) { sm.owner_pre = k; sm.owner_carry = bb; break; }
        bb += c;
      }
    }
    g.sync();
    if (w == 0) {
      const int og = (int)sm.owner_pre;
      long long carry = sm.owner_carry;
      int found = INT_MAX;
      for (int k = sl.grp_lo(og); k < sl.grp_hi(og) && found == INT_MAX; ++k) {
        const int j0 = k * kSegIds + lane * kEpt;
        Raw8<T> r;
        load_raw8<T>(row, al, V, j0, r);
        uint32_t bb[kEpt];
        unpack_raw8<T>(r, bb);
        int c = 0;
#pragma unroll
        for (int e = 0; e < kEpt; ++e) c += (__uint_as_float(bb[e]) == val) ? 1 : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int tv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += tv;
        }
        const long long lp = carry + (incl - c);
        int hit = INT_MAX;
        if (c > 0 && lp < n && n <= lp + c) {
          long long kk = lp;
#pragma unroll
          for (int e = 0; e < kEpt; ++e)
            if (hit == INT_MAX && __uint_as_float(bb[e]) == val && ++kk == n) hit = j0 + e;
        }
        found = __reduce_min_sync(0xFFFFFFFFu, hit);
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) sm.result = found;
    }
  }
  cluster.sync();
  if (t == 0) sm.cv_res = (owner >= 0) ? *cluster.map_shared_rank(&sm.result, (unsigned)owner) : LLONG_MAX;
  cluster.sync();  // the owner's shared memory is read before anyone moves on
  const long long id = sm.cv_res;
  return (id == LLONG_MAX || id == INT_MAX) ? INT_MAX : (int)id;
}

// ---------------------------------------------------------------------------------
// The kept-set draw.  When p has a cut (top-k / top-p), every token outside p's kept set
// has p = 0 and so neither a residual nor a bonus weight: the CTAs scan their slices of p's
// row for the tokens at or above p's cut value (a compare per token), hold them in per-warp
// lists in id order, and weigh only those (q is read at their ids alone).  Cut-value ties
// are ranked from the lists: p's from its own candidates, q's from the ids of q's cut-value
// tokens collected in the same pass.  Returns W (the same in every CTA), or NaN when some
// list of the cluster overflowed (the streamed draw takes over).
// ---------------------------------------------------------------------------------

// Appends the lanes' marked ids (bit e of m: id j0 + e) to a warp list in id order; vals
// (optional) are the matching logits.  n: the list length (lane-uniform); false on overflow.
template <int CAP>
__device__ __forceinline__ bool warp_list_append(int* ids, float* vals, int& n, unsigned m, int j0,
                                                 const uint32_t (&bits)[kEpt]) {
  const int lane = threadIdx.x & 31;
  if (__ballot_sync(0xFFFFFFFFu, m != 0u) == 0u) return true;
  const int c = __popc(m);
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  const int tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (n + tot > CAP) { n = CAP + 1; return false; }
  int pos = n + incl - c;
#pragma unroll
  for (int e = 0; e < kEpt; ++e)
    if ((m >> e) & 1u) {
      ids[pos] = j0 + e;
      if (vals) vals[pos] = __uint_as_float(bits[e]);
      ++pos;
    }
  n += tot;
  return true;
}

// Id of the k-th (1-based, id order) candidate of this CTA with value val: INT_MAX if the
// CTA holds fewer (one full warp; every lane returns it).
__device__ __forceinline__ int kth_candidate(const KeptSmem& K, float val, long long k) {
  const int lane = threadIdx.x & 31;
  int w = 0;
  for (; w < kWarps && k > K.pc[w]; ++w) k -= K.pc[w];
  if (w == kWarps || k < 1) return INT_MAX;
  for (int i0 = 0; i0 < K.n[w]; i0 += 32) {
    const int i = i0 + lane;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, i < K.n[w] && K.v[w][i] == val);
    const int c = __popc(m);
    if (k <= c) return K.id[w][i0 + (int)__fns(m, 0, (int)k)];
    k -= c;
  }
  return INT_MAX;
}
// Id of the k-th (1-based, id order) listed q cut-value token of this CTA (any thread).
__device__ __forceinline__ int kth_qcut(const KeptSmem& K, long long k) {
  for (int w = 0; w < kWarps; ++w) {
    if (k >= 1 && k <= K.qn[w]) return K.qid[w][k - 1];
    k -= K.qn[w];
  }
  return INT_MAX;
}

template <typename T, bool QR = false>
__device__ double draw_kept(cg::cluster_group& cluster, const Group& g, SessSmem& sm, const T* prow,
                           const T* qrow, bool residual, bool al_p, bool al_q, int V, DrawRow pr, DrawRow qr,
                           int np_cut, int nq_cut, double u1, int32_t* out) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  int sa, sb;
  sl.warp_range(w, kWarps, sa, sb);
  const bool pp = np_cut != INT_MAX;              // p's cut value is kept in part
  const bool qp = residual && nq_cut != INT_MAX;  // q's cut value is kept in part
  KeptSmem& K = sm.kept;
  // pass: p's candidates and q's cut-value ids of the warp's segments, in id order
  int nc = 0, nq = 0;
  constexpr int U = (sizeof(T) == 2) ? 4 : 2;
  for (int k = sa; k < sb; k += U) {
    Raw8<T> rp[U], rq[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (k + u < sb) {
        load_raw8<T>(prow, al_p, V, (k + u) * kSegIds + lane * kEpt, rp[u]);
        if (qp) load_raw8<T>(qrow, al_q, V, (k + u) * kSegIds + lane * kEpt, rq[u]);
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (k + u >= sb) break;
      const int j0 = (k + u) * kSegIds + lane * kEpt;
      uint32_t bb[kEpt];
      unpack_raw8<T>(rp[u], bb);
      unsigned m = 0u;
#pragma unroll
      for (int e = 0; e < kEpt; ++e) m |= (j0 + e < V && __uint_as_float(bb[e]) >= pr.thr ? 1u : 0u) << e;
      (void)warp_list_append<kKeptW>(K.id[w], K.v[w], nc, nc > kKeptW ? 0u : m, j0, bb);
      if (qp) {
        unpack_raw8<T>(rq[u], bb);
        unsigned mq = 0u;
#pragma unroll
        for (int e = 0; e < kEpt; ++e) mq |= (j0 + e < V && __uint_as_float(bb[e]) == qr.thr ? 1u : 0u) << e;
        (void)warp_list_append<kQCutW>(K.qid[w], nullptr, nq, nq > kQCutW ? 0u : mq, j0, bb);
      }
    }
  }
  // p's cut-value candidates of the warp
  int pc = 0;
  if (pp && nc <= kKeptW) {
    for (int i = lane; i < nc; i += 32) pc += (K.v[w][i] == pr.thr) ? 1 : 0;
    pc = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)pc);
  }
  if (lane == 0) { K.n[w] = nc; K.qn[w] = nq; K.pc[w] = pc; }
  g.sync();
  if (t == 0) {
    int ovf = 0, tp = 0, tq = 0;
    for (int i = 0; i < kWarps; ++i) {
      ovf |= (K.n[i] > kKeptW || K.qn[i] > kQCutW) ? 1 : 0;
      tp += K.pc[i];
      tq += K.qn[i];
    }
    K.cta_ovf = ovf; K.cta_pc = tp; K.cta_qc = tq;
    K.tie_p = INT_MAX; K.tie_q = INT_MAX;
  }
  int tie_p = INT_MAX, tie_q = INT_MAX;
  bool bad = false;
  if (pp || qp) {  // the ids of the np_cut-th / nq_cut-th cut-value tokens over the cluster
    cluster.sync();
    cluster_copy(cluster, &K.cta_ovf, sm.cv_ovf);
    cluster_copy(cluster, &K.cta_pc, sm.cv_i0);
    cluster_copy(cluster, &K.cta_qc, sm.cv_i1);
    g.sync();  // the copies, before their readers (the values are not written again here)
    long long bp = 0, bq = 0, ap = 0, aq = 0;
    int op = -1, oq = -1;
    for (unsigned r = 0; r < C; ++r) {
      bad |= sm.cv_ovf[r] != 0;
      const int cp = sm.cv_i0[r], cq = sm.cv_i1[r];
      if (r == rank) { bp = ap; bq = aq; }
      if (op < 0 && ap < np_cut && np_cut <= ap + cp) op = (int)r;
      if (oq < 0 && aq < nq_cut && nq_cut <= aq + cq) oq = (int)r;
      ap += cp;
      aq += cq;
    }
    if (!bad && w == 0) {
      if (pp && op == (int)rank) {
        const int id = kth_candidate(K, pr.thr, np_cut - bp);
        if (lane == 0) K.tie_p = id;
      }
      if (qp && oq == (int)rank && lane == 0) K.tie_q = kth_qcut(K, nq_cut - bq);
    }
    cluster.sync();
    if (t == 0 && pp && op >= 0) sm.cv_i0[0] = *cluster.map_shared_rank(&K.tie_p, (unsigned)op);
    if (t == 1 && qp && oq >= 0) sm.cv_i1[0] = *cluster.map_shared_rank(&K.tie_q, (unsigned)oq);
    g.sync();
    if (pp && op >= 0) tie_p = sm.cv_i0[0];
    if (qp && oq >= 0) tie_q = sm.cv_i1[0];
  }
  // weights of the warp's candidates, and their running sums in id order
  pr.tie = pp ? tie_p : INT_MAX;
  qr.tie = qp ? tie_q : INT_MAX;
  float run = 0.f;
  if (!bad && nc <= kKeptW) {
    if (residual)  // q at the candidates' ids (the loads all in flight at once)
      for (int i = lane; i < nc; i += 32)
        K.r[w][i] = QR ? __ldg(reinterpret_cast<const float*>(qrow) + K.id[w][i])
                       : __uint_as_float(load_bits(qrow, K.id[w][i]));
    __syncwarp();
    for (int i0 = 0; i0 < nc; i0 += 32) {
      const int i = i0 + lane;
      float x = 0.f;
      int j = 0;
      if (i < nc) {
        j = K.id[w][i];
        const float v = K.v[w][i];
        const bool kp = v > pr.thr || (v == pr.thr && j <= pr.tie);
        x = kp ? row_weight(pr, v) : 0.f;
        if (residual && x > 0.f) {
          const float vq = K.r[w][i];
          if (QR) {
            x = fmaxf(x - vq, 0.f);  // q as given
          } else {
            const bool kq = vq > qr.thr || (vq == qr.thr && j <= qr.tie);
            if (kq) x = fmaxf(x - row_weight(qr, vq), 0.f);
          }
        }
      }
      float incl = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (i < nc) { K.r[w][i] = x; K.pre[w][i] = run + (incl - x); }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  if (lane == 0) K.wsum[w] = run;
  g.sync();
  if (t == 0) {
    float s = 0.f;
    for (int i = 0; i < kWarps; ++i) { K.wbase[i] = s; s += K.wsum[i]; }
    sm.cta_sum = s;
    sm.cta_ovf = K.cta_ovf;
  }
  cluster.sync();
  cluster_copy(cluster, &sm.cta_ovf, sm.cv_ovf);
  cluster_copy(cluster, &sm.cta_sum, sm.cv_sum);
  cluster.sync();  // every CTA has read the slice totals
  if (t == 0) {
    double W = 0.0, acc = 0.0, cbase = 0.0;
    int owner = -1, lastr = -1, bd = 0;
    for (unsigned r = 0; r < C; ++r) {
      bd |= sm.cv_ovf[r] != 0;
      const double sr = sm.cv_sum[r];
      if (sr > 0.0) lastr = (int)r;
      W += sr;
    }
    const double target = u1 * W;
    for (unsigned r = 0; r < C; ++r) {
      const double sr = sm.cv_sum[r];
      if (sr > 0.0 && acc <= target) { owner = (int)r; cbase = acc; }
      acc += sr;
    }
    if (owner < 0) { owner = lastr; cbase = 0.0; }
    sm.d_W = W; sm.d_target = target; sm.d_base = cbase; sm.d_owner = owner; sm.d_bad = bd;
  }
  g.sync();
  bad |= sm.d_bad != 0;
  const double W = sm.d_W;
  if (bad) return kNaN64;
  if (!(W > 0.0)) return W;
  if (sm.d_owner != (int)rank) return W;
  // the owner: the last candidate with weight whose interval starts at or below the target
  // (a target past every interval, from rounding, takes the last token with weight); the
  // target's offset past the warp's base is rounded down to a float once per warp, so each
  // candidate's start compares exactly as it would with that offset in fp64
  const float dt = __double2float_rd(sm.d_target - (sm.d_base + (double)K.wbase[w]));
  int best = -1;
  for (int i = lane; i < nc; i += 32) {
    const float x = K.r[w][i];
    if (x > 0.f && K.pre[w][i] <= dt) best = i;
  }
  const int wb = __reduce_max_sync(0xFFFFFFFFu, (unsigned)(best + 1)) - 1;
  int anyw = -1;
  for (int i = lane; i < nc; i += 32) if (K.r[w][i] > 0.f) anyw = i;
  const int wl = __reduce_max_sync(0xFFFFFFFFu, (unsigned)(anyw + 1)) - 1;
  if (lane == 0) { K.best[w] = wb; K.last[w] = wl; }
  g.sync();
  if (t == 0) {
    int tok = -1;
    for (int i = kWarps - 1; i >= 0 && tok < 0; --i)
      if (K.best[i] >= 0) tok = K.id[i][K.best[i]];
    if (tok < 0)
      for (int i = kWarps - 1; i >= 0 && tok < 0; --i)
        if (K.last[i] >= 0) tok = K.id[i][K.last[i]];
    *out = tok;
  }
  return W;
}

// Rule 2's draw for session b whose first rejection is a (a == M: the bonus from p_M).
// QR: q is given as rows of binary32 probabilities (A.q_rows), used as given.
template <typename T, bool QR = false>
__device__ void session_draw(const SessIO& A, cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                             unsigned char* ring, int32_t b, int a) {
  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const int64_t M = off1 - off0;
  const int64_t R_T = A.total + A.B;
  const int V = (int)A.V;
  const T* trow = reinterpret_cast<const T*>(A.target) + (off0 + b + a) * (int64_t)V;
  // the residual max(0, p_a - q_a) at Rule 2's first rejection; else a draw from p_a alone
  // (Rule 2's bonus, and every draw of the relaxed rule)
  bool residual = (a < M) && P.rule_id == 2u;
  const T* drow = !residual ? reinterpret_cast<const T*>(A.target) + (off0 + b + a) * (int64_t)V
                  : QR ? reinterpret_cast<const T*>(A.q_rows + (off0 + a) * (int64_t)V)
                       : reinterpret_cast<const T*>(A.draft) + (off0 + a) * (int64_t)V;
  const RowStat sp = sm.stash[0];  // target row a and draft row a, left by the verdict
  const RowStat sq = (residual && !QR) ? sm.stash[1] : sp;
  const float c = profile_c(P.temperature_milli);
  const bool al_p = ((uintptr_t)trow & 15u) == 0, al_q = ((uintptr_t)drow & 15u) == 0;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const bool filt_p = sp.thr_key != 0u || sp.thr_n != INT_MAX;
  const bool filt_q = residual && !QR && (sq.thr_key != 0u || sq.thr_n != INT_MAX);
  DrawRow pr, qr;
  pr.c = qr.c = c;
  pr.lmax = sp.lmax;
  qr.lmax = sq.lmax;
  pr.inv_s = __fdiv_rn(1.f, sp.s);
  qr.inv_s = __fdiv_rn(1.f, sq.s);
  pr.thr = filt_p ? key_value(sp.thr_key) : -INFINITY;
  qr.thr = filt_q ? key_value(sq.thr_key) : -INFINITY;
  pr.tie = INT_MAX;
  qr.tie = INT_MAX;
  // the additional token's random value: only thread 0 forms the draw's target from it
  const double u1 = (threadIdx.x == 0) ? session_uniform(A, b, P, (uint32_t)a, 1u) : 0.0;
  int32_t* out = A.out_tokens + off0 + b + a;
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (QR && residual) {
      // q as given: p's kept tokens where the slices are short, else a pass from global
      // memory (p's cut-value tie found first)
      double W = kNaN64;
      const int np_cut = sp.thr_n;
      if (filt_p && (long long)((V + (int)C - 1) / (int)C) * (long long)sizeof(T) <= kKeptSliceBytes)
        W = draw_kept<T, true>(cluster, g, sm, trow, drow, true, al_p, al_q, V, pr, qr, np_cut, INT_MAX, u1, out);
      if (W != W) {
        pr.tie = (np_cut == INT_MAX) ? INT_MAX : cut_tie_id<T>(cluster, g, sm, trow, al_p, V, pr.thr, np_cut);
        W = filt_p ? draw_token<T, true, true>(cluster, g, sm, trow, drow, true, al_p, al_q, V, pr, qr, u1, out)
                   : draw_token<T, false, true>(cluster, g, sm, trow, drow, true, al_p, al_q, V, pr, qr, u1, out);
      }
      if (!(W > 0.0)) {  // residual mass lost to rounding: use p
        residual = false;
        pr.tie = INT_MAX;
        continue;
      }
      break;
    }
    const bool filt = filt_p || (residual && filt_q);
    const int np_cut = sp.thr_n, nq_cut = residual ? sq.thr_n : INT_MAX;
    const bool ties = np_cut != INT_MAX || nq_cut != INT_MAX;
    double W = kNaN64;
    // first choice where p has a cut and the slices are short: weigh p's kept tokens only
    if (filt_p && (long long)((V + (int)C - 1) / (int)C) * (long long)sizeof(T) <= kKeptSliceBytes)
      W = draw_kept<T>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, np_cut, nq_cut, u1, out);
    // else stream the slice through shared memory (the same decision in every CTA)
    bool ok_all = true;
    for (unsigned r = 0; r < C; ++r) ok_all = ok_all && stream_ok<T>(V, C, r, al_p && (al_q || !residual), ties);
    if (W != W && attempt == 0 && ok_all) {
      if (ties) W = draw_stream<T, true, true>(cluster, g, sm, ring, trow, drow, residual, V, pr, qr, np_cut, nq_cut, u1, out);
      else if (filt) W = draw_stream<T, true, false>(cluster, g, sm, ring, trow, drow, residual, V, pr, qr, np_cut, nq_cut, u1, out);
      else W = draw_stream<T, false, false>(cluster, g, sm, ring, trow, drow, residual, V, pr, qr, np_cut, nq_cut, u1, out);
    }
    if (W != W && ties) {  // from global memory: one pass with the lists, else tie ids first
      W = draw_token_ties<T>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, np_cut, nq_cut, u1, out);
      if (W != W) {
        pr.tie = (np_cut == INT_MAX) ? INT_MAX : cut_tie_id<T>(cluster, g, sm, trow, al_p, V, pr.thr, np_cut);
        qr.tie = (nq_cut == INT_MAX) ? INT_MAX : cut_tie_id<T>(cluster, g, sm, drow, al_q, V, qr.thr, nq_cut);
        W = draw_token<T, true>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, u1, out);
      }
    } else if (W != W) {
      W = filt ? draw_token<T, true>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, u1, out)
               : draw_token<T, false>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, u1, out);
    }
    if (!(W > 0.f) && residual) {  // residual mass lost to rounding: use p
      residual = false;
      pr.tie = INT_MAX;
      continue;
    }
    if (!(W > 0.f) && rank == 0 && threadIdx.x == 0) *out = -1;
    break;
  }
}

// Verdict in every CTA of the cluster (rank 0 writes it), then the draw if Rule 2 needs one.
template <typename T, bool QR = false>
__device__ void complete_session(const SessIO& A, cg::cluster_group& cluster, const Group& g,
                                              SessSmem& sm, unsigned char* ring, int32_t b) {
  if ((threadIdx.x >> 5) == 0) {
    const Verdict v = session_verdict(A, b, cluster.block_rank() == 0, sm.stash);
    if ((threadIdx.x & 31) == 0) { sm.st = v.st; sm.a = v.a; sm.draw = v.draw ? 1 : 0; }
  }
  g.sync();
  const int a = sm.a, draw = sm.draw;
  g.sync();
  if (draw) session_draw<T, QR>(A, cluster, g, sm, ring, b, a);  // the same in every CTA of the cluster
}

}  // namespace sdcp
