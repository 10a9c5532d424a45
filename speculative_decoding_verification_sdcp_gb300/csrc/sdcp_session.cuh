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

#include "sdcp_device.cuh"

namespace sdcp {

constexpr int kSegIds = 32 * kEpt;  // ids per segment: 8 per lane
constexpr int kSegCap = 2048;       // segment-group sums held in shared memory

// Shared memory of one CTA of a session's cluster.
struct SessSmem {
  float seg[kSegCap];  // per segment group of the CTA's slice: weight sums or tie counts
  float fscr[2 * 32 + 4];
  long long lscr[2 * 32 + 4];
  float cta_sum;       // the slice's total weight (read by the cluster)
  long long cta_cnt;   // the slice's tie count (read by the cluster)
  float owner_base;
  long long owner_pre, owner_carry;
  long long result;    // a tie id found by this CTA (read by the cluster)
  int st, a, draw;
};

// Verdict of a session: status, accepted count, and whether Rule 2 still draws a token.
struct Verdict {
  int st, a;
  bool draw;
};

// A row statistic as the other CTAs of the grid left it in L2 (never a stale L1 line).
__device__ __forceinline__ RowStat load_stat(const RowStat* p) {
  union { float4 v[2]; RowStat s; } u;
  u.v[0] = __ldcg(reinterpret_cast<const float4*>(p));
  u.v[1] = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  return u.s;
}

// ---------------------------------------------------------------------------------
// Verdict (one full warp; every lane returns the same value).  Writes status, accepted,
// n_out and every output slot except the drawn token.
// ---------------------------------------------------------------------------------
static __device__ __noinline__ Verdict session_verdict(const SessIO& A, int32_t b, bool write) {
  const int lane = threadIdx.x & 31;
  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const bool offsets_ok = off0 >= 0 && off1 >= off0 && off1 <= A.total && A.m_offsets[0] == 0 &&
                          (int64_t)A.m_offsets[A.B] == A.total;
  const int64_t M = off1 - off0;
  const int64_t R_T = A.total + A.B;
  const int64_t V = A.V;
  const bool rule2 = (P.rule_id == 2u);
  const uint32_t tm = P.temperature_milli;
  const float c = (tm == 0u) ? 0.f : profile_c(tm);
  int st = SDCP_S_OK;
  if ((P.rule_id != 1u && P.rule_id != 2u) || P.top_p_milli > 1000u) st = SDCP_S_BAD_PARAMS;
  else if (!offsets_ok) st = SDCP_S_BAD_PARAMS;
  else if (M < 1 || M > SDCP_MAX_M) st = SDCP_S_LIMIT;
  else if (rule2 && A.draft == nullptr) st = SDCP_S_Q_UNAVAILABLE;
  if (st == SDCP_S_OK && __ldcg(A.error) != 0u) st = SDCP_S_INTERNAL;
  int a = 0;
  int32_t xr[2] = {-1, -1};
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
        if (sp.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
        if (rule2) {
          const RowStat sq = load_stat(A.stats + R_T + off0 + i);
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
            const double u = verifier_uniform(P, (uint32_t)i, 0u);
            rej[h] = !(u < (double)ratio);
          }
        } else {
          rej[h] = (x != sp.argmax);
        }
      }
    }
    if (lane == 0) {  // the bonus / last target row must be valid too
      const RowStat sl = load_stat(A.stats + off0 + b + M);
      if (sl.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
    }
    if (__any_sync(0xFFFFFFFFu, range_bad)) st = SDCP_S_BAD_PROPOSAL;
    else if (__any_sync(0xFFFFFFFFu, row_bad)) st = SDCP_S_BAD_PARAMS;
    else if (rule2 && __any_sync(0xFFFFFFFFu, q_zero)) st = SDCP_S_BAD_PROPOSAL;
    const unsigned r0 = __ballot_sync(0xFFFFFFFFu, rej[0]);
    const unsigned r1 = __ballot_sync(0xFFFFFFFFu, rej[1]);
    a = r0 ? (__ffs(r0) - 1) : (r1 ? 32 + __ffs(r1) - 1 : (int)M);
    if (a > M) a = (int)M;
  }
  const bool ok = (st == SDCP_S_OK);
  const bool draw = ok && rule2 && tm != 0u;
  if (write && lane == 0) {
    A.status[b] = st;
    A.accepted[b] = ok ? a : 0;
    A.n_out[b] = ok ? a + 1 : 0;
  }
  if (write && offsets_ok) {
    const int64_t slot0 = off0 + b;
    int32_t extra = -1;
    if (ok && !draw) extra = load_stat(A.stats + off0 + b + a).argmax;
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

// Weight of token j: p_j = 2^(l_j c - bias) over the kept set, where c = log2(e) 1000/T and
// bias = lmax c + log2(S); kept = value above the cut value, or the cut value and id <= tie
// (values compare as floats: -0 and +0 are one value, as their order keys are).
struct DrawRow {
  float c, bias;
  float thr;  // the cut value (-inf: no cut)
  int tie;    // INT_MAX: every token of the cut value is kept
};
template <bool FILT>
__device__ __forceinline__ float draw_weight(const DrawRow& r, uint32_t bits, int j) {
  const float v = __uint_as_float(bits);
  const float e = ex2(fmaf(v, r.c, -r.bias));
  if (!FILT) return e;
  return (v > r.thr || (v == r.thr && j <= r.tie)) ? e : 0.f;
}

// Raw words of the 8 ids [j0, j0 + 8) of a row: bf16 one 16-byte vector, fp32 two.  Ids at
// or past `end` (and every id of a group that is not 16-byte aligned) are read one by one,
// those past `end` as -inf.
template <typename T> struct Raw8 { static constexpr int W = (sizeof(T) == 2) ? 1 : 2; uint4 v[W]; };

template <typename T>
__device__ __forceinline__ void load_raw8(const T* row, bool aligned16, int end, int j0, Raw8<T>& r) {
  if (aligned16 && j0 + kEpt <= end) {
#pragma unroll
    for (int w = 0; w < Raw8<T>::W; ++w) r.v[w] = __ldg(reinterpret_cast<const uint4*>(row + j0) + w);
  } else {
    uint32_t b[kEpt];
#pragma unroll
    for (int e = 0; e < kEpt; ++e) b[e] = (j0 + e < end) ? load_bits(row, j0 + e) : 0xFF800000u;
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

// The segments of one CTA's slice of a row (ids are int: V <= SDCP_MAX_VOCAB): segments
// [s0, s1) of 256 ids, grouped G at a time into ngrp <= kSegCap groups; warp w owns groups
// [ngrp w / 8, ngrp (w + 1) / 8).
struct SegSlice {
  int nseg, s0, s1, G, ngrp;
  __device__ __forceinline__ SegSlice(int V, unsigned C, unsigned rank) {
    nseg = (V + kSegIds - 1) / kSegIds;
    s0 = (int)((long long)nseg * rank / C);
    s1 = (int)((long long)nseg * (rank + 1) / C);
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
template <typename T, bool FILT>
__device__ __forceinline__ float piece_weights(const Raw8<T>& rp, const Raw8<T>& rq, bool residual,
                                               const DrawRow& pr, const DrawRow& qr, int j0,
                                               float (&w)[kEpt]) {
  uint32_t bp[kEpt], bq[kEpt];
  unpack_raw8<T>(rp, bp);
  if (residual) unpack_raw8<T>(rq, bq);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kEpt; ++e) {
    float x = draw_weight<FILT>(pr, bp[e], j0 + e);
    if (residual) x = fmaxf(x - draw_weight<FILT>(qr, bq[e], j0 + e), 0.f);
    w[e] = x;
    s += x;
  }
  return s;
}

// This CTA's slice: sm.seg[k] = weight of segment group k (ids in order within a group).
template <typename T, bool FILT>
__device__ void draw_pass(const SegSlice& sl, SessSmem& sm, const T* prow, const T* qrow, bool residual,
                          bool al_p, bool al_q, int V, const DrawRow& pr, const DrawRow& qr) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int a, b;
  sl.warp_range(w, kWarps, a, b);
  // segments whose loads are in flight together (fewer with the cut test: registers)
  constexpr int U = ((sizeof(T) == 2) ? 8 : 4) / (FILT ? 2 : 1);
  float gacc = 0.f;
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
      if (kk < b) {
        float wv[kEpt];
        const float ls = piece_weights<T, FILT>(rp[u], rq[u], residual, pr, qr, kk * kSegIds + lane * kEpt, wv);
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
template <typename T, bool FILT>
__device__ int draw_walk(const T* prow, const T* qrow, bool residual, bool al_p, bool al_q, int V,
                         const DrawRow& pr, const DrawRow& qr, int k0, int k1, float carry,
                         float target, bool last_only) {
  const int lane = threadIdx.x & 31;
  int lastpos = -1;
  for (int k = k0; k < k1; ++k) {
    const int j0 = k * kSegIds + lane * kEpt;
    Raw8<T> rp, rq;
    load_raw8<T>(prow, al_p, V, j0, rp);
    if (residual) load_raw8<T>(qrow, al_q, V, j0, rq);
    float wv[kEpt];
    const float ls = piece_weights<T, FILT>(rp, rq, residual, pr, qr, j0, wv);
    int lp = -1;
#pragma unroll
    for (int e = 0; e < kEpt; ++e) if (wv[e] > 0.f) lp = j0 + e;
    lastpos = max(lastpos, __reduce_max_sync(0xFFFFFFFFu, lp));
    if (last_only) continue;
    float incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float tv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += tv;
    }
    const float start = carry + (incl - ls);
    int hit = INT_MAX;
    if (start <= target && target < start + ls) {
      float cc = start;
#pragma unroll
      for (int e = 0; e < kEpt; ++e) {
        cc += wv[e];
        if (hit == INT_MAX && wv[e] > 0.f && cc > target) hit = j0 + e;
      }
    }
    const int found = __reduce_min_sync(0xFFFFFFFFu, hit);
    if (found != INT_MAX) return found;
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  return lastpos;
}

// The draw over the cluster: the token goes to out (by the one CTA that finds it).  Returns
// W, the total weight (the same in every CTA).
template <typename T, bool FILT>
__device__ __noinline__ float draw_token(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                         const T* prow, const T* qrow, bool residual, bool al_p,
                                         bool al_q, int V, const DrawRow& pr, const DrawRow& qr,
                                         double u1, int32_t* out) {
  const int t = threadIdx.x, w = t >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  draw_pass<T, FILT>(sl, sm, prow, qrow, residual, al_p, al_q, V, pr, qr);
  g.sync();
  // this slice's groups in id order: thread t owns groups [t gpt, t gpt + gpt)
  const int gpt = (sl.ngrp + g.nthreads - 1) / g.nthreads;
  float loc = 0.f;
  for (int i = 0; i < gpt; ++i) {
    const int k = t * gpt + i;
    if (k < sl.ngrp) loc += sm.seg[k];
  }
  float Wc;
  const float pre = group_excl_scan(g, loc, sm.fscr, &Wc);
  if (t == 0) sm.cta_sum = Wc;
  cluster.sync();
  // the slices in rank order
  float W = 0.f, base = 0.f;
  int owner = -1, lastr = -1;
  float obase = 0.f;
  for (unsigned r = 0; r < C; ++r) {
    const float sr = *cluster.map_shared_rank(&sm.cta_sum, r);
    if (r == rank) base = W;
    W += sr;
    if (sr > 0.f) lastr = (int)r;
  }
  const float target = (float)(u1 * (double)W);
  {
    float acc = 0.f;
    for (unsigned r = 0; r < C; ++r) {
      const float sr = *cluster.map_shared_rank(&sm.cta_sum, r);
      if (owner < 0 && sr > 0.f && acc <= target && target < acc + sr) { owner = (int)r; obase = acc; }
      acc += sr;
    }
  }
  cluster.sync();  // every CTA has read the slice totals
  if (!(W > 0.f)) return W;
  const bool mine = (owner == (int)rank) || (owner < 0 && lastr == (int)rank);
  if (!mine) return W;
  // this CTA's slice holds the token: its segment group, then the walk
  long long cand = LLONG_MAX, lastg = -1;
  float cbase = 0.f;
  if (owner >= 0) {
    float bsum = obase + pre;
    for (int i = 0; i < gpt; ++i) {
      const int k = t * gpt + i;
      if (k >= sl.ngrp) break;
      const float sk = sm.seg[k];
      if (cand == LLONG_MAX && sk > 0.f && bsum <= target && target < bsum + sk) { cand = k; cbase = bsum; }
      bsum += sk;
    }
  }
  for (int i = 0; i < gpt; ++i) {
    const int k = t * gpt + i;
    if (k < sl.ngrp && sm.seg[k] > 0.f) lastg = k;
  }
  const long long og = group_min_i64(g, cand, sm.lscr);
  if (og != LLONG_MAX && cand == og) sm.owner_base = cbase;
  const long long lg = group_max_i64(g, lastg, sm.lscr);
  g.sync();
  if (w == 0) {
    int tok;
    if (og != LLONG_MAX) {
      tok = draw_walk<T, FILT>(prow, qrow, residual, al_p, al_q, V, pr, qr, sl.grp_lo((int)og),
                               sl.grp_hi((int)og), sm.owner_base, target, false);
    } else {  // u * W rounded up to the end: the largest id with positive weight
      tok = draw_walk<T, FILT>(prow, qrow, residual, al_p, al_q, V, pr, qr, sl.grp_lo((int)lg),
                               sl.grp_hi((int)lg), 0.f, 0.f, true);
    }
    if ((t & 31) == 0) *out = tok;
  }
  return W;
}

// Id of the n-th token (1-based, id order) with value `val` over the cluster (every CTA
// gets it); INT_MAX if none.
template <typename T>
__device__ __noinline__ int cut_tie_id(cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                                       const T* row, bool al, int V, float val, int n) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned C = cluster.num_blocks(), rank = cluster.block_rank();
  const SegSlice sl(V, C, rank);
  int a, b;
  sl.warp_range(w, kWarps, a, b);
  constexpr int U = (sizeof(T) == 2) ? 16 : 8;
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
  long long base = 0, acc = 0;
  int owner = -1;
  for (unsigned r = 0; r < C; ++r) {
    const long long cr = *cluster.map_shared_rank(&sm.cta_cnt, r);
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
  const long long id = (owner >= 0) ? *cluster.map_shared_rank(&sm.result, (unsigned)owner) : LLONG_MAX;
  cluster.sync();  // the owner's shared memory is read before anyone moves on
  return (id == LLONG_MAX || id == INT_MAX) ? INT_MAX : (int)id;
}

// Rule 2's draw for session b whose first rejection is a (a == M: the bonus from p_M).
template <typename T>
__device__ void session_draw(const SessIO& A, cg::cluster_group& cluster, const Group& g, SessSmem& sm,
                             int32_t b, int a) {
  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const int64_t M = off1 - off0;
  const int64_t R_T = A.total + A.B;
  const int V = (int)A.V;
  const T* trow = reinterpret_cast<const T*>(A.target) + (off0 + b + a) * (int64_t)V;
  const T* drow = reinterpret_cast<const T*>(A.draft) + (off0 + (a < M ? a : 0)) * (int64_t)V;
  const RowStat sp = load_stat(A.stats + off0 + b + a);
  const RowStat sq = (a < M) ? load_stat(A.stats + R_T + off0 + a) : sp;
  const float c = profile_c(P.temperature_milli);
  const bool al_p = ((uintptr_t)trow & 15u) == 0, al_q = ((uintptr_t)drow & 15u) == 0;
  bool residual = (a < M);
  const bool filt_p = sp.thr_key != 0u || sp.thr_n != INT_MAX;
  const bool filt_q = residual && (sq.thr_key != 0u || sq.thr_n != INT_MAX);
  DrawRow pr, qr;
  pr.c = qr.c = c;
  pr.bias = fmaf(sp.lmax, c, log2f(sp.s));
  qr.bias = fmaf(sq.lmax, c, log2f(sq.s));
  pr.thr = filt_p ? key_value(sp.thr_key) : -INFINITY;
  qr.thr = filt_q ? key_value(sq.thr_key) : -INFINITY;
  // id bound of the kept tokens at the cut value, where the cut falls inside a value
  pr.tie = (sp.thr_n == INT_MAX) ? INT_MAX : cut_tie_id<T>(cluster, g, sm, trow, al_p, V, pr.thr, sp.thr_n);
  qr.tie = (!residual || sq.thr_n == INT_MAX) ? INT_MAX
                                              : cut_tie_id<T>(cluster, g, sm, drow, al_q, V, qr.thr, sq.thr_n);
  const double u1 = verifier_uniform(P, (uint32_t)a, 1u);
  const bool filt = filt_p || filt_q;
  int32_t* out = A.out_tokens + off0 + b + a;
  for (int attempt = 0; attempt < 2; ++attempt) {
    const float W = filt ? draw_token<T, true>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, u1, out)
                         : draw_token<T, false>(cluster, g, sm, trow, drow, residual, al_p, al_q, V, pr, qr, u1, out);
    if (!(W > 0.f) && residual) { residual = false; continue; }  // residual mass lost to rounding: use p
    if (!(W > 0.f) && cluster.block_rank() == 0 && threadIdx.x == 0) *out = -1;
    break;
  }
}

// Verdict in every CTA of the cluster (rank 0 writes it), then the draw if Rule 2 needs one.
template <typename T>
__device__ __noinline__ void complete_session(const SessIO& A, cg::cluster_group& cluster, const Group& g,
                                              SessSmem& sm, int32_t b) {
  if ((threadIdx.x >> 5) == 0) {
    const Verdict v = session_verdict(A, b, cluster.block_rank() == 0);
    if ((threadIdx.x & 31) == 0) { sm.st = v.st; sm.a = v.a; sm.draw = v.draw ? 1 : 0; }
  }
  g.sync();
  const int a = sm.a, draw = sm.draw;
  g.sync();
  if (draw) session_draw<T>(A, cluster, g, sm, b, a);  // the same in every CTA of the cluster
}

}  // namespace sdcp
