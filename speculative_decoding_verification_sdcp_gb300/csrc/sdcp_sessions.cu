// sdcp_sessions.cu - phase 2 of the acceptance step: per session, the precondition,
// the acceptance tests, the first rejection, and the additional token (SDCP draft
// draft-li-mlc-inference-acceleration-00, Section 6.3 "Preconditions of the rule" and
// Section 6.4 Rules 1 and 2; verdict fields of Section 5.2).
//
// One thread-block cluster per session, launched as a programmatic dependent of the row
// kernel: it reads its inputs (parameters, offsets, tokens) while the row kernel still
// runs, then waits for the row statistics.  Every CTA of the cluster evaluates the M
// acceptance tests from the row statistics (one lane per position, fp64 ratio, Philox
// uniform of purpose 0) and takes the first rejection a with a ballot; rank 0 writes the
// verdict.  Rule 2 then needs one draw: from the residual max(0, p_a - q_a) when a < M,
// from p_M otherwise (purpose 1).  The cluster splits the ids into slices, each thread of
// a CTA sums the weights of one contiguous run of ids, a block scan orders the runs, the
// slice totals are exchanged through distributed shared memory, and the thread whose run
// holds u * W walks it again to find the smallest id whose cumulative weight exceeds u*W.
#include "sdcp_device.cuh"

namespace sdcp {

struct SliceInfo {
  float total;
  int pad;
  long long lastpos;  // largest id with positive weight in the slice (-1: none)
};

struct SessSmem {
  int st, a;
  int x[SDCP_MAX_M];
  SliceInfo slice;
  long long tie_slice, tie_found;
  long long w_cnt[kWarps], w_cpre[kWarps];
  float w_sum[kWarps], w_pre[kWarps];
  long long w_last[kWarps];
  float fscr[3 * kWarps + 4];
  long long lscr[3 * kWarps + 4];
};

// Weight of token j for the draw: p_j (bonus, or residual fallen back to p) or
// max(0, p_j - q_j) (residual).  p_j = exp((l_j - lmax) * 1000/T) / S over the kept set.
struct DrawRow {
  float lmax, cexp, inv_s;
  uint32_t thr_key;
  long long thr_id;
};
__device__ __forceinline__ float prob_of(const DrawRow& r, uint32_t bits, long long j) {
  const uint32_t k = order_key(bits);
  const bool kept = k > r.thr_key || (k == r.thr_key && j <= r.thr_id);
  return kept ? ex2((__uint_as_float(bits) - r.lmax) * r.cexp) * r.inv_s : 0.f;
}

// kEpt consecutive elements from j0 (j0 % 8 == 0); past `end` they read as -inf.
template <typename T>
__device__ __forceinline__ void load8(const T* row, bool aligned16, int64_t end, int64_t j0,
                                      uint32_t (&b)[kEpt]) {
  if (aligned16 && j0 + kEpt <= end) {
    if (sizeof(T) == 2) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(row + j0));
      uint32_t t[8];
      Elem<__nv_bfloat16>::unpack(q, t);
#pragma unroll
      for (int e = 0; e < kEpt; ++e) b[e] = t[e];
    } else {
      const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(row + j0));
      const uint4 q1 = __ldg(reinterpret_cast<const uint4*>(row + j0 + 4));
      b[0] = q0.x; b[1] = q0.y; b[2] = q0.z; b[3] = q0.w;
      b[4] = q1.x; b[5] = q1.y; b[6] = q1.z; b[7] = q1.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kEpt; ++e) b[e] = (j0 + e < end) ? load_bits(row, j0 + e) : 0xFF800000u;
  }
}

// Raw words of the 8 ids [j0, j0 + 8) of a row: bf16 one 16-byte vector, fp32 two.  Ids at
// or past `end` (and every id of a group that is not 16-byte aligned) are read one by one,
// those past `end` as -inf.
template <typename T> struct Raw8 { static constexpr int W = (sizeof(T) == 2) ? 1 : 2; uint4 v[W]; };

template <typename T>
__device__ __forceinline__ void load_raw8(const T* row, bool aligned16, int64_t end, int64_t j0, Raw8<T>& r) {
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

template <typename T>
__device__ __forceinline__ void weights8(const T* prow, const T* qrow, bool residual, const DrawRow& pr,
                                         const DrawRow& qr, bool al_p, bool al_q, int64_t end,
                                         int64_t j0, float (&w)[kEpt]) {
  uint32_t bp[kEpt];
  load8<T>(prow, al_p, end, j0, bp);
  if (residual) {
    uint32_t bq[kEpt];
    load8<T>(qrow, al_q, end, j0, bq);
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
      const bool in = j0 + e < end;
      const float p = in ? prob_of(pr, bp[e], j0 + e) : 0.f;
      const float q = in ? prob_of(qr, bq[e], j0 + e) : 0.f;
      w[e] = fmaxf(p - q, 0.f);
    }
  } else {
#pragma unroll
    for (int e = 0; e < kEpt; ++e) w[e] = (j0 + e < end) ? prob_of(pr, bp[e], j0 + e) : 0.f;
  }
}

// Id of the n-th token (1-based, id order) whose order key is `key`, over the cluster.  Each
// warp counts its chunk (coalesced 256-id segments), the warps' counts in id order and the
// slices' totals (distributed shared memory) locate the chunk holding it, and that chunk's
// warp walks it again with a warp scan.  A row cut inside one value keeps the first tokens
// of that value; this finds the id bound of the kept ones.
template <typename T>
__device__ long long cut_tie_id(cg::cluster_group& cluster, unsigned C, unsigned rank, SessSmem& sm,
                                const T* row, bool aligned, int64_t wl, int64_t wh, uint32_t key,
                                long long n) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int64_t kSeg = 32 * kEpt;
  constexpr int U = 4;
  long long cnt = 0;
  for (int64_t s0 = wl; s0 < wh; s0 += U * kSeg) {
    Raw8<T> r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t j0 = s0 + u * kSeg + (int64_t)lane * kEpt;
      if (j0 < wh) load_raw8<T>(row, aligned, wh, j0, r[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t j0 = s0 + u * kSeg + (int64_t)lane * kEpt;
      if (j0 >= wh) continue;
      uint32_t b[kEpt];
      unpack_raw8<T>(r[u], b);
#pragma unroll
      for (int e = 0; e < kEpt; ++e) cnt += (j0 + e < wh && order_key(b[e]) == key) ? 1 : 0;
    }
  }
  cnt = warp_sum_ll(cnt);
  if (lane == 0) sm.w_cnt[wid] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long acc = 0;
    for (int i = 0; i < kWarps; ++i) { sm.w_cpre[i] = acc; acc += sm.w_cnt[i]; }
    sm.tie_slice = acc;
    sm.tie_found = -1;
  }
  cluster.sync();
  long long base = 0, acc = 0;
  int owner = -1;
  for (unsigned r = 0; r < C; ++r) {
    const long long tr = *cluster.map_shared_rank(&sm.tie_slice, r);
    if (r == rank) base = acc;
    if (owner < 0 && acc < n && n <= acc + tr) owner = (int)r;
    acc += tr;
  }
  if ((unsigned)owner == rank) {
    const long long pre = base + sm.w_cpre[wid];
    if (pre < n && n <= pre + sm.w_cnt[wid]) {  // this warp's chunk holds it
      long long carry = pre;
      for (int64_t s0 = wl; s0 < wh; s0 += kSeg) {
        const int64_t j0 = s0 + (int64_t)lane * kEpt;
        uint32_t b[kEpt];
        int c = 0;
        if (j0 < wh) {
          Raw8<T> r;
          load_raw8<T>(row, aligned, wh, j0, r);
          unpack_raw8<T>(r, b);
#pragma unroll
          for (int e = 0; e < kEpt; ++e) c += (j0 + e < wh && order_key(b[e]) == key) ? 1 : 0;
        }
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int tv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += tv;
        }
        const long long lane_pre = carry + (incl - c);
        if (c > 0 && lane_pre < n && n <= lane_pre + c) {
          long long k = lane_pre;
          for (int e = 0; e < kEpt; ++e)
            if (j0 + e < wh && order_key(b[e]) == key && ++k == n) { sm.tie_found = j0 + e; break; }
        }
        const long long total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        if (carry + total >= n) break;
        carry += total;
      }
    }
  }
  cluster.sync();
  const long long id = (owner >= 0) ? *cluster.map_shared_rank(&sm.tie_found, (unsigned)owner) : -1;
  cluster.sync();  // the owner's shared memory is read before anyone moves on
  return id < 0 ? LLONG_MAX : id;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 3) session_kernel(SessArgs A) {
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned C = cluster.num_blocks();
  const unsigned rank = cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31;
  const int32_t b = (int32_t)(blockIdx.x / C);
  __shared__ SessSmem sm;

  // ---- inputs of the call (not written by the row kernel): read before the wait -------
  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const bool offsets_ok = off0 >= 0 && off1 >= off0 && off1 <= A.total &&
                          A.m_offsets[0] == 0 && (int64_t)A.m_offsets[A.B] == A.total;
  const int64_t M = off1 - off0;
  const int64_t R_T = A.total + A.B;
  const int64_t V = A.V;
  const bool rule2 = (P.rule_id == 2u);
  const uint32_t tm = P.temperature_milli;
  int st0 = SDCP_S_OK;
  if ((P.rule_id != 1u && P.rule_id != 2u) || P.top_p_milli > 1000u) st0 = SDCP_S_BAD_PARAMS;
  else if (!offsets_ok) st0 = SDCP_S_BAD_PARAMS;
  else if (M < 1 || M > SDCP_MAX_M) st0 = SDCP_S_LIMIT;
  else if (rule2 && A.draft == nullptr) st0 = SDCP_S_Q_UNAVAILABLE;
  if (tid < 32 && st0 == SDCP_S_OK) {
    for (int i = lane; i < M; i += 32) sm.x[i] = A.tokens[off0 + i];
  }

  pdl_wait_primary();  // row statistics and the error word are complete from here on

  // ---- status and the acceptance scan (warp 0; identical in every CTA) -------------
  if (tid < 32) {
    int st = st0;
    if (st == SDCP_S_OK && *A.error != 0u) st = SDCP_S_INTERNAL;
    int a = 0;
    if (st == SDCP_S_OK) {
      bool range_bad = false, row_bad = false, q_zero = false;
      bool rej[2] = {false, false};
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < M) {
          const int32_t x = sm.x[i];
          if (x < 0 || (int64_t)x >= V) range_bad = true;
          const RowStat sp = A.stats[off0 + b + i];
          if (sp.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
          if (rule2) {
            const RowStat sq = A.stats[R_T + off0 + i];
            if (sq.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED)) row_bad = true;
            if (!(sq.flags & SDCP_ROW_X_KEPT)) q_zero = true;
            if (tm == 0u) {
              rej[h] = (x != sp.argmax);
            } else {
              const double scale = 1000.0 / (double)tm;
              const double lp = (sp.flags & SDCP_ROW_X_KEPT)
                                    ? (double)sp.dlx * scale - log((double)sp.s) : -INFINITY;
              const double lq = (double)sq.dlx * scale - log((double)sq.s);
              double ratio = (lp == -INFINITY) ? 0.0 : exp(lp - lq);
              ratio = ratio > 1.0 ? 1.0 : ratio;
              const double u = verifier_uniform(P, (uint32_t)i, 0u);
              rej[h] = !(u < ratio);
            }
          } else {
            rej[h] = (x != sp.argmax);
          }
        }
      }
      {  // the bonus / last target row must be valid too
        const RowStat sl = A.stats[off0 + b + M];
        if (lane == 0 && (sl.flags & (SDCP_ROW_INVALID | SDCP_ROW_SKIPPED))) row_bad = true;
      }
      if (__any_sync(0xFFFFFFFFu, range_bad)) st = SDCP_S_BAD_PROPOSAL;
      else if (__any_sync(0xFFFFFFFFu, row_bad)) st = SDCP_S_BAD_PARAMS;
      else if (rule2 && __any_sync(0xFFFFFFFFu, q_zero)) st = SDCP_S_BAD_PROPOSAL;
      const unsigned r0 = __ballot_sync(0xFFFFFFFFu, rej[0]);
      const unsigned r1 = __ballot_sync(0xFFFFFFFFu, rej[1]);
      a = r0 ? (__ffs(r0) - 1) : (r1 ? 32 + __ffs(r1) - 1 : (int)M);
      if (a > M) a = (int)M;
    }
    if (lane == 0) { sm.st = st; sm.a = a; }
  }
  __syncthreads();
  const int st = sm.st, a = sm.a;

  // ---- the verdict (rank 0) ------------------------------------------------------------
  const bool need_draw = (st == SDCP_S_OK) && rule2 && tm != 0u;
  if (rank == 0) {
    const int64_t slot0 = off0 + b;
    if (tid == 0) {
      A.status[b] = st;
      A.accepted[b] = (st == SDCP_S_OK) ? a : 0;
      A.n_out[b] = (st == SDCP_S_OK) ? a + 1 : 0;
    }
    if (offsets_ok) {
      for (int64_t j = tid; j <= M; j += kThreads) {
        int v = -1;
        if (st == SDCP_S_OK) {
          if (j < a) v = sm.x[j];
          else if (j == a) {
            if (need_draw) continue;  // written once, by the thread that finds the draw
            v = A.stats[off0 + b + a].argmax;
          }
        }
        A.out_tokens[slot0 + j] = v;
      }
    }
  }
  if (!need_draw) return;  // uniform over the cluster

  // ---- the draw: residual max(0, p_a - q_a) if a < M, else p_M ---------------------
  const T* trow = reinterpret_cast<const T*>(A.target) + (off0 + b + a) * V;
  const T* drow = reinterpret_cast<const T*>(A.draft) + (off0 + (a < M ? a : 0)) * V;
  const RowStat sp = A.stats[off0 + b + a];
  const RowStat sq = (a < M) ? A.stats[R_T + off0 + a] : sp;
  const float cexp = (float)(1000.0 / (double)tm * 1.4426950408889634);
  const bool al_p = ((uintptr_t)trow & 15u) == 0, al_q = ((uintptr_t)drow & 15u) == 0;
  // slice of this CTA, and chunk of each warp in it (multiples of 8 ids), read in coalesced
  // 256-id segments
  const int64_t lo = (rank == 0) ? 0 : ((V * rank / C) & ~(int64_t)7);
  const int64_t hi = (rank == C - 1) ? V : ((V * (rank + 1) / C) & ~(int64_t)7);
  const int wid = tid >> 5;
  const int64_t span = hi - lo;
  const int64_t wl = lo + ((span * wid / kWarps) & ~(int64_t)7);
  const int64_t wh = (wid == kWarps - 1) ? hi : lo + ((span * (wid + 1) / kWarps) & ~(int64_t)7);
  constexpr int64_t kSeg = 32 * kEpt;
  // id bound of the kept tokens at the cut value, where the cut falls inside a value
  const long long p_tie = (sp.thr_n == INT_MAX) ? LLONG_MAX
                          : cut_tie_id<T>(cluster, C, rank, sm, trow, al_p, wl, wh, sp.thr_key, sp.thr_n);
  const long long q_tie = (a >= M || sq.thr_n == INT_MAX) ? LLONG_MAX
                          : cut_tie_id<T>(cluster, C, rank, sm, drow, al_q, wl, wh, sq.thr_key, sq.thr_n);
  const DrawRow pr{sp.lmax, cexp, 1.f / sp.s, sp.thr_key, p_tie};
  const DrawRow qr{sq.lmax, cexp, 1.f / sq.s, sq.thr_key, q_tie};
  const double u1 = verifier_uniform(P, (uint32_t)a, 1u);

  bool residual = (a < M);
  for (int attempt = 0; attempt < 2; ++attempt) {
    // pass 1: each lane sums its 8-id pieces of every segment of the warp's chunk; the
    // loads of U segments are issued before any of their arithmetic
    float ls = 0.f;
    long long lastpos = -1;
    constexpr int U = (sizeof(T) == 2) ? 4 : 2;
    for (int64_t s0 = wl; s0 < wh; s0 += U * kSeg) {
      Raw8<T> rp[U], rq[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j0 = s0 + u * kSeg + (int64_t)lane * kEpt;
        if (j0 < wh) {
          load_raw8<T>(trow, al_p, wh, j0, rp[u]);
          if (residual) load_raw8<T>(drow, al_q, wh, j0, rq[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j0 = s0 + u * kSeg + (int64_t)lane * kEpt;
        if (j0 >= wh) continue;
        uint32_t bp[kEpt], bq[kEpt];
        unpack_raw8<T>(rp[u], bp);
        if (residual) unpack_raw8<T>(rq[u], bq);
#pragma unroll
        for (int e = 0; e < kEpt; ++e) {
          const int64_t j = j0 + e;
          float w = (j < wh) ? prob_of(pr, bp[e], j) : 0.f;
          if (residual) w = fmaxf(w - ((j < wh) ? prob_of(qr, bq[e], j) : 0.f), 0.f);
          ls += w;
          if (w > 0.f) lastpos = j;
        }
      }
    }
    const float wtot = warp_reduce(ls, [](float x, float y) { return x + y; });
    const long long wlast = warp_max_i64(lastpos);
    if (lane == 0) { sm.w_sum[wid] = wtot; sm.w_last[wid] = wlast; }
    __syncthreads();
    if (tid == 0) {  // warps in id order
      float acc = 0.f;
      long long sl = -1;
      for (int i = 0; i < kWarps; ++i) { sm.w_pre[i] = acc; acc += sm.w_sum[i]; sl = max(sl, sm.w_last[i]); }
      sm.slice.total = acc;
      sm.slice.lastpos = sl;
    }
    cluster.sync();
    float W = 0.f, base = 0.f;
    long long glast = -1;
    for (unsigned r = 0; r < C; ++r) {
      const SliceInfo si = *cluster.map_shared_rank(&sm.slice, r);
      if (r == rank) base = W;
      W += si.total;
      glast = max(glast, si.lastpos);
    }
    const bool retry = !(W > 0.f) && residual;  // residual mass lost to rounding: use p
    float target = 0.f;
    int owner = -1;
    if (!retry && W > 0.f) {
      target = (float)(u1 * (double)W);
      float acc = 0.f;
      for (unsigned r = 0; r < C; ++r) {
        const SliceInfo si = *cluster.map_shared_rank(&sm.slice, r);
        const float nxt = acc + si.total;
        if (owner < 0 && acc <= target && target < nxt) owner = (int)r;
        acc = nxt;
      }
    }
    cluster.sync();  // every CTA is done reading the slice totals
    if (retry) { residual = false; continue; }
    if (owner < 0) {
      // u * W rounded up to W: the largest id with positive weight (-1 if none)
      if (rank == 0 && tid == 0) A.out_tokens[off0 + b + a] = (int32_t)glast;
      break;
    }
    if ((unsigned)owner != rank) break;
    // the owner CTA: the warp whose chunk holds the target walks it segment by segment,
    // a warp scan carrying the cumulative weight
    int ow = -1;
    long long olast = -1;
    for (int i = 0; i < kWarps; ++i) {
      const float st = base + sm.w_pre[i];
      if (st <= target) olast = max(olast, sm.w_last[i]);
      if (ow < 0 && st <= target && target < st + sm.w_sum[i]) ow = i;
    }
    if (wid == ow) {
      float carry = base + sm.w_pre[ow];
      long long found = LLONG_MAX, wlastp = -1;
      for (int64_t s0 = wl; s0 < wh && found == LLONG_MAX; s0 += kSeg) {
        const int64_t j0 = s0 + (int64_t)lane * kEpt;
        float w[kEpt];
        float lsum = 0.f;
        long long lp = -1;
        if (j0 < wh) {
          weights8<T>(trow, drow, residual, pr, qr, al_p, al_q, wh, j0, w);
#pragma unroll
          for (int e = 0; e < kEpt; ++e) { lsum += w[e]; if (w[e] > 0.f) lp = j0 + e; }
        }
        float incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float tv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += tv;
        }
        const float lane_start = carry + (incl - lsum);
        long long hit = LLONG_MAX;
        if (j0 < wh && lane_start <= target && lane_start + lsum > target) {
          float cc = lane_start;
#pragma unroll
          for (int e = 0; e < kEpt; ++e) {
            cc += w[e];
            if (hit == LLONG_MAX && w[e] > 0.f && cc > target) hit = j0 + e;
          }
        }
        found = warp_min_i64(hit);
        if (lane_start <= target) wlastp = max(wlastp, lp);
        wlastp = warp_max_i64(wlastp);
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) A.out_tokens[off0 + b + a] = (int32_t)(found != LLONG_MAX ? found : max(wlastp, olast));
    } else if (ow < 0 && tid == 0) {
      A.out_tokens[off0 + b + a] = (int32_t)olast;  // rounding left no warp: last positive
    }
    break;
  }
}

template __global__ void session_kernel<float>(SessArgs);
template __global__ void session_kernel<__nv_bfloat16>(SessArgs);

int launch_sessions(const SessArgs& a, int dtype, int cluster, bool pdl, cudaStream_t stream) {
  if (a.B <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.B * cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  cudaError_t e;
  if (dtype == SDCP_BF16)
    e = cudaLaunchKernelEx(&cfg, session_kernel<__nv_bfloat16>, a);
  else
    e = cudaLaunchKernelEx(&cfg, session_kernel<float>, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp
