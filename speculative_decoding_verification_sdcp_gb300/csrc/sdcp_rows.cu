// sdcp_rows.cu - phase 1 of the acceptance step: per-row statistics of the sampling
// profile (SDCP draft draft-li-mlc-inference-acceleration-00, Section 4.1: temperature,
// then top-k, then top-p; temperature 0 selects the argmax, ties to the smallest id).
//
// One thread-block cluster of C CTAs per logits row (C = 1..8).  CTA r of the cluster
// streams slice r of the row from HBM once (16-byte non-allocating loads) and keeps, per
// thread, the running maximum and the sum of exp relative to it (online softmax), or the
// order-key maximum with its smallest id when the row needs an argmax.  The CTAs merge
// their partials in rank order through distributed shared memory, so every result is
// independent of scheduling.
//
// Top-k / top-p on bf16 rows: one more pass over the row (it is still in L2) builds an
// exact-value histogram of the 2048 bf16 values just below the row maximum (integer
// shared-memory atomics: deterministic).  Because all tokens that share a bf16 value have
// the same probability, the mass of a bin is count * exp(value - max): the k-th token and
// the top-p crossing come out of one block scan over the bins.  A tie at the cut value is
// broken by id with a cluster-wide list of the tied ids.  Rows the window cannot decide
// (fp32 logits with filters, or a distribution too flat for 2048 bins) take a generic
// bisection over the order-key space on the cluster's rank 0.
#include "sdcp_device.cuh"

namespace sdcp {


// What one CTA publishes for its cluster after the streaming pass.
struct Partial {
  float fm;        // running maximum used as the reference of s
  float s;         // sum of exp((l - fm) * scale) over the slice
  uint32_t kmax;   // largest order key
  uint32_t kmin;   // smallest order key
  long long amax;  // smallest id holding kmax (LLONG_MAX: none)
  int bad;         // NaN seen (sum mode)
  int pad;
};

// Decision of rank 0 after the window histogram, read by the cluster.
struct Decision {
  int use_fallback;
  int need_tie;
  uint32_t tie_key16;
  int tie_n;        // 1-based rank (id order) of the last kept token among the tied ones
  uint32_t thr_key;
  int kept;
  float s_kept;
  int pad;
};

struct __align__(16) RowSmem {
  Partial part;
  Decision dec;
  uint32_t hist[kWindowBins];
  int tie_count;
  int tie_ids[kTieListCap];
  float fscr[3 * kWarps + 4];
  long long lscr[3 * kWarps + 4];
  // broadcast slots of rank 0's scans
  int b_dk, b_tk, b_dp, b_np, b_found;
  float b_sk1, b_massbefore_p, b_s_kept;
  int b_countbefore_p;
  int b_tie_id;
};

// --------------------------------------------------------------------------------------
// Streaming pass over a set of elements.
// --------------------------------------------------------------------------------------
struct ThreadAcc {
  float fm, s;
  uint32_t kmax, kmin;
  long long amax;
  int bad;
};

// FMODE: 0 no float statistics, 1 running maximum only, 2 maximum and online sum.
template <bool KEYS, int FMODE>
__device__ __forceinline__ void acc_element(ThreadAcc& a, uint32_t bits, long long id, float c) {
  if (KEYS) {
    uint32_t k = order_key(bits);
    if (k > a.kmax) { a.kmax = k; a.amax = id; }
    a.kmin = min(a.kmin, k);
  }
  if (FMODE >= 1) {
    float v = __uint_as_float(bits);
    if (v != v) a.bad = 1;
    if (v > a.fm) {
      if (FMODE == 2) a.s = a.s * ex2((a.fm - v) * c);
      a.fm = v;
    }
    if (FMODE == 2 && a.fm != -INFINITY) a.s += ex2((v - a.fm) * c);
  }
}

template <typename T, bool KEYS, int FMODE>
__device__ __forceinline__ void acc_vector(ThreadAcc& a, const uint4& q, long long id0, float c) {
  constexpr int E = Elem<T>::kPerVec;
  uint32_t b[E];
  Elem<T>::unpack(q, b);
  if (KEYS) {
    uint32_t k[E];
    uint32_t vmax = 0, vmin = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < E; ++e) { k[e] = order_key(b[e]); vmax = max(vmax, k[e]); vmin = min(vmin, k[e]); }
    a.kmin = min(a.kmin, vmin);
    if (vmax > a.kmax) {
      int first = E - 1;
#pragma unroll
      for (int e = E - 1; e >= 0; --e) if (k[e] == vmax) first = e;
      a.kmax = vmax;
      a.amax = id0 + first;
    }
  }
  if (FMODE >= 1) {
    float v[E];
    float vm = -INFINITY;
#pragma unroll
    for (int e = 0; e < E; ++e) { v[e] = __uint_as_float(b[e]); vm = fmax_nan(vm, v[e]); }
    if (vm != vm) a.bad = 1;
    if (vm > a.fm) {
      if (FMODE == 2) a.s = a.s * ex2((a.fm - vm) * c);
      a.fm = vm;
    }
    if (FMODE == 2 && a.fm != -INFINITY) {
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) t += ex2((v[e] - a.fm) * c);
      a.s += t;
    }
  }
}

// Elements [e_lo, e_hi) of the row, split as head / vectors / tail.
template <typename T, bool KEYS, int FMODE>
__device__ void stream_slice(const T* __restrict__ row, const RowLayout& L, int64_t vec_lo,
                             int64_t vec_hi, bool head, bool tail, int64_t V, float c,
                             ThreadAcc& a) {
  constexpr int E = Elem<T>::kPerVec;
  const int tid = threadIdx.x;
  if (head) {
    for (int64_t j = tid; j < L.head; j += kThreads) acc_element<KEYS, FMODE>(a, load_bits(row, j), j, c);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(row + L.head);
  constexpr int U = 4;
  int64_t v = vec_lo + tid;
  for (; v + (U - 1) * kThreads < vec_hi; v += U * kThreads) {
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) q[u] = ld_stream(vp + v + u * kThreads);
#pragma unroll
    for (int u = 0; u < U; ++u) acc_vector<T, KEYS, FMODE>(a, q[u], L.head + (v + u * kThreads) * E, c);
  }
  for (; v < vec_hi; v += kThreads) acc_vector<T, KEYS, FMODE>(a, ld_stream(vp + v), L.head + v * E, c);
  if (tail) {
    for (int64_t j = L.tail0 + tid; j < V; j += kThreads) acc_element<KEYS, FMODE>(a, load_bits(row, j), j, c);
  }
}

// --------------------------------------------------------------------------------------
// Generic element visitor over a slice (used by the window, tie and fallback passes).
// --------------------------------------------------------------------------------------
template <typename T, typename F>
__device__ __forceinline__ void visit_slice(const T* __restrict__ row, const RowLayout& L,
                                            int64_t vec_lo, int64_t vec_hi, bool head, bool tail,
                                            int64_t V, F f) {
  constexpr int E = Elem<T>::kPerVec;
  const int tid = threadIdx.x;
  if (head)
    for (int64_t j = tid; j < L.head; j += kThreads) f(load_bits(row, j), j);
  const uint4* vp = reinterpret_cast<const uint4*>(row + L.head);
  for (int64_t v = vec_lo + tid; v < vec_hi; v += kThreads) {
    uint4 q = __ldg(vp + v);
    uint32_t b[E];
    Elem<T>::unpack(q, b);
    long long id0 = L.head + v * E;
#pragma unroll
    for (int e = 0; e < E; ++e) f(b[e], id0 + e);
  }
  if (tail)
    for (int64_t j = L.tail0 + tid; j < V; j += kThreads) f(load_bits(row, j), j);
}

// Whole-row generic passes run by one CTA (the fallback).
template <typename T>
struct WholeRow {
  const T* row;
  RowLayout L;
  int64_t V;
  template <typename F>
  __device__ __forceinline__ void visit(F f) const { visit_slice<T>(row, L, 0, L.nvec, true, true, V, f); }
};

// Id (1-based rank n in id order) among the tokens whose key satisfies pred, by one CTA:
// each thread owns a contiguous chunk of ids, counts, scans, and the owner walks.
template <typename T, typename P>
__device__ long long nth_matching_id(const WholeRow<T>& R, long long n, P pred, long long* lscr) {
  const int tid = threadIdx.x;
  int64_t chunk = (R.V + kThreads - 1) / kThreads;
  int64_t j0 = (int64_t)tid * chunk, j1 = min(R.V, j0 + chunk);
  long long cnt = 0;
  for (int64_t j = j0; j < j1; ++j) cnt += pred(load_bits(R.row, j), j) ? 1 : 0;
  long long tot;
  long long excl = block_exclusive_scan_ll(cnt, lscr, &tot);
  long long found = LLONG_MAX;
  if (excl < n && n <= excl + cnt) {
    long long c = excl;
    for (int64_t j = j0; j < j1; ++j) {
      if (pred(load_bits(R.row, j), j)) {
        if (++c == n) { found = j; break; }
      }
    }
  }
  return block_min_i64(found, lscr);
}

// --------------------------------------------------------------------------------------
// The row kernel.
// --------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(RowArgs A) {
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned C = cluster.num_blocks();
  const unsigned rank = cluster.block_rank();
  const int tid = threadIdx.x;
  const int64_t row_id = (int64_t)blockIdx.x / C;
  const int64_t R_T = A.total + A.B;
  const bool is_target = row_id < R_T;

  __shared__ RowSmem sm;
  __shared__ int s_b;

  // ---- which session / position this row belongs to ------------------------------
  if (tid < 32) {
    int32_t b = find_session(A.m_offsets, A.B, is_target ? row_id : row_id - R_T, is_target);
    if (tid == 0) s_b = b;
  }
  __syncthreads();
  const int32_t b = s_b;
  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const int64_t M = off1 - off0;
  const int64_t pos = is_target ? row_id - off0 - b : (row_id - R_T) - off0;
  // draft token carried by the row: target row i < M and draft row i carry x[i]
  const int64_t tok_idx = is_target ? row_id - b : row_id - R_T;
  const bool has_x = (pos >= 0 && pos < M && tok_idx >= 0 && tok_idx < A.total);

  const bool params_ok = (P.top_p_milli <= 1000u);
  const bool session_ok = params_ok && (P.rule_id == 1u || P.rule_id == 2u) && M >= 1 &&
                          M <= SDCP_MAX_M && off0 >= 0 && off1 <= A.total;
  bool skip;
  bool want_argmax, want_profile;
  if (A.stats_mode) {
    skip = !params_ok;
    want_argmax = true;
    want_profile = true;
  } else {
    const bool rule2 = (P.rule_id == 2u);
    skip = !session_ok || (!is_target && !rule2) || (!is_target && A.draft == nullptr);
    want_argmax = !rule2 || P.temperature_milli == 0u;
    want_profile = rule2 && P.temperature_milli != 0u;
  }
  RowStat* out = A.stats + row_id;
  if (skip) {
    if (rank == 0 && tid == 0) {
      RowStat r{};
      r.flags = SDCP_ROW_SKIPPED;
      *out = r;
      if (A.pub) {
        sdcp_row_stat q{};
        q.flags = SDCP_ROW_SKIPPED;
        q.lp_x = __int_as_float(0x7FC00000);
        A.pub[row_id] = q;
      }
    }
    return;  // uniform over the cluster: no cluster barrier is pending
  }

  const int64_t V = A.V;
  const T* base = reinterpret_cast<const T*>(is_target ? A.target : A.draft);
  const T* row = base + (is_target ? row_id : row_id - R_T) * V;
  const RowLayout L = row_layout(row, V);
  const int64_t vec_lo = L.nvec * rank / C, vec_hi = L.nvec * (rank + 1) / C;
  const bool do_head = (rank == 0), do_tail = (rank == C - 1);

  const uint32_t tm = P.temperature_milli;
  const bool one_hot = (tm == 0u);
  const double scale_d = one_hot ? 0.0 : 1000.0 / (double)tm;
  const float c = (float)(scale_d * 1.4426950408889634);  // log2(e) * 1000/T
  const bool topk = !one_hot && want_profile && P.top_k != 0u && (int64_t)P.top_k < V;
  const bool topp = !one_hot && want_profile && P.top_p_milli < 1000u;
  const bool filters = topk || topp;
  const bool need_keys = want_argmax || one_hot;
  const bool need_sum = want_profile && !one_hot && !topk;
  const bool need_max = want_profile && !one_hot;

  // ---- pass A: one streaming read of the slice ------------------------------------
  ThreadAcc acc;
  acc.fm = -INFINITY; acc.s = 0.f; acc.kmax = 0u; acc.kmin = 0xFFFFFFFFu; acc.amax = LLONG_MAX; acc.bad = 0;
  if (need_keys && need_sum)
    stream_slice<T, true, 2>(row, L, vec_lo, vec_hi, do_head, do_tail, V, c, acc);
  else if (need_keys && need_max)
    stream_slice<T, true, 1>(row, L, vec_lo, vec_hi, do_head, do_tail, V, c, acc);
  else if (need_keys)
    stream_slice<T, true, 0>(row, L, vec_lo, vec_hi, do_head, do_tail, V, c, acc);
  else if (need_sum)
    stream_slice<T, false, 2>(row, L, vec_lo, vec_hi, do_head, do_tail, V, c, acc);
  else
    stream_slice<T, false, 1>(row, L, vec_lo, vec_hi, do_head, do_tail, V, c, acc);

  // ---- block merge (fixed order) ----------------------------------------------------
  {
    float bfm = warp_reduce(acc.fm, [](float x, float y) { return fmax_nan(x, y); });
    const int w = tid >> 5, l = tid & 31;
    if (l == 0) sm.fscr[w] = bfm;
    __syncthreads();
    bfm = sm.fscr[0];
    for (int i = 1; i < kWarps; ++i) bfm = fmax_nan(bfm, sm.fscr[i]);
    float mine = (acc.s == 0.f || acc.fm == -INFINITY) ? 0.f : acc.s * ex2((acc.fm - bfm) * c);
    if (need_sum) mine = block_sum(mine, sm.fscr); else mine = 0.f;
    uint32_t kmx = warp_max_u32(acc.kmax), kmn = warp_min_u32(acc.kmin);
    __syncthreads();
    if (l == 0) { sm.lscr[w] = kmx; sm.lscr[kWarps + w] = kmn; }
    __syncthreads();
    kmx = 0; kmn = 0xFFFFFFFFu;
    for (int i = 0; i < kWarps; ++i) { kmx = max(kmx, (uint32_t)sm.lscr[i]); kmn = min(kmn, (uint32_t)sm.lscr[kWarps + i]); }
    long long am = (acc.kmax == kmx) ? acc.amax : LLONG_MAX;
    am = block_min_i64(am, sm.lscr);
    int bad = __syncthreads_or(acc.bad);
    if (tid == 0) {
      sm.part.fm = bfm; sm.part.s = mine; sm.part.kmax = kmx; sm.part.kmin = kmn;
      sm.part.amax = am; sm.part.bad = bad;
    }
  }
  cluster.sync();  // S1: partials visible

  // ---- cluster merge in rank order (identical in every CTA) ------------------------
  float lmax = -INFINITY, s_all = 0.f;
  uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
  long long amax = LLONG_MAX;
  int bad = 0;
  {
    Partial pr[kMaxCluster];
    for (unsigned r = 0; r < C; ++r) pr[r] = *cluster.map_shared_rank(&sm.part, r);
    for (unsigned r = 0; r < C; ++r) { lmax = fmax_nan(lmax, pr[r].fm); kmax = max(kmax, pr[r].kmax); kmin = min(kmin, pr[r].kmin); bad |= pr[r].bad; }
    for (unsigned r = 0; r < C; ++r) {
      if (pr[r].kmax == kmax) amax = min(amax, pr[r].amax);
      if (need_sum && pr[r].s != 0.f && pr[r].fm != -INFINITY) s_all += pr[r].s * ex2((pr[r].fm - lmax) * c);
    }
  }
  if (need_keys) {
    if (kmax >= kKeyPosInf || kmin < kKeyNegInf || kmax <= kKeyNegInf) bad = 1;
    if (!need_max) lmax = key_value(kmax);
  }
  if (need_max) {
    if (lmax != lmax || lmax == INFINITY || lmax == -INFINITY) bad = 1;
    if (need_sum && !(s_all < INFINITY)) bad = 1;  // NaN or overflow through the sum
  }
  const uint32_t kmax_f = need_keys ? kmax : order_key(__float_as_uint(lmax));

  // ---- filters: window histogram (bf16), else generic fallback ----------------------
  int use_fallback = 0;
  int kept = 0;
  float s_kept = 1.f;
  uint32_t thr_key = 0u;
  long long thr_id = LLONG_MAX;
  bool need_final_fallback = false;
  Decision dec{};
  const bool do_filters = filters && !bad;
  if (do_filters) {
    const bool is_bf16 = (sizeof(T) == 2);
    const uint32_t kmax16 = kmax_f >> 16;
    int nb = kWindowBins;
    if (is_bf16) {
      if ((int64_t)nb > (int64_t)kmax16 - (int64_t)(kKeyNegInf >> 16) + 1)
        nb = (int)((int64_t)kmax16 - (int64_t)(kKeyNegInf >> 16) + 1);
      if (topp && !topk && s_all > 0.f) {
        // Tokens more than R below the max (z units) hold < 1% of the (1-P) mass left
        // outside the nucleus, so the crossing lies above them.
        double R = log((double)V / (0.01 * (1.0 - P.top_p_milli / 1000.0) * (double)s_all));
        double lo = (double)lmax - R / scale_d;
        if (lo > -3.0e38 && lo < (double)lmax) {
          uint32_t klo16 = order_key(__float_as_uint((float)lo)) >> 16;
          klo16 = klo16 > 0 ? klo16 - 1 : 0;
          if (klo16 < kmax16 && (int64_t)(kmax16 - klo16 + 1) < nb) nb = (int)(kmax16 - klo16 + 1);
        }
      }
      for (int i = tid; i < kWindowBins; i += kThreads) sm.hist[i] = 0u;
      __syncthreads();
      visit_slice<T>(row, L, vec_lo, vec_hi, do_head, do_tail, V, [&](uint32_t bits, long long) {
        uint32_t d = kmax16 - (order_key(bits) >> 16);
        if (d < (uint32_t)nb) atomicAdd(&sm.hist[d], 1u);
      });
      __syncthreads();
    }
    cluster.sync();  // S2: histograms visible
    if (rank == 0) {
      if (tid == 0) { sm.dec = Decision{}; sm.dec.use_fallback = is_bf16 ? 0 : 1; }
      __syncthreads();
      if (is_bf16) {
        // sum the cluster's histograms into rank 0's (rank order; integer: exact)
        for (unsigned r = 1; r < C; ++r) {
          const uint32_t* rh = cluster.map_shared_rank(sm.hist, r);
          for (int i = tid; i < nb; i += kThreads) sm.hist[i] += rh[i];
        }
        __syncthreads();
        // thread t owns bins [8t, 8t+8), in descending value order
        constexpr int BPT = kWindowBins / kThreads;
        long long cnt_t = 0;
        float e1[BPT];
        uint32_t cn[BPT];
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
          int d = tid * BPT + i;
          cn[i] = (d < nb) ? sm.hist[d] : 0u;
          float v = key_value((kmax16 - (uint32_t)min(d, nb - 1)) << 16);
          e1[i] = (d < nb) ? ex2((v - lmax) * c) : 0.f;
          cnt_t += cn[i];
        }
        long long cnt_tot;
        long long cnt_ex = block_exclusive_scan_ll(cnt_t, sm.lscr, &cnt_tot);
        // top-k: the bin of the k-th token and how many of its tokens are kept
        int dk = INT_MAX, tk = 0;
        if (topk) {
          const long long k = P.top_k;
          if (tid == 0) { sm.b_dk = -1; sm.b_tk = 0; }
          __syncthreads();
          if (cnt_ex < k && k <= cnt_ex + cnt_t) {
            long long cc = cnt_ex;
            for (int i = 0; i < BPT; ++i) {
              if (cc + cn[i] >= k) { sm.b_dk = tid * BPT + i; sm.b_tk = (int)(k - cc); break; }
              cc += cn[i];
            }
          }
          __syncthreads();
          dk = sm.b_dk; tk = sm.b_tk;
        }
        if (topk && dk < 0) {
          if (tid == 0) sm.dec.use_fallback = 1;  // fewer than k tokens in the window
        } else {
          // masses of the kept top-k bins (bins past dk hold nothing, bin dk holds tk)
          float m_t = 0.f;
          float mb[BPT];
#pragma unroll
          for (int i = 0; i < BPT; ++i) {
            int d = tid * BPT + i;
            float m = 0.f;
            if (!topk || d < dk) m = (float)cn[i] * e1[i];
            else if (d == dk) m = (float)tk * e1[i];
            mb[i] = m;
            m_t += m;
          }
          float m_tot;
          float m_ex = block_exclusive_scan(m_t, sm.fscr, &m_tot);
          const float s_base = topk ? m_tot : s_all;
          int my_d = INT_MAX, my_n = 0;
          float my_before = 0.f;
          long long my_cbefore = 0;
          if (topp) {
            // the first bin whose cumulative mass reaches P * S, and how many of its
            // (equal-mass) tokens are needed
            const float target = (float)((double)P.top_p_milli / 1000.0 * (double)s_base);
            float cum = m_ex;
            long long cc = cnt_ex;
            for (int i = 0; i < BPT; ++i) {
              int d = tid * BPT + i;
              if (topk && d > dk) break;
              float nxt = cum + mb[i];
              if (mb[i] > 0.f && nxt >= target) {
                long long avail = (topk && d == dk) ? tk : (long long)cn[i];
                double need = ceil(((double)target - (double)cum) / (double)e1[i]);
                long long n = (long long)need;
                if (n < 1) n = 1;
                if (n > avail) n = avail;
                my_d = d; my_n = (int)n; my_before = cum; my_cbefore = cc;
                break;
              }
              cum = nxt;
              cc += cn[i];
            }
          }
          int best = topp ? (int)block_min_i64(my_d, sm.lscr) : INT_MAX;
          if (tid == 0) sm.b_found = 0;
          __syncthreads();
          if (best != INT_MAX && my_d == best) {
            sm.b_dp = best; sm.b_np = my_n; sm.b_massbefore_p = my_before;
            sm.b_countbefore_p = (int)my_cbefore; sm.b_found = 1;
          }
          __syncthreads();
          if (tid == 0) {
            Decision d0{};
            if (topp && sm.b_found) {
              const int dcut = sm.b_dp, ncut = sm.b_np;
              const float e1c = ex2((key_value((kmax16 - (uint32_t)dcut) << 16) - lmax) * c);
              d0.s_kept = sm.b_massbefore_p + (float)ncut * e1c;
              d0.kept = sm.b_countbefore_p + ncut;
              d0.thr_key = (kmax16 - (uint32_t)dcut) << 16;
              d0.need_tie = (ncut < (int)sm.hist[dcut]) ? 1 : 0;
              d0.tie_key16 = kmax16 - (uint32_t)dcut;
              d0.tie_n = ncut;
            } else if (topk) {
              // top-k alone, or a nucleus that covers the whole top-k set
              d0.s_kept = m_tot;
              d0.kept = (int)P.top_k;
              d0.thr_key = (kmax16 - (uint32_t)dk) << 16;
              d0.need_tie = (tk < (int)sm.hist[dk]) ? 1 : 0;
              d0.tie_key16 = kmax16 - (uint32_t)dk;
              d0.tie_n = tk;
            } else {
              d0.use_fallback = 1;  // the nucleus reaches below the window
            }
            sm.dec = d0;
          }
        }
      }
    }
    cluster.sync();  // S3: decision visible
    dec = *cluster.map_shared_rank(&sm.dec, 0);
    if (!dec.use_fallback && dec.need_tie) {
      // tie pass: ids with the cut value in this CTA's slice
      if (tid == 0) sm.tie_count = 0;
      __syncthreads();
      const uint32_t tk16 = dec.tie_key16;
      visit_slice<T>(row, L, vec_lo, vec_hi, do_head, do_tail, V, [&](uint32_t bits, long long id) {
        if ((order_key(bits) >> 16) == tk16) {
          int slot = atomicAdd(&sm.tie_count, 1);
          if (slot < kTieListCap) sm.tie_ids[slot] = (int)id;
        }
      });
      __syncthreads();
      cluster.sync();  // S4: tie lists visible
      if (rank == 0) {
        // find the CTA (id order = rank order) holding the n-th tied id
        int before = 0, owner = -1, overflow = 0, cnt_owner = 0;
        for (unsigned r = 0; r < C; ++r) {
          int cr = *cluster.map_shared_rank(&sm.tie_count, r);
          if (owner < 0 && before + cr >= dec.tie_n) { owner = (int)r; cnt_owner = cr; }
          else if (owner < 0) before += cr;
        }
        if (owner < 0 || cnt_owner > kTieListCap) overflow = 1;
        if (tid == 0) sm.b_tie_id = -1;
        __syncthreads();
        if (!overflow) {
          const int* ids = cluster.map_shared_rank(sm.tie_ids, (unsigned)owner);
          const int want = dec.tie_n - before;  // 1-based within the owner's list
          for (int i = tid; i < cnt_owner; i += kThreads) {
            int my = ids[i], rnk = 0;
            for (int j = 0; j < cnt_owner; ++j) rnk += (ids[j] < my) ? 1 : 0;
            if (rnk == want - 1) sm.b_tie_id = my;
          }
        }
        __syncthreads();
        thr_id = (sm.b_tie_id >= 0) ? (long long)sm.b_tie_id : LLONG_MAX;
        if (overflow || sm.b_tie_id < 0) need_final_fallback = true;  // generic id search
      }
    }
    if (!dec.use_fallback) {
      thr_key = dec.thr_key;
      kept = dec.kept;
      s_kept = dec.s_kept;
      if (!dec.need_tie) thr_id = LLONG_MAX;
    } else {
      use_fallback = 1;
    }
  }
  cluster.sync();  // final: no CTA reads another's shared memory after this
  if (rank != 0) return;

  // ---- rank 0 alone from here ---------------------------------------------------------
  WholeRow<T> R{row, L, V};
  uint32_t flags = 0;
  if (bad) flags |= SDCP_ROW_INVALID;

  if (!bad && do_filters && need_final_fallback && !use_fallback) {
    // tie list overflowed: find the tie_n-th id with the cut value over the whole row
    const uint32_t tk16 = dec.tie_key16;
    thr_id = nth_matching_id<T>(R, dec.tie_n, [&](uint32_t bits, long long) {
      return (order_key(bits) >> 16) == tk16;
    }, sm.lscr);
  }
  if (!bad && do_filters && use_fallback) {
    flags |= SDCP_ROW_FALLBACK;
    // Generic search: bisection over the order-key space with block-wide reductions.
    auto count_ge = [&](uint32_t kk) -> long long {
      long long cnt = 0;
      R.visit([&](uint32_t bits, long long) { cnt += (order_key(bits) >= kk) ? 1 : 0; });
      return block_sum_ll(cnt, sm.lscr);
    };
    uint32_t kk1 = 0u;
    long long id1 = LLONG_MAX, k1count = V;
    if (topk) {
      const long long k = P.top_k;
      uint32_t lo = 0u, hi = kmax_f;  // count_ge(lo) >= k, answer in [lo, hi]
      while (lo < hi) {
        uint32_t mid = lo + (uint32_t)(((uint64_t)hi - lo + 1) / 2);
        if (count_ge(mid) >= k) lo = mid; else hi = mid - 1;
      }
      kk1 = lo;
      long long above = (kk1 == 0xFFFFFFFFu) ? 0 : count_ge(kk1 + 1);
      long long eq = count_ge(kk1) - above;
      long long t = k - above;
      id1 = (t < eq) ? nth_matching_id<T>(R, t, [&](uint32_t bits, long long) { return order_key(bits) == kk1; }, sm.lscr)
                     : LLONG_MAX;
      k1count = k;
    }
    auto in_k1 = [&](uint32_t key, long long id) { return key > kk1 || (key == kk1 && id <= id1); };
    auto mass_ge = [&](uint32_t kk) -> float {
      float m = 0.f;
      R.visit([&](uint32_t bits, long long id) {
        uint32_t key = order_key(bits);
        if (key >= kk && in_k1(key, id)) m += ex2((__uint_as_float(bits) - lmax) * c);
      });
      return block_sum(m, sm.fscr);
    };
    uint32_t kcut = kk1;
    long long idcut = id1, keptc = k1count;
    float s1 = mass_ge(0u);
    float skept = s1;
    if (topp) {
      const float target = (float)((double)P.top_p_milli / 1000.0 * (double)s1);
      uint32_t lo = 0u, hi = kmax_f;  // mass_ge(lo) >= target (s1 >= target)
      while (lo < hi) {
        uint32_t mid = lo + (uint32_t)(((uint64_t)hi - lo + 1) / 2);
        if (mass_ge(mid) >= target) lo = mid; else hi = mid - 1;
      }
      const uint32_t kp = lo;
      const float above = (kp == 0xFFFFFFFFu) ? 0.f : mass_ge(kp + 1);
      long long cnt_above = 0, avail = 0;
      {
        long long ca = 0, av = 0;
        R.visit([&](uint32_t bits, long long id) {
          uint32_t key = order_key(bits);
          if (in_k1(key, id)) { ca += (key > kp) ? 1 : 0; av += (key == kp) ? 1 : 0; }
        });
        cnt_above = block_sum_ll(ca, sm.lscr);
        avail = block_sum_ll(av, sm.lscr);
      }
      const float e1 = ex2((key_value(kp) - lmax) * c);
      long long n = (long long)ceil(((double)target - (double)above) / (double)e1);
      if (n < 1) n = 1;
      if (n > avail) n = avail;
      kcut = kp;
      keptc = cnt_above + n;
      skept = above + (float)n * e1;
      idcut = (n < avail) ? nth_matching_id<T>(R, n, [&](uint32_t bits, long long id) {
                              uint32_t key = order_key(bits);
                              return key == kp && in_k1(key, id);
                            }, sm.lscr)
                          : (kp == kk1 ? id1 : LLONG_MAX);
    } else {
      skept = s1;
    }
    thr_key = kcut;
    thr_id = idcut;
    kept = (int)keptc;
    s_kept = skept;
  }

  if (tid != 0) return;
  RowStat st;
  st.lmax = lmax;
  st.argmax = (amax == LLONG_MAX) ? -1 : (int32_t)amax;
  if (one_hot) {
    st.s = 1.f;
    st.thr_key = kmax;
    st.thr_id = st.argmax;
    st.kept = 1;
  } else if (do_filters) {
    st.s = s_kept;
    st.thr_key = thr_key;
    st.thr_id = (thr_id == LLONG_MAX) ? INT_MAX : (int32_t)thr_id;
    st.kept = kept;
  } else {
    st.s = s_all;
    st.thr_key = 0u;
    st.thr_id = INT_MAX;
    st.kept = (int32_t)V;
  }
  st.dlx = __int_as_float(0x7FC00000);
  if (has_x && !bad) {
    const int32_t x = A.tokens[tok_idx];
    if (x >= 0 && (int64_t)x < V) {
      flags |= kRowHasX;
      const uint32_t xb = load_bits(row, x);
      const float lx = __uint_as_float(xb);
      const uint32_t xk = order_key(xb);
      const bool kept_x = one_hot ? (x == st.argmax)
                                  : (xk > st.thr_key || (xk == st.thr_key && x <= st.thr_id));
      st.dlx = lx - lmax;
      if (kept_x && lx != -INFINITY) flags |= SDCP_ROW_X_KEPT;
    }
  }
  st.flags = flags;
  *out = st;
  if (A.pub) {
    sdcp_row_stat q;
    q.lmax = st.lmax;
    q.log_s = bad ? __int_as_float(0x7FC00000) : (float)log((double)st.s);
    q.argmax = st.argmax;
    q.kept = st.kept;
    q.thr_key = st.thr_key;
    q.thr_id = st.thr_id;
    q.flags = flags & ~kRowHasX;
    if (!(flags & kRowHasX)) q.lp_x = __int_as_float(0x7FC00000);
    else if (!(flags & SDCP_ROW_X_KEPT)) q.lp_x = -INFINITY;
    else if (one_hot) q.lp_x = 0.f;
    else q.lp_x = (float)((double)st.dlx * scale_d - log((double)st.s));
    A.pub[row_id] = q;
  }
}

template __global__ void row_stats_kernel<float>(RowArgs);
template __global__ void row_stats_kernel<__nv_bfloat16>(RowArgs);

// Host-side launcher.
int launch_row_stats(const RowArgs& a, int dtype, int cluster, cudaStream_t stream) {
  int64_t rows = a.total + a.B + a.total;
  if (rows <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (dtype == SDCP_BF16)
    e = cudaLaunchKernelEx(&cfg, row_stats_kernel<__nv_bfloat16>, a);
  else
    e = cudaLaunchKernelEx(&cfg, row_stats_kernel<float>, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp
