// sdcp_sessions.cu - phase 2 of the acceptance step: per session, the precondition,
// the acceptance tests, the first rejection, and the additional token (SDCP draft
// draft-li-mlc-inference-acceleration-00, Section 6.3 "Preconditions of the rule" and
// Section 6.4 Rules 1 and 2; verdict fields of Section 5.2).
//
// One thread-block cluster per session.  Every CTA of the cluster evaluates the M
// acceptance tests from the row statistics (one lane per position, fp64 ratio, Philox
// uniform of purpose 0) and takes the first rejection a with a ballot; the cluster's rank
// 0 writes the verdict.  Rule 2 then needs one draw: from the residual max(0, p_a - q_a)
// when a < M, from p_M otherwise (purpose 1).  The cluster splits the row (pair) into
// tiles; each CTA sums the weights of its tiles with fixed-order block scans, the slice
// totals are exchanged through distributed shared memory, and the CTA whose slice holds
// u * W re-scans one tile to find the smallest id whose cumulative weight exceeds u * W.
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
  float fscr[3 * kWarps + 4];
  long long lscr[3 * kWarps + 4];
  int found_tile;
};

// Weight of token j for the draw: p_j (bonus, or residual fallen back to p) or
// max(0, p_j - q_j) (residual).  p_j = exp((l_j - lmax) * 1000/T) / S over the kept set.
struct DrawRow {
  float lmax, cexp, inv_s;
  uint32_t thr_key;
  long long thr_id;
};
__device__ __forceinline__ float prob_of(const DrawRow& r, uint32_t bits, long long j) {
  uint32_t k = order_key(bits);
  bool kept = k > r.thr_key || (k == r.thr_key && j <= r.thr_id);
  return kept ? ex2((__uint_as_float(bits) - r.lmax) * r.cexp) * r.inv_s : 0.f;
}

template <typename T>
__device__ __forceinline__ void load8(const T* row, bool aligned16, int64_t V, int64_t j0,
                                      uint32_t (&b)[kEpt]) {
  if (aligned16 && j0 + kEpt <= V) {
    if (sizeof(T) == 2) {
      uint4 q = __ldg(reinterpret_cast<const uint4*>(row + j0));
      uint32_t t[8];
      Elem<__nv_bfloat16>::unpack(q, t);
#pragma unroll
      for (int e = 0; e < kEpt; ++e) b[e] = t[e];
    } else {
      uint4 q0 = __ldg(reinterpret_cast<const uint4*>(row + j0));
      uint4 q1 = __ldg(reinterpret_cast<const uint4*>(row + j0 + 4));
      b[0] = q0.x; b[1] = q0.y; b[2] = q0.z; b[3] = q0.w;
      b[4] = q1.x; b[5] = q1.y; b[6] = q1.z; b[7] = q1.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kEpt; ++e) b[e] = (j0 + e < V) ? load_bits(row, j0 + e) : 0xFF800000u;
  }
}

// Weights of the kEpt tokens of this thread in tile `tile`.
template <typename T>
__device__ __forceinline__ void tile_weights(const T* prow, const T* qrow, bool residual,
                                             const DrawRow& pr, const DrawRow& qr, bool al_p,
                                             bool al_q, int64_t V, int64_t tile, float (&w)[kEpt]) {
  const int64_t j0 = tile * (int64_t)(kThreads * kEpt) + (int64_t)threadIdx.x * kEpt;
  uint32_t bp[kEpt];
  load8<T>(prow, al_p, V, j0, bp);
  if (residual) {
    uint32_t bq[kEpt];
    load8<T>(qrow, al_q, V, j0, bq);
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
      float p = (j0 + e < V) ? prob_of(pr, bp[e], j0 + e) : 0.f;
      float q = (j0 + e < V) ? prob_of(qr, bq[e], j0 + e) : 0.f;
      w[e] = fmaxf(p - q, 0.f);
    }
  } else {
#pragma unroll
    for (int e = 0; e < kEpt; ++e) w[e] = (j0 + e < V) ? prob_of(pr, bp[e], j0 + e) : 0.f;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) session_kernel(SessArgs A) {
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned C = cluster.num_blocks();
  const unsigned rank = cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31;
  const int32_t b = (int32_t)(blockIdx.x / C);
  __shared__ SessSmem sm;
  extern __shared__ float tile_incl[];  // inclusive prefix of this CTA's tile totals

  const sdcp_session_params P = A.params[b];
  const int64_t off0 = A.m_offsets[b], off1 = A.m_offsets[b + 1];
  const bool offsets_ok = off0 >= 0 && off1 >= off0 && off1 <= A.total &&
                          A.m_offsets[0] == 0 && (int64_t)A.m_offsets[A.B] == A.total;
  const int64_t M = off1 - off0;
  const int64_t R_T = A.total + A.B;
  const int64_t V = A.V;
  const bool rule2 = (P.rule_id == 2u);
  const uint32_t tm = P.temperature_milli;

  // ---- status and the acceptance scan (warp 0; identical in every CTA) -------------
  if (tid < 32) {
    int st = SDCP_S_OK;
    if ((P.rule_id != 1u && P.rule_id != 2u) || P.top_p_milli > 1000u) st = SDCP_S_BAD_PARAMS;
    else if (!offsets_ok) st = SDCP_S_BAD_PARAMS;
    else if (M < 1 || M > SDCP_MAX_M) st = SDCP_S_LIMIT;
    else if (rule2 && A.draft == nullptr) st = SDCP_S_Q_UNAVAILABLE;
    int a = 0;
    if (st == SDCP_S_OK) {
      bool range_bad = false, row_bad = false, q_zero = false;
      bool rej[2] = {false, false};
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < M) {
          const int32_t x = A.tokens[off0 + i];
          sm.x[i] = x;
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
              double lp = (sp.flags & SDCP_ROW_X_KEPT)
                              ? (double)sp.dlx * scale - log((double)sp.s) : -INFINITY;
              double lq = (double)sq.dlx * scale - log((double)sq.s);
              double ratio = (lp == -INFINITY) ? 0.0 : exp(lp - lq);
              ratio = ratio > 1.0 ? 1.0 : ratio;
              double u = verifier_uniform(P, (uint32_t)i, 0u);
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
      unsigned r0 = __ballot_sync(0xFFFFFFFFu, rej[0]);
      unsigned r1 = __ballot_sync(0xFFFFFFFFu, rej[1]);
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
            if (need_draw) continue;  // written once, by the CTA that finds the draw
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
  const DrawRow pr{sp.lmax, cexp, 1.f / sp.s, sp.thr_key, (long long)sp.thr_id};
  const DrawRow qr{sq.lmax, cexp, 1.f / sq.s, sq.thr_key, (long long)sq.thr_id};
  const bool al_p = ((uintptr_t)trow & 15u) == 0, al_q = ((uintptr_t)drow & 15u) == 0;
  const int64_t tile_elems = (int64_t)kThreads * kEpt;
  const int64_t nt = (V + tile_elems - 1) / tile_elems;
  const int64_t t0 = nt * rank / C, t1 = nt * (rank + 1) / C;
  const double u1 = verifier_uniform(P, (uint32_t)a, 1u);

  bool residual = (a < M);
  for (int attempt = 0; attempt < 2; ++attempt) {
    // pass 1: tile totals of this slice
    long long lastpos = -1;
    for (int64_t t = t0; t < t1; ++t) {
      float w[kEpt];
      tile_weights<T>(trow, drow, residual, pr, qr, al_p, al_q, V, t, w);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < kEpt; ++e) {
        s += w[e];
        if (w[e] > 0.f) lastpos = t * tile_elems + (int64_t)tid * kEpt + e;
      }
      float tot;
      (void)block_exclusive_scan(s, sm.fscr, &tot);
      if (tid == 0) tile_incl[t - t0] = tot;
    }
    lastpos = block_max_i64(lastpos, sm.lscr);
    __syncthreads();
    // inclusive prefix over this slice's tiles (sequential per thread, scanned across)
    {
      const int64_t n = t1 - t0;
      const int64_t per = (n + kThreads - 1) / kThreads;
      const int64_t i0 = (int64_t)tid * per, i1 = min(n, i0 + per);
      float s = 0.f;
      for (int64_t i = i0; i < i1; ++i) s += tile_incl[i];
      float tot;
      float ex = block_exclusive_scan(s, sm.fscr, &tot);
      float c = ex;
      for (int64_t i = i0; i < i1; ++i) { c += tile_incl[i]; tile_incl[i] = c; }
      if (tid == 0) { sm.slice.total = (n > 0) ? tot : 0.f; sm.slice.lastpos = lastpos; }
      __syncthreads();
      if (n > 0 && tid == 0) tile_incl[n - 1] = tot;  // slice total == last prefix, exactly
    }
    __syncthreads();
    cluster.sync();
    // slice totals in rank order: W, this slice's base, global last positive id
    float W = 0.f, base = 0.f;
    long long glast = -1;
    int owner = -1;
    for (unsigned r = 0; r < C; ++r) {
      SliceInfo si = *cluster.map_shared_rank(&sm.slice, r);
      if (r == rank) base = W;
      W += si.total;
      glast = max(glast, si.lastpos);
    }
    const bool retry = !(W > 0.f) && residual;  // residual mass lost to rounding: use p
    float target = 0.f;
    if (!retry && W > 0.f) {
      target = (float)(u1 * (double)W);
      float acc = 0.f;
      for (unsigned r = 0; r < C; ++r) {
        SliceInfo si = *cluster.map_shared_rank(&sm.slice, r);
        float nxt = acc + si.total;
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
    // the owner: first tile whose inclusive prefix exceeds the target
    const int64_t n = t1 - t0;
    if (tid == 0) sm.found_tile = INT_MAX;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kThreads)
      if (base + tile_incl[i] > target) atomicMin(&sm.found_tile, (int)i);
    __syncthreads();
    const int ti = (sm.found_tile == INT_MAX) ? (int)(n > 0 ? n - 1 : 0) : sm.found_tile;
    const float pre = base + (ti > 0 ? tile_incl[ti - 1] : 0.f);
    float w[kEpt];
    tile_weights<T>(trow, drow, residual, pr, qr, al_p, al_q, V, t0 + ti, w);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < kEpt; ++e) s += w[e];
    float tot;
    float ex = block_exclusive_scan(s, sm.fscr, &tot);
    long long found = LLONG_MAX, lastp = -1;
    float cc = pre + ex;
    const int64_t j0 = (t0 + ti) * tile_elems + (int64_t)tid * kEpt;
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
      cc += w[e];
      if (w[e] > 0.f) {
        lastp = j0 + e;
        if (found == LLONG_MAX && cc > target) found = j0 + e;
      }
    }
    found = block_min_i64(found, sm.lscr);
    lastp = block_max_i64(lastp, sm.lscr);
    if (tid == 0) A.out_tokens[off0 + b + a] = (int32_t)(found != LLONG_MAX ? found : lastp);
    break;
  }
}

template __global__ void session_kernel<float>(SessArgs);
template __global__ void session_kernel<__nv_bfloat16>(SessArgs);

int launch_sessions(const SessArgs& a, int dtype, int cluster, cudaStream_t stream) {
  if (a.B <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.B * cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)a.max_tiles_per_cta * sizeof(float);
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
    e = cudaLaunchKernelEx(&cfg, session_kernel<__nv_bfloat16>, a);
  else
    e = cudaLaunchKernelEx(&cfg, session_kernel<float>, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp
