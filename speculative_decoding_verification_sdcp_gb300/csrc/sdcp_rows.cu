// sdcp_rows.cu - phase 1 of the acceptance step: per-row statistics of the sampling
// profile (SDCP draft draft-li-mlc-inference-acceleration-00, Section 4.1: temperature,
// then top-k, then top-p; temperature 0 selects the argmax, ties to the smallest id).
//
// A persistent kernel, two CTAs per SM.  In each CTA one producer warp claims rows from a
// grid-wide counter (so CTAs that meet slow rows take fewer) and streams each row from HBM
// into a ring of three 32 KB shared-memory stages with bulk copies (TMA) that complete on
// mbarriers; eight consumer warps reduce each stage as it lands (eight 16-byte vectors per
// thread) and hand it back.  The HBM stream therefore does not wait for the per-row work:
// every logits byte is read from HBM once, and up to 96 KB per CTA are in flight.
//
// Per row the consumers keep, per thread, the running maximum, its smallest id when the row
// needs an argmax, and the sum of exp relative to it (online softmax) when it needs one;
// warps merge in a fixed order, so every result is independent of scheduling.
//
// Top-k / top-p on bf16 rows: all tokens that share a bf16 value have the same
// probability, so the exact count of every value in a window below the row maximum decides
// both cuts (the mass of a value is count * exp(v - max)).  The window (8 nats below the
// maximum of the row's first stage; for top-k, down to a bound on the k-th largest token
// from the first stage's thread maxima) is counted while the row streams, with a shared-memory
// histogram of up to 2048 values: the stage loop marks the vectors whose maximum reaches
// the window, each warp lists its marked vectors and counts them one vector per lane with
// full-warp reductions; one warp then scans the bins for the k-th token and the top-p
// crossing.  A cut inside one value keeps its first tokens in id order; only
// their number is recorded.  Rows the window cannot decide are searched again from L2
// (wider windows, then a bisection over the order-key space).
#include <climits>
#include <mutex>

#include "sdcp_session.cuh"

namespace sdcp {

constexpr int kConsWarps = 8;
constexpr int kCons = kConsWarps * 32;  // consumer threads
constexpr int kProducerWarp = kConsWarps;
constexpr int kRowThreads = kCons + 32;
constexpr int kStages = 3;
constexpr int kChunk = 32768;            // bytes per ring stage (8 vectors per consumer thread)
constexpr int kConsBar = 1;              // named barrier of the consumer warps
constexpr int kRowCtasPerSm = 2;
constexpr int kVecPerThread = kChunk / 16 / kCons;
static_assert(kCons == kThreads, "the consumer group runs session completions");

// What a row needs, from its session (resolved once, by the producer warp).
struct RowCtx {
  float c, inv_scale;  // log2(e) 1000/T; T/1000
  uint32_t top_k, top_p_milli, temperature_milli;
  int mode;
  bool has_x, one_hot, topk, topp, need_keys, need_sum, window;
};

struct RowPlan {
  long long row_id;  // < 0: no more work for the CTA
  int nchunks;
  int32_t xt;        // the row's draft token as the token array holds it (-1: none)
  bool skip;         // the row needs no statistics (its first stage was copied before that was
                     // known): the consumers hand the stage back and record it as skipped
  RowCtx x;
};

struct RowShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  RowPlan plan[kStages];
  volatile int abort;
  // per-warp partials (w_m0: the first stage's maxima, for the window's anchor)
  float w_fm[32], w_s[32], w_m0[32];
  long long w_amax[32];
  float fscr[2 * 32 + 4];
  long long lscr[2 * 32 + 4];
  uint32_t xbits;  // the draft token's logit bits
  // the merged row and its cut (warp 0 -> group)
  float r_lmax, r_s, r_skept;
  long long r_amax, r_thr_n;
  uint32_t r_thr_key;
  int r_kept, r_done, r_fallback;
  uint32_t hist[kWindowBins];
  uint32_t kbins[32];     // thread maxima of the first stage by depth below its maximum (top-k)
  uint32_t hist_pad[32];  // one word per lane: where a lane with nothing to count adds 0
  uint16_t hits[kConsWarps][kVecPerThread * 32];  // per warp: stage vectors that reach the window
};

// --------------------------------------------------------------------------------------
// Per-thread accumulation.  Every row keeps the running maximum fm (max.NaN, so a NaN
// poisons it); ARGMAX rows also keep the smallest id holding fm (float equality, so -0 and
// +0 tie and go to the smaller id); SUM rows keep s = sum exp((l - fm) * 1000/T), the sum
// being rescaled whenever fm grows (online softmax).  The sum is compensated (Kahan: one
// correction term sc per thread, added once per vector), so a thread's thousands of terms
// leave S with about one rounding of relative error, not one per term.
// --------------------------------------------------------------------------------------
struct ThreadAcc {
  float fm, fmc, s, sc;  // fmc = fm * c; sc: the compensation of s (s - sc is the sum)
  long long amax;
  __device__ __forceinline__ void reset() { fm = -INFINITY; fmc = -INFINITY; s = 0.f; sc = 0.f; amax = LLONG_MAX; }
  __device__ __forceinline__ void add(float t) {  // s += t, compensated
    const float y = t - sc;
    const float z = s + y;
    sc = (z - s) - y;
    s = z;
  }
  __device__ __forceinline__ void rescale(float f) { s *= f; sc *= f; }
};

template <bool ARGMAX, bool SUM>
__device__ __forceinline__ void acc_element(ThreadAcc& a, uint32_t bits, long long id, float c) {
  const float v = __uint_as_float(bits);
  const float nm = fmax_nan(a.fm, v);
  if (!(nm == a.fm)) {  // grew, or became NaN
    if (SUM) {
      if (a.fm == -INFINITY) { a.s = 0.f; a.sc = 0.f; }
      else a.rescale(ex2(a.fmc - nm * c));
    }
    if (ARGMAX) a.amax = id;
    a.fm = nm;
    a.fmc = nm * c;
  }
  if (SUM && a.fm != -INFINITY) a.add(ex2(fmaf(v, c, -a.fmc)));
}

// Maximum of one 16-byte vector, NaN-propagating (bf16: three packed bf16x2 max.NaN).
__device__ __forceinline__ float vec_max(const uint4& q, float) {
  float m0 = fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y));
  float m1 = fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w));
  return fmax_nan(m0, m1);
}
__device__ __forceinline__ float vec_max(const uint4& q, __nv_bfloat16) {
  const __nv_bfloat162 a = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&q.x),
                                       *reinterpret_cast<const __nv_bfloat162*>(&q.y));
  const __nv_bfloat162 b = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&q.z),
                                       *reinterpret_cast<const __nv_bfloat162*>(&q.w));
  const __nv_bfloat162 ab = __hmax2_nan(a, b);
  const uint32_t m = *reinterpret_cast<const uint32_t*>(&ab);
  return fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

template <typename T, bool ARGMAX, bool SUM>
__device__ __forceinline__ float acc_vector(ThreadAcc& a, const uint4& q, long long id0, float c) {
  constexpr int E = Elem<T>::kPerVec;
  uint32_t b[E];
  Elem<T>::unpack(q, b);
  float v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = __uint_as_float(b[e]);
  const float vm = vec_max(q, T());
  const float nm = fmax_nan(a.fm, vm);
  if (!(nm == a.fm)) {  // the maximum grew (or a NaN arrived): rare after the first vectors
    if (SUM) {
      if (a.fm == -INFINITY) { a.s = 0.f; a.sc = 0.f; }
      else a.rescale(ex2(a.fmc - nm * c));
    }
    if (ARGMAX) {
      int first = E - 1;
#pragma unroll
      for (int e = E - 1; e >= 0; --e) if (v[e] == nm) first = e;
      a.amax = id0 + first;
    }
    a.fm = nm;
    a.fmc = nm * c;
  }
  if (SUM && a.fm != -INFINITY) {
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) t += ex2(fmaf(v[e], c, -a.fmc));
    a.add(t);
  }
  return vm;
}

// --------------------------------------------------------------------------------------
// Window histogram.  Bin d counts the tokens whose bf16 value key is top16 - d (d < nb).
// Every element of a bf16 row with a filter updates the bin of its value under a predicate.
// Positive windows (bottom above +0): with h the bf16 bit pattern as a signed 16-bit number,
// value order is h order and d = (top16 - 0x8000) - h is in [0, nb) exactly for the
// window's values (negative values have h < 0, values above the top give d < 0).  Other
// windows go through the order key: d = top16 - key16.
// --------------------------------------------------------------------------------------
// hist[d] += 1 when d < nb, else pad[lane] += 0: every lane takes part in every reduction
// (shared-memory reductions with some lanes masked off cost about twice a full-warp one;
// the pad words are one per bank, so lanes with nothing to count add no conflicts).
__device__ __forceinline__ void hist_add_if(uint32_t hist_base, uint32_t pad_lane, uint32_t d, uint32_t nb) {
  const bool in = d < nb;
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(in ? hist_base + 4u * d : pad_lane), "r"(in ? 1u : 0u)
               : "memory");
}
template <bool POS>
__device__ __forceinline__ void win_word(uint32_t hist_base, uint32_t pad_lane, uint32_t wd, uint32_t top,
                                         uint32_t nb) {
  uint32_t d0, d1;
  if (POS) {
    d0 = top - (uint32_t)((int32_t)(wd << 16) >> 16);
    d1 = top - (uint32_t)((int32_t)wd >> 16);
  } else {
    d0 = top - (order_key(wd << 16) >> 16);
    d1 = top - (order_key(wd & 0xFFFF0000u) >> 16);
  }
  hist_add_if(hist_base, pad_lane, d0, nb);
  hist_add_if(hist_base, pad_lane, d1, nb);
}
// The row's window as the stage loop carries it.  The stage loop only marks, per thread,
// the vectors whose maximum reaches the lowest bin (one compare per vector); each warp then
// lists its marked vectors and counts them 32 at a time, one vector per lane, so the
// per-element reductions run for marked vectors only.
struct Window {
  uint32_t top, nb;  // win_word's top (positive windows: top16 - 0x8000) and bin count
  float bot;         // value of the lowest bin: every element in the window is >= bot
};
// hm: bit i marks vector threadIdx.x + i * kCons of the stage sv.
template <bool POS>
__device__ __forceinline__ void win_hits(RowShared& sh, const uint4* sv, uint32_t hm, const Window& wn) {
  const int l = threadIdx.x & 31;
  const uint32_t n = (uint32_t)__popc(hm);
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (l >= o) incl += v;
  }
  const uint32_t H = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (H == 0u) return;
  uint16_t* list = sh.hits[threadIdx.x >> 5];
  uint32_t pos = incl - n;
  while (hm != 0u) {
    const int i = __ffs(hm) - 1;
    hm &= hm - 1u;
    list[pos++] = (uint16_t)(threadIdx.x + i * kCons);
  }
  __syncwarp();
  const uint32_t hb = smem_u32(sh.hist), pl = smem_u32(sh.hist_pad + l);
  // every lane runs every round (lanes past H count a vector of -inf, which has no bin)
  const uint4 none = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  for (uint32_t e0 = 0; e0 < H; e0 += 32) {
    const uint32_t e = e0 + (uint32_t)l;
    const uint4 q = (e < H) ? sv[list[e]] : none;
    win_word<POS>(hb, pl, q.x, wn.top, wn.nb);
    win_word<POS>(hb, pl, q.y, wn.top, wn.nb);
    win_word<POS>(hb, pl, q.z, wn.top, wn.nb);
    win_word<POS>(hb, pl, q.w, wn.top, wn.nb);
  }
  __syncwarp();  // the list is free for the next stage
}

// One element (bits of a bf16 value in the upper half) of the row's unaligned ends.
__device__ __forceinline__ void win_scalar(RowShared& sh, uint32_t bits, uint32_t top16, uint32_t nb) {
  const uint32_t d = top16 - (order_key(bits) >> 16);
  if (d < nb) atomicAdd(sh.hist + d, 1u);
}

// Vectors [0, nv) of one ring stage (nv <= kVecPerThread * kCons); vector v is element
// id0 + v * E of the row and belongs to consumer thread v % kCons.  WIN: returns the mask of
// the thread's vectors whose maximum is >= bot (bit i: vector t + i * kCons).  Vectors past
// nv read as -inf, which changes no statistic and marks nothing.
template <typename T, bool ARGMAX, bool SUM, bool WIN>
__device__ __forceinline__ uint32_t acc_stage(ThreadAcc& a, const uint4* sv, int nv, long long id0, float c,
                                              float bot) {
  constexpr int E = Elem<T>::kPerVec;
  const int t = threadIdx.x;
  const uint32_t ninf = (sizeof(T) == 2) ? 0xFF80FF80u : 0xFF800000u;
  const uint4 pad = make_uint4(ninf, ninf, ninf, ninf);
  uint32_t hm = 0u;
#pragma unroll 1
  for (int i0 = 0; i0 < kVecPerThread; i0 += 4) {
    uint4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = t + (i0 + u) * kCons;
      q[u] = (v < nv) ? sv[v] : pad;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = t + (i0 + u) * kCons;
      const float vm = acc_vector<T, ARGMAX, SUM>(a, q[u], id0 + (long long)v * E, c);
      if (WIN) hm |= (vm >= bot ? 1u : 0u) << (i0 + u);
    }
  }
  return hm;
}

// The marks of a stage that was reduced before the window was placed (the first).
template <typename T>
__device__ __forceinline__ uint32_t window_marks(const uint4* sv, int nv, float bot) {
  const int t = threadIdx.x;
  uint32_t hm = 0u;
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const int v = t + i * kCons;
    if (v < nv && vec_max(sv[v], T()) >= bot) hm |= 1u << i;
  }
  return hm;
}

template <typename T, bool ARGMAX, bool SUM>
__device__ __forceinline__ void acc_scalars(ThreadAcc& a, const T* row, const RowLayout& L, int64_t V, float c) {
  for (int64_t j = threadIdx.x; j < L.head; j += kCons) acc_element<ARGMAX, SUM>(a, load_bits(row, j), j, c);
  for (int64_t j = L.tail0 + threadIdx.x; j < V; j += kCons) acc_element<ARGMAX, SUM>(a, load_bits(row, j), j, c);
}

// Row modes: which statistics a row needs.
enum RowMode { kModeMax = 0, kModeArgmax = 1, kModeSum = 2, kModeArgmaxSum = 3 };

template <typename T, bool WIN>
__device__ __forceinline__ uint32_t acc_stage_mode(int mode, ThreadAcc& a, const uint4* sv, int nv, long long id0,
                                                   float c, float bot = 0.f) {
  switch (mode) {
    case kModeMax: return acc_stage<T, false, false, WIN>(a, sv, nv, id0, c, bot);
    case kModeArgmax: return acc_stage<T, true, false, WIN>(a, sv, nv, id0, c, bot);
    case kModeSum: return acc_stage<T, false, true, WIN>(a, sv, nv, id0, c, bot);
    default: return acc_stage<T, true, true, WIN>(a, sv, nv, id0, c, bot);
  }
}
template <typename T>
__device__ __forceinline__ void acc_scalars_mode(int mode, ThreadAcc& a, const T* row, const RowLayout& L,
                                                 int64_t V, float c) {
  switch (mode) {
    case kModeMax: acc_scalars<T, false, false>(a, row, L, V, c); break;
    case kModeArgmax: acc_scalars<T, true, false>(a, row, L, V, c); break;
    case kModeSum: acc_scalars<T, false, true>(a, row, L, V, c); break;
    default: acc_scalars<T, true, true>(a, row, L, V, c); break;
  }
}

// --------------------------------------------------------------------------------------
// What a row needs, from its session.
// --------------------------------------------------------------------------------------

// Row row_id of session b; skip: the row needs no statistics; tok_idx: its draft token's
// index in the token array (when has_x).
__device__ __forceinline__ RowCtx row_ctx(const RowArgs& A, long long row_id, int b, bool bf16, bool& skip,
                                          long long& tok_idx) {
  RowCtx x;
  const long long R_T = A.io.total + A.io.B;
  const bool is_target = row_id < R_T;
  const sdcp_session_params P = A.io.params[b];
  const long long off0 = A.io.m_offsets[b], off1 = A.io.m_offsets[b + 1];
  const long long M = off1 - off0;
  const long long pos = is_target ? row_id - off0 - b : (row_id - R_T) - off0;
  tok_idx = is_target ? row_id - b : row_id - R_T;
  x.has_x = (pos >= 0 && pos < M && tok_idx >= 0 && tok_idx < A.io.total);
  const bool params_ok = (P.top_p_milli <= 1000u);
  const bool session_ok = params_ok && (P.rule_id == 1u || P.rule_id == 2u || P.rule_id == SDCP_RULE_RELAXED_TOP_K) && M >= 1 &&
                          M <= SDCP_MAX_M && off0 >= 0 && off1 <= A.io.total;
  bool want_argmax, want_profile;
  if (A.stats_mode) {
    skip = !params_ok;
    want_argmax = true;
    want_profile = true;
  } else {
    const bool rule2 = (P.rule_id == 2u);
    const bool profiled = rule2 || P.rule_id == SDCP_RULE_RELAXED_TOP_K;  // p after the profile
    // draft rows are read for Rule 2's q from logits only (q given as probability rows, or
    // no draft logits at all, leaves them unread)
    skip = !session_ok || (!is_target && (!rule2 || A.io.draft == nullptr || A.io.q_rows != nullptr));
    want_argmax = !profiled || P.temperature_milli == 0u;
    want_profile = profiled && P.temperature_milli != 0u;
  }
  const uint32_t tm = P.temperature_milli;
  x.top_k = P.top_k;
  x.top_p_milli = P.top_p_milli;
  x.temperature_milli = tm;
  x.one_hot = (tm == 0u);
  x.c = x.one_hot ? 0.f : profile_c(tm);
  x.inv_scale = profile_inv_scale(tm);
  x.topk = !x.one_hot && want_profile && P.top_k != 0u && (int64_t)P.top_k < A.io.V;
  x.topp = !x.one_hot && want_profile && P.top_p_milli < 1000u;
  x.need_keys = want_argmax || x.one_hot;  // the argmax is needed
  x.need_sum = want_profile && !x.one_hot && !x.topk;
  x.mode = x.need_keys ? (x.need_sum ? kModeArgmaxSum : kModeArgmax) : (x.need_sum ? kModeSum : kModeMax);
  x.window = (x.topk || x.topp) && bf16;
  return x;
}

template <typename T>
__device__ __forceinline__ const T* row_ptr(const RowArgs& A, long long row_id) {
  const long long R_T = A.io.total + A.io.B;
  const T* base = reinterpret_cast<const T*>(row_id < R_T ? A.io.target : A.io.draft);
  return base + (row_id < R_T ? row_id : row_id - R_T) * A.io.V;
}

__device__ __forceinline__ void write_skipped(const RowArgs& A, long long row_id) {
  RowStat r{};
  r.flags = SDCP_ROW_SKIPPED;
  A.stats[row_id] = r;
  if (A.pub) {
    sdcp_row_stat q{};
    q.flags = SDCP_ROW_SKIPPED;
    q.lp_x = __int_as_float(0x7FC00000);
    A.pub[row_id] = q;
  }
}

// --------------------------------------------------------------------------------------
// Whole-row passes by the consumer group (second reads hit L2).
// --------------------------------------------------------------------------------------
template <typename T, typename F>
__device__ __forceinline__ void visit_row(const T* __restrict__ row, const RowLayout& L, int64_t V, F f) {
  constexpr int E = Elem<T>::kPerVec;
  const int t = threadIdx.x;
  for (int64_t j = t; j < L.head; j += kCons) f(load_bits(row, j), j);
  const uint4* vp = reinterpret_cast<const uint4*>(row + L.head);
  int64_t v = t;
  for (; v + kCons < L.nvec; v += 2 * kCons) {
    const uint4 q0 = __ldg(vp + v), q1 = __ldg(vp + v + kCons);
    uint32_t b0[E], b1[E];
    Elem<T>::unpack(q0, b0);
    Elem<T>::unpack(q1, b1);
    const long long i0 = L.head + v * E, i1 = L.head + (v + kCons) * E;
#pragma unroll
    for (int e = 0; e < E; ++e) f(b0[e], i0 + e);
#pragma unroll
    for (int e = 0; e < E; ++e) f(b1[e], i1 + e);
  }
  if (v < L.nvec) {
    const uint4 q = __ldg(vp + v);
    uint32_t b[E];
    Elem<T>::unpack(q, b);
    const long long i0 = L.head + v * E;
#pragma unroll
    for (int e = 0; e < E; ++e) f(b[e], i0 + e);
  }
  for (int64_t j = L.tail0 + t; j < V; j += kCons) f(load_bits(row, j), j);
}

// Coalesced pass over a row from global memory (L2) by the consumer group, eight 16-byte
// loads in flight per thread.  f(bits[E], id of bits[0], count of valid elements).
template <typename T, typename F>
__device__ __forceinline__ void scan_row(const T* __restrict__ row, const RowLayout& L, int64_t V, F f) {
  constexpr int E = Elem<T>::kPerVec;
  constexpr int U = 4;
  const int t = threadIdx.x;
  for (int64_t j = t; j < L.head; j += kCons) {
    uint32_t b[E];
    b[0] = load_bits(row, j);
#pragma unroll
    for (int e = 1; e < E; ++e) b[e] = 0xFF800000u;
    f(b, j, 1);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(row + L.head);
  for (int64_t v0 = t; v0 < L.nvec; v0 += (int64_t)U * kCons) {
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + (int64_t)u * kCons;
      q[u] = (v < L.nvec) ? __ldg(vp + v) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + (int64_t)u * kCons;
      if (v >= L.nvec) break;
      uint32_t b[E];
      Elem<T>::unpack(q[u], b);
      f(b, L.head + v * E, E);
    }
  }
  for (int64_t j = L.tail0 + t; j < V; j += kCons) {
    uint32_t b[E];
    b[0] = load_bits(row, j);
#pragma unroll
    for (int e = 1; e < E; ++e) b[e] = 0xFF800000u;
    f(b, j, 1);
  }
}

// Id of the n-th (1-based, id order) token satisfying pred: each consumer thread owns a
// contiguous run of ids, counts, scans, and the owner walks its run again.
template <typename T, typename P>
__device__ long long nth_matching_id(const Group& g, const T* row, int64_t V, long long n, P pred,
                                     long long* lscr) {
  const int t = threadIdx.x;
  const int64_t chunk = (V + kCons - 1) / kCons;
  const int64_t j0 = (int64_t)t * chunk, j1 = min(V, j0 + chunk);
  long long cnt = 0;
  for (int64_t j = j0; j < j1; ++j) cnt += pred(load_bits(row, j), j) ? 1 : 0;
  long long tot;
  const long long ex = group_excl_scan_ll(g, cnt, lscr, &tot);
  long long found = LLONG_MAX;
  if (ex < n && n <= ex + cnt) {
    long long cc = ex;
    for (int64_t j = j0; j < j1; ++j)
      if (pred(load_bits(row, j), j) && ++cc == n) { found = j; break; }
  }
  return group_min_i64(g, found, lscr);
}

struct Thresholds {
  uint32_t thr_key;
  long long thr_n;  // kept tokens with key thr_key, first ones in id order (LLONG_MAX: all)
  int kept;
  float s_kept;
  bool fallback;
};

// Exact-value selection by one warp from hist, where bin d counts the tokens whose bf16
// value key is top16 - d (d < nb, descending values).  Lane l owns bins [l bpl, l bpl +
// bpl).  Returns false when the window cannot decide (fewer than k tokens in it, or less
// mass than the nucleus needs).  A cut inside a value keeps the first tokens of that value
// in id order; only their number is recorded (all of them have the same probability).
__device__ bool warp_select(const RowCtx& x, float lmax, float s_all, const uint32_t* hist,
                            uint32_t top16, int nb, Thresholds& out) {
  const int l = threadIdx.x & 31;
  const int bpl = (nb + 31) >> 5;
  const int d0 = min(nb, l * bpl), d1 = min(nb, d0 + bpl);
  auto e_of = [&](int d) { return ex2((key_value((top16 - (uint32_t)d) << 16) - lmax) * x.c); };
  // masses are summed with compensation (Kahan): a lane adds up to 64 bins, and the kept
  // mass S sets every probability of the row
  auto kadd = [](float& sum, float& comp, float t) {
    const float y = t - comp;
    const float z = sum + y;
    comp = (z - sum) - y;
    sum = z;
  };
  long long cnt = 0;
  float mass = 0.f, mass_c = 0.f;
  for (int d = d0; d < d1; d += 4) {  // four bins at a time (the loads and exps overlap)
    uint32_t c[4];
    float e[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      c[u] = (d + u < d1) ? hist[d + u] : 0u;
      e[u] = e_of(d + u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c[u] != 0u) { cnt += c[u]; kadd(mass, mass_c, (float)c[u] * e[u]); }
  }
  mass -= mass_c;
  // exclusive prefixes over the lanes (bins before the lane's first)
  long long ci = cnt;
  float mi = mass;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long tc = __shfl_up_sync(0xFFFFFFFFu, ci, o);
    const float tm = __shfl_up_sync(0xFFFFFFFFu, mi, o);
    if (l >= o) { ci += tc; mi += tm; }
  }
  long long cpre = __shfl_up_sync(0xFFFFFFFFu, ci, 1);
  float mpre = __shfl_up_sync(0xFFFFFFFFu, mi, 1);
  if (l == 0) { cpre = 0; mpre = 0.f; }
  int dk = nb, tk = 0;
  float s_base = s_all;  // mass of the set the nucleus is taken from
  const long long k = x.top_k;
  if (x.topk) {
    const unsigned m = __ballot_sync(0xFFFFFFFFu, cpre < k && k <= cpre + cnt);
    if (m == 0u) return false;  // fewer than k tokens in the window
    const int src = __ffs(m) - 1;
    int my_dk = 0, my_tk = 0;
    float my_s = 0.f;
    if (l == src) {
      long long cc = cpre;
      float mm = mpre, mm_c = 0.f;
      for (int d = d0; d < d1; ++d) {
        const uint32_t c = hist[d];
        if (c == 0u) continue;
        const float e = e_of(d);
        if (cc + c >= k) { my_dk = d; my_tk = (int)(k - cc); kadd(mm, mm_c, (float)my_tk * e); my_s = mm - mm_c; break; }
        cc += c;
        kadd(mm, mm_c, (float)c * e);
      }
    }
    dk = __shfl_sync(0xFFFFFFFFu, my_dk, src);
    tk = __shfl_sync(0xFFFFFFFFu, my_tk, src);
    s_base = __shfl_sync(0xFFFFFFFFu, my_s, src);
  }
  int dcut = dk, ncut = tk;
  if (x.topp) {
    const float target = (float)x.top_p_milli * 0.001f * s_base;
    int cd = -1, cn = 0;
    float cb = 0.f;
    long long ccb = 0;
    float cum = mpre, cum_c = 0.f;  // cum - cum_c: the compensated running mass
    long long cc = cpre;
    const int dend = min(d1, dk + 1);
    for (int d = d0; d < dend && cd < 0; d += 4) {  // four bins at a time, then in order
      uint32_t c4[4];
      float e4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c4[u] = (d + u < dend) ? hist[d + u] : 0u;
        e4[u] = e_of(d + u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t c = c4[u];
        if (cd >= 0 || c == 0u) continue;
        const float e = e4[u];
        const long long avail = (x.topk && d + u == dk) ? tk : (long long)c;
        const float md = (float)avail * e;
        float nxt = cum, nxt_c = cum_c;
        kadd(nxt, nxt_c, md);
        if (md > 0.f && nxt - nxt_c >= target) {
          const float base = cum - cum_c;
          long long n = (long long)ceilf(__fdiv_rn(target - base, e));
          if (n < 1) n = 1;
          if (n > avail) n = avail;
          cd = d + u; cn = (int)n; cb = base; ccb = cc;
          continue;
        }
        cum = nxt;
        cum_c = nxt_c;
        cc += c;
      }
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, cd >= 0);
    if (m != 0u) {
      const int src = __ffs(m) - 1;
      dcut = __shfl_sync(0xFFFFFFFFu, cd, src);
      ncut = __shfl_sync(0xFFFFFFFFu, cn, src);
      cb = __shfl_sync(0xFFFFFFFFu, cb, src);
      ccb = __shfl_sync(0xFFFFFFFFu, ccb, src);
      out.s_kept = cb + (float)ncut * e_of(dcut);
      out.kept = (int)(ccb + ncut);
    } else if (x.topk) {  // rounding kept the crossing out of reach: the whole top-k set
      out.s_kept = s_base;
      out.kept = (int)k;
    } else {
      return false;  // the nucleus reaches below the window
    }
  } else {
    out.s_kept = s_base;
    out.kept = (int)k;
  }
  const uint32_t ccut = hist[dcut];
  out.thr_key = (top16 - (uint32_t)dcut) << 16;
  out.thr_n = ((uint32_t)ncut >= ccut) ? LLONG_MAX : ncut;
  out.fallback = false;
  return true;
}

// Publishes a warp-0 result to the group (through sh.r_*).
__device__ __forceinline__ void put_thresholds(RowShared& sh, bool done, const Thresholds& th) {
  sh.r_done = done ? 1 : 0;
  sh.r_thr_key = th.thr_key;
  sh.r_thr_n = th.thr_n;
  sh.r_kept = th.kept;
  sh.r_skept = th.s_kept;
  sh.r_fallback = th.fallback ? 1 : 0;
}
__device__ __forceinline__ bool get_thresholds(const RowShared& sh, Thresholds& th) {
  th.thr_key = sh.r_thr_key;
  th.thr_n = sh.r_thr_n;
  th.kept = sh.r_kept;
  th.s_kept = sh.r_skept;
  th.fallback = sh.r_fallback != 0;
  return sh.r_done != 0;
}

// Window histogram of the tokens within dz nats below the row maximum (dz = 0: the 2048
// values below it), from a pass over the row in L2, then the selection (group).
template <typename T>
__device__ bool window_thresholds(const Group& g, RowShared& sh, const T* row, const RowLayout& L,
                                  const RowCtx& x, int64_t V, float lmax, float s_all, float dz,
                                  Thresholds& out) {
  const int t = threadIdx.x;
  const uint32_t kmax16 = order_key(__float_as_uint(lmax)) >> 16;
  int nb = kWindowBins;
  if ((int64_t)nb > (int64_t)kmax16 - (int64_t)(kKeyNegInf >> 16) + 1)
    nb = (int)((int64_t)kmax16 - (int64_t)(kKeyNegInf >> 16) + 1);
  if (dz > 0.f) {
    const float lo = lmax - dz * x.inv_scale;
    if (lo > -3.0e38f && lo < lmax) {
      uint32_t klo16 = order_key(__float_as_uint(lo)) >> 16;
      klo16 = klo16 > 0 ? klo16 - 1 : 0;
      if (klo16 < kmax16 && (int64_t)(kmax16 - klo16 + 1) < nb) nb = (int)(kmax16 - klo16 + 1);
    }
  }
  g.sync();  // earlier readers of the histogram are done
  for (int i = t; i < kWindowBins; i += kCons) sh.hist[i] = 0u;
  g.sync();
  const uint32_t hb = smem_u32(sh.hist), pl = smem_u32(sh.hist_pad + (t & 31));
  scan_row<T>(row, L, V, [&](const uint32_t (&b)[Elem<T>::kPerVec], long long, int n) {
#pragma unroll
    for (int e = 0; e < Elem<T>::kPerVec; ++e)
      hist_add_if(hb, pl, e < n ? kmax16 - (order_key(b[e]) >> 16) : (uint32_t)nb, (uint32_t)nb);
  });
  g.sync();
  if ((t >> 5) == 0) {
    Thresholds th = out;
    const bool done = warp_select(x, lmax, s_all, sh.hist, kmax16, nb, th);
    if ((t & 31) == 0) put_thresholds(sh, done, th);
  }
  g.sync();
  const bool done = get_thresholds(sh, out);
  return done;
}

// Generic search: bisection over the order-key space with group-wide reductions.
template <typename T>
__device__ void generic_thresholds(const Group& g, RowShared& sh, const T* row, const RowLayout& L,
                                   const RowCtx& x, int64_t V, float lmax, uint32_t kmax_f,
                                   Thresholds& out) {
  auto count_ge = [&](uint32_t kk) -> long long {
    long long cnt = 0;
    visit_row<T>(row, L, V, [&](uint32_t bits, long long) { cnt += (order_key(bits) >= kk) ? 1 : 0; });
    return group_sum_ll(g, cnt, sh.lscr);
  };
  uint32_t kk1 = 0u;
  long long id1 = LLONG_MAX, k1count = V;
  if (x.topk) {
    const long long k = x.top_k;
    uint32_t lo = 0u, hi = kmax_f;
    while (lo < hi) {
      const uint32_t mid = lo + (uint32_t)(((uint64_t)hi - lo + 1) / 2);
      if (count_ge(mid) >= k) lo = mid; else hi = mid - 1;
    }
    kk1 = lo;
    const long long above = (kk1 == 0xFFFFFFFFu) ? 0 : count_ge(kk1 + 1);
    const long long eq = count_ge(kk1) - above;
    const long long tt = k - above;
    id1 = (tt < eq) ? nth_matching_id<T>(g, row, V, tt, [&](uint32_t bits, long long) { return order_key(bits) == kk1; }, sh.lscr)
                    : LLONG_MAX;
    k1count = k;
  }
  auto in_k1 = [&](uint32_t key, long long id) { return key > kk1 || (key == kk1 && id <= id1); };
  auto mass_ge = [&](uint32_t kk) -> float {
    float m = 0.f, mc = 0.f;  // compensated per-thread sum
    visit_row<T>(row, L, V, [&](uint32_t bits, long long id) {
      const uint32_t key = order_key(bits);
      if (key >= kk && in_k1(key, id)) {
        const float y = ex2((__uint_as_float(bits) - lmax) * x.c) - mc;
        const float z = m + y;
        mc = (z - m) - y;
        m = z;
      }
    });
    return group_sum(g, m - mc, sh.fscr);
  };
  uint32_t kcut = kk1;
  long long idcut = id1, keptc = k1count;
  const float s1 = mass_ge(0u);
  float skept = s1;
  if (x.topp) {
    const float target = (float)x.top_p_milli * 0.001f * s1;
    uint32_t lo = 0u, hi = kmax_f;
    while (lo < hi) {
      const uint32_t mid = lo + (uint32_t)(((uint64_t)hi - lo + 1) / 2);
      if (mass_ge(mid) >= target) lo = mid; else hi = mid - 1;
    }
    const uint32_t kp = lo;
    const float above = (kp == 0xFFFFFFFFu) ? 0.f : mass_ge(kp + 1);
    long long ca = 0, av = 0;
    visit_row<T>(row, L, V, [&](uint32_t bits, long long id) {
      const uint32_t key = order_key(bits);
      if (in_k1(key, id)) { ca += (key > kp) ? 1 : 0; av += (key == kp) ? 1 : 0; }
    });
    const long long cnt_above = group_sum_ll(g, ca, sh.lscr);
    const long long avail = group_sum_ll(g, av, sh.lscr);
    const float e1 = ex2((key_value(kp) - lmax) * x.c);
    long long n = (long long)ceilf(__fdiv_rn(target - above, e1));
    if (n < 1) n = 1;
    if (n > avail) n = avail;
    kcut = kp;
    keptc = cnt_above + n;
    skept = above + (float)n * e1;
    idcut = (n < avail) ? nth_matching_id<T>(g, row, V, n, [&](uint32_t bits, long long id) {
                            const uint32_t key = order_key(bits);
                            return key == kp && in_k1(key, id);
                          }, sh.lscr)
                        : (kp == kk1 ? id1 : LLONG_MAX);
  }
  out.thr_key = kcut;
  out.kept = (int)keptc;
  out.s_kept = skept;
  out.fallback = true;
  if (idcut == LLONG_MAX) {
    out.thr_n = LLONG_MAX;
  } else {  // tokens of the cut key up to idcut, in id order
    long long cnt = 0;
    visit_row<T>(row, L, V, [&](uint32_t bits, long long id) { cnt += (order_key(bits) == kcut && id <= idcut) ? 1 : 0; });
    out.thr_n = group_sum_ll(g, cnt, sh.lscr);
  }
}

// Tokens with order key `key` and an id below xt (group; second read of the row, from L2).
template <typename T>
__device__ long long count_key_before(const Group& g, RowShared& sh, const T* row, int64_t xt, uint32_t key) {
  const bool al = ((uintptr_t)row & 15u) == 0;
  long long c = 0;
#pragma unroll 4
  for (int64_t j0 = (int64_t)threadIdx.x * kEpt; j0 < xt; j0 += (int64_t)kCons * kEpt) {
    Raw8<T> r;
    load_raw8<T>(row, al, xt, j0, r);
    uint32_t b[kEpt];
    unpack_raw8<T>(r, b);
#pragma unroll
    for (int e = 0; e < kEpt; ++e) c += (j0 + e < xt && order_key(b[e]) == key) ? 1 : 0;
  }
  return group_sum_ll(g, c, sh.lscr);
}

// --------------------------------------------------------------------------------------
// Consumers: finish one row after its stages were reduced.  Returns true (every thread)
// when a bounded wait of the row gave up: nothing is written, the kernel stops.
// --------------------------------------------------------------------------------------
template <typename T>
__device__ bool finish_row(const RowArgs& A, RowShared& sh, const RowCtx& x, const RowPlan& plan,
                           ThreadAcc& acc, int w_on, uint32_t w_top16, uint32_t w_nb) {
  const Group g{kCons, kConsBar};
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  const int64_t V = A.io.V;
  const long long row_id = plan.row_id;
  const T* row = row_ptr<T>(A, row_id);
  const RowLayout L = row_layout(row, V);
  acc_scalars_mode<T>(x.mode, acc, row, L, V, x.c);
  if (x.window && w_on) {  // the row's unaligned ends go into the window too
    for (int64_t j = t; j < L.head; j += kCons) win_scalar(sh, load_bits(row, j), w_top16, w_nb);
    for (int64_t j = L.tail0 + t; j < V; j += kCons) win_scalar(sh, load_bits(row, j), w_top16, w_nb);
  }
  // warp merge (fixed butterfly), then the warps in order
  const float wfm = warp_reduce(acc.fm, [](float a, float b) { return fmax_nan(a, b); });
  const float mine = (acc.s == 0.f || acc.fm == -INFINITY) ? 0.f : (acc.s - acc.sc) * ex2((acc.fm - wfm) * x.c);
  const float ws = x.need_sum ? warp_reduce(mine, [](float a, float b) { return a + b; }) : 0.f;
  const long long wam = warp_min_i64(acc.fm == wfm ? acc.amax : LLONG_MAX);
  if (l == 0) { sh.w_fm[w] = wfm; sh.w_s[w] = ws; sh.w_amax[w] = wam; }
  g.sync();  // partials and the window histogram are complete
  if (sh.abort) return true;
  const bool filt = x.topk || x.topp;
  auto is_bad = [&](float lm, float s) {
    return (lm != lm || lm == INFINITY || lm == -INFINITY) || (x.need_sum && !(s < INFINITY));
  };
  float lmax = 0.f, s_all = 0.f;
  long long amax = LLONG_MAX;
  Thresholds th{0u, LLONG_MAX, (int)V, 0.f, false};
  bool done = false;
  if (w == 0) {  // the merged row (every lane of warp 0), and the window's cut
    float fm = -INFINITY;
    for (int i = 0; i < kConsWarps; ++i) fm = fmax_nan(fm, sh.w_fm[i]);
    float s = 0.f;
    long long am = LLONG_MAX;
    for (int i = 0; i < kConsWarps; ++i) {
      if (x.need_sum && sh.w_s[i] != 0.f && sh.w_fm[i] != -INFINITY) s += sh.w_s[i] * ex2((sh.w_fm[i] - fm) * x.c);
      if (sh.w_fm[i] == fm) am = min(am, (long long)sh.w_amax[i]);
    }
    lmax = fm; s_all = s; amax = am;
    th.s_kept = s_all;
    if (filt && !is_bad(lmax, s_all) && x.window && w_on) {
      const uint32_t kmax16 = order_key(__float_as_uint(lmax)) >> 16;
      const uint32_t top16 = w_top16, lo16 = top16 - (w_nb - 1u);
      if (kmax16 >= lo16 && kmax16 <= top16)
        done = warp_select(x, lmax, s_all, sh.hist + (top16 - kmax16), kmax16, (int)(kmax16 - lo16 + 1), th);
    }
    if (filt && l == 0) { sh.r_lmax = lmax; sh.r_s = s_all; sh.r_amax = amax; put_thresholds(sh, done, th); }
  }
  if (filt) {  // the group takes the cut (and searches again where the window did not decide)
    g.sync();
    lmax = sh.r_lmax; s_all = sh.r_s; amax = sh.r_amax;
    done = get_thresholds(sh, th);
    if (!is_bad(lmax, s_all) && !done) {
      th = Thresholds{0u, LLONG_MAX, (int)V, s_all, false};
      if (sizeof(T) == 2) {
        // the streamed window (8 nats below the first stage's maximum) missed the cut: 12
        // nats below the row maximum, then 24, then the 2048 values below it
        const float dz1 = 12.f;
        done = window_thresholds<T>(g, sh, row, L, x, V, lmax, s_all, dz1, th);
        if (!done) done = window_thresholds<T>(g, sh, row, L, x, V, lmax, s_all, 2.f * dz1, th);
        if (!done) done = window_thresholds<T>(g, sh, row, L, x, V, lmax, s_all, 0.f, th);
      }
      if (!done) generic_thresholds<T>(g, sh, row, L, x, V, lmax, order_key(__float_as_uint(lmax)), th);
    }
  }
  const bool bad = is_bad(lmax, s_all);  // exact in warp 0 and, for filtered rows, everywhere
  const uint32_t kmax = order_key(__float_as_uint(lmax));
  const bool filters = filt && !bad;
  uint32_t thr_key = 0u;
  long long thr_n = LLONG_MAX;
  if (x.one_hot) { thr_key = kmax; thr_n = 1; }
  else if (filters) { thr_key = th.thr_key; thr_n = th.thr_n; }
  // the draft token of the row: kept?  (Its rank among the tokens of the cut value when the
  // cut falls inside that value; counted over the ids before it.)
  int32_t xt = -1;
  uint32_t xb = 0u;
  bool kept_x = false;
  if (x.has_x && !bad) {
    xt = plan.xt;
    if (xt >= 0 && (int64_t)xt < V) {
      xb = sh.xbits;
      const uint32_t xk = order_key(xb);
      if (x.one_hot) kept_x = (xt == amax);
      else if (xk > thr_key) kept_x = true;
      else if (xk == thr_key) kept_x = (thr_n == LLONG_MAX) || count_key_before<T>(g, sh, row, xt, thr_key) < thr_n;
    } else {
      xt = -2;  // out of range: reported through the session status
    }
  }
  if (t == 0) {
    uint32_t flags = bad ? SDCP_ROW_INVALID : 0u;
    if (filters && th.fallback) flags |= SDCP_ROW_FALLBACK;
    RowStat st;
    st.lmax = lmax;
    st.argmax = (amax == LLONG_MAX) ? -1 : (int32_t)amax;
    st.thr_key = thr_key;
    st.thr_n = (thr_n == LLONG_MAX) ? INT_MAX : (int32_t)thr_n;
    if (x.one_hot) {
      st.s = 1.f; st.kept = 1;
    } else if (filters) {
      st.s = th.s_kept; st.kept = th.kept;
    } else {
      st.s = s_all; st.kept = (int32_t)V;
    }
    st.dlx = __int_as_float(0x7FC00000);
    if (xt >= 0) {
      flags |= kRowHasX;
      const float lx = __uint_as_float(xb);
      st.dlx = lx - lmax;
      if (kept_x && lx != -INFINITY) flags |= SDCP_ROW_X_KEPT;
    }
    st.flags = flags;
    A.stats[row_id] = st;
    if (A.pub) {
      sdcp_row_stat q;
      q.lmax = st.lmax;
      q.log_s = bad ? __int_as_float(0x7FC00000) : (float)log((double)st.s);
      q.argmax = st.argmax;
      q.kept = st.kept;
      q.thr_key = st.thr_key;
      q.thr_n = st.thr_n;
      q.flags = flags & ~kRowHasX;
      if (!(flags & kRowHasX)) q.lp_x = __int_as_float(0x7FC00000);
      else if (!(flags & SDCP_ROW_X_KEPT)) q.lp_x = -INFINITY;
      else if (x.one_hot) q.lp_x = 0.f;
      else q.lp_x = (float)((double)st.dlx * (1000.0 / (double)x.temperature_milli) - log((double)st.s));
      A.pub[row_id] = q;
    }
  }
  // no closing barrier: the next row's first barrier orders every later use of the scratch
  return false;
}

// A row claimed by the producer warp.
struct SlotInfo {
  long long row_id;  // -1: none
  bool skip;
  int32_t xt;        // the row's draft token (-1: none)
  RowCtx x;
};

// Row r (whole warp): its session and what it needs.
template <typename T>
__device__ SlotInfo resolve_row(const RowArgs& A, long long r) {
  SlotInfo s;
  s.row_id = -1;
  s.skip = true;
  s.xt = -1;
  const SessIO& io = A.io;
  const long long R_T = io.total + io.B;
  if (r >= R_T + io.total) return s;
  const bool is_target = r < R_T;
  const int32_t b = find_session(io.m_offsets, io.B, is_target ? r : r - R_T, is_target);
  // the draft token is loaded with the session's parameters and offsets (its index needs b
  // only), and kept when the row turns out to have one
  const long long tok_guess = is_target ? r - b : r - R_T;
  const int32_t tok = (tok_guess >= 0 && tok_guess < io.total) ? io.tokens[tok_guess] : -1;
  long long tok_idx = 0;
  s.x = row_ctx(A, r, b, sizeof(T) == 2, s.skip, tok_idx);
  s.row_id = r;
  s.xt = s.x.has_x ? tok : -1;
  return s;
}

// --------------------------------------------------------------------------------------
// The persistent row kernel.
// --------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kRowThreads, kRowCtasPerSm) row_stats_kernel(RowArgs A) {
  extern __shared__ __align__(128) unsigned char ring[];  // kStages * kChunk bytes
  __shared__ RowShared sh;
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  const long long nrows = 2 * A.io.total + A.io.B;
  pdl_launch_dependents();  // the session kernel may start its prologue now

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&sh.full[s], 1); mbar_init(&sh.empty[s], kConsWarps); }
    sh.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (w == kProducerWarp) {
    // ---------------- producer: claim rows, stream them into the ring ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    uint32_t issued = 0u, issued_par = 0u;  // lane 0: stages with a copy issued, and its parity
    // rows 0 .. gridDim.x - 1 go to the CTAs of the same index; later ones are claimed
    auto fetch = [&]() -> long long {
      unsigned long long r = 0;
      if (l == 0) r = atomicAdd(&A.hdr->next_slot, 1ull);
      return (long long)gridDim.x + (long long)__shfl_sync(0xFFFFFFFFu, r, 0);
    };
    const long long R_T = A.io.total + A.io.B;
    long long rcur = blockIdx.x;
    while (ok && rcur < nrows) {
      // A target row is copied before its session is looked up: its address needs no
      // context, the lookup then runs while the copy is in flight, and the row's plan is
      // published by the producer's arrival, which the stage's phase needs besides the copy's
      // bytes (an mbarrier's transaction count may go below zero until that arrival).  A
      // draft row is looked up first: a draft row that needs no statistics is not read.
      const bool early = rcur < R_T;
      SlotInfo cur;
      cur.row_id = rcur;
      cur.skip = false;
      cur.xt = -1;
      if (!early) {
        cur = resolve_row<T>(A, rcur);
        if (cur.skip) {
          if (l == 0) write_skipped(A, cur.row_id);
          rcur = fetch();
          continue;
        }
      }
      const T* row = row_ptr<T>(A, rcur);
      const RowLayout L = row_layout(row, A.io.V);
      const long long vbytes = L.nvec * 16;
      const int nch = (int)max(1ll, (vbytes + kChunk - 1) / kChunk);
      const char* src = reinterpret_cast<const char*>(row + L.head);
      long long rnext = nrows;
      for (int c = 0; c < nch && ok; ++c) {
        const long long off = (long long)c * kChunk;
        const uint32_t bytes = (uint32_t)max(0ll, min((long long)kChunk, vbytes - off));
        if (l == 0 && (!mbar_wait_spin(&sh.empty[stage], phase ^ 1u, &sh.abort) || sh.abort)) ok = false;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
        if (!ok) break;
        const bool first_early = (c == 0) && early;
#ifdef SDCP_TEST_WAIT_EXPIRY
        // test build: CTA 0 leaves the stage of its first row's first chunk unfilled (no copy,
        // no arrival), so its consumers' bounded wait runs out and the call reports
        // SDCP_S_INTERNAL; the stage is not marked issued, so no drain waits for it
        if (blockIdx.x == 0 && rcur == 0 && c == 0) {
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
          if (c == nch - 1) { rnext = fetch(); break; }
          continue;
        }
#endif
        if (l == 0) {
          if (first_early && bytes > 0) bulk_copy_g2s(ring + (size_t)stage * kChunk, src, bytes, &sh.full[stage]);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        }
        if (first_early) cur = resolve_row<T>(A, rcur);  // whole warp, the copy in flight
        const bool stop = first_early && cur.skip;       // only this stage was copied
        if (l == 0) {
          if (c == 0) sh.plan[stage] = RowPlan{cur.row_id, stop ? 1 : nch, cur.xt, stop, cur.x};
          mbar_arrive_expect_tx(&sh.full[stage], bytes);
          if (!first_early && bytes > 0)
            bulk_copy_g2s(ring + (size_t)stage * kChunk, src + off, bytes, &sh.full[stage]);
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
        // the next row once this row's last stage is issued; claiming earlier would let a
        // busy CTA hold a row that an idle one could take, which lengthens the tail
        if (c == nch - 1 || stop) {
          rnext = fetch();
          break;
        }
      }
      rcur = rnext;
    }
    if (l == 0) {
      if (ok && mbar_wait_for(&sh.empty[stage], phase ^ 1u, &sh.abort) && !sh.abort) {
        sh.plan[stage].row_id = -1;
        mbar_arrive_expect_tx(&sh.full[stage], 0);
      } else {
        sh.abort = 1;
        atomicOr(&A.hdr->error, 1u);
        // before the CTA may exit, the last copy issued into each stage must have landed
        // (at most one per stage is outstanding: a stage is refilled only after its last
        // copy was consumed); each wait is bounded by wall time
        for (int s = 0; s < kStages; ++s)
          if ((issued >> s) & 1u) (void)mbar_wait_for(&sh.full[s], (issued_par >> s) & 1u, nullptr);
      }
    }
    return;
  } else {
    // ---------------- consumers ----------------
    const Group g{kCons, kConsBar};
    int stage = 0;
    uint32_t phase = 0;
    ThreadAcc acc;
    acc.reset();
    while (true) {
      if (!mbar_wait_for(&sh.full[stage], phase, &sh.abort)) sh.abort = 1;
      g.sync();
      if (sh.abort) break;
      const RowPlan plan = sh.plan[stage];
      if (plan.row_id < 0) break;
      if (plan.skip) {  // copied before it was known to need nothing
        __syncwarp();
        if (l == 0) mbar_arrive(&sh.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
        if (t == 0) write_skipped(A, plan.row_id);
        continue;
      }
      const RowCtx& x = plan.x;
      const T* row = row_ptr<T>(A, plan.row_id);
      const RowLayout L = row_layout(row, A.io.V);
      if (x.window) {  // fresh window for this row (ordered before use by the anchor's barriers)
        for (int i = t; i < kWindowBins; i += kCons) sh.hist[i] = 0u;
        if (t < 32) sh.kbins[t] = 0u;
      }
      // the draft token's logit, loaded while the first stage is reduced
      const bool want_x = x.has_x && plan.xt >= 0 && (int64_t)plan.xt < A.io.V;
      uint32_t xbits = 0u;
      if (t == 0 && want_x) xbits = load_bits(row, plan.xt);
      bool fail = false;
      // the row's window (every thread holds the same copy; thread 0 also leaves it in
      // shared memory for finish_row)
      int w_on = 0, w_pos = 0;
      uint32_t w_top16 = 0u, w_nb = 0u;
      Window wn{0u, 0u, 0.f};
      for (int c = 0; c < plan.nchunks; ++c) {
        if (c > 0 && !mbar_wait_for(&sh.full[stage], phase, &sh.abort)) { fail = true; break; }
        const long long off = (long long)c * kChunk;
        const int nv = (int)(max(0ll, min((long long)kChunk, L.nvec * 16 - off)) / 16);
        const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)stage * kChunk);
        const long long id0 = L.head + (off / 16) * Elem<T>::kPerVec;
        if (!x.window || (c > 0 && !w_on)) {
          acc_stage_mode<T, false>(x.mode, acc, sv, nv, id0, x.c);
        } else if (c > 0) {
          const uint32_t hm = acc_stage_mode<T, true>(x.mode, acc, sv, nv, id0, x.c, wn.bot);
          if (w_pos) win_hits<true>(sh, sv, hm, wn);
          else win_hits<false>(sh, sv, hm, wn);
        } else {
          acc_stage_mode<T, false>(x.mode, acc, sv, nv, id0, x.c);
          // anchor: the maximum of the first stage; the window keeps every token within dz
          // nats of it, and room for values up to 2047 bf16 steps above its bottom
          const float wm = warp_reduce(acc.fm, [](float a, float b) { return fmax_nan(a, b); });
          if (l == 0) sh.w_m0[w] = wm;
          g.sync();  // the window histogram was cleared before this barrier too
          float m0 = -INFINITY;
          for (int i = 0; i < kConsWarps; ++i) m0 = fmax_nan(m0, sh.w_m0[i]);
          const float dz = 8.f;
          float lo = m0 - dz * x.inv_scale;
          if (x.topk && x.top_k <= (uint32_t)kCons && m0 == m0 && m0 > -INFINITY && m0 < INFINITY) {
            // top-k: the thread maxima of this stage are maxima of disjoint sets of tokens, so
            // if k of them are >= b, the row's k-th largest token is >= b.  b from a histogram
            // of their depths below m0, in half units of log2 (32 bins): the window then holds
            // the top-k cut, whatever the row's shape
            const float dd = (m0 - acc.fm) * x.c;
            atomicAdd(&sh.kbins[(dd >= 0.f && dd < 15.5f) ? (int)(dd * 2.f) : 31], 1u);
            g.sync();
            uint32_t cum = sh.kbins[l];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, cum, o);
              if (l >= o) cum += v;
            }
            const unsigned km = __ballot_sync(0xFFFFFFFFu, cum >= x.top_k);
            const int kb = km ? __ffs(km) - 1 : 32;
            if (kb < 31) lo = m0 - (float)(kb + 1) * 0.5f / x.c;  // one bf16 step of margin below
          }
          w_on = (m0 == m0 && m0 > -INFINITY && m0 < INFINITY && lo > -3.0e38f) ? 1 : 0;
          if (w_on) {
            uint32_t lo16 = order_key(__float_as_uint(lo)) >> 16;
            lo16 = lo16 > (kKeyNegInf >> 16) ? lo16 - 1 : (kKeyNegInf >> 16);
            w_top16 = min(lo16 + (uint32_t)(kWindowBins - 1), 0xFF7Fu);
            w_nb = w_top16 - lo16 + 1u;
            w_pos = lo16 > 0x8000u ? 1 : 0;
            wn = Window{w_pos ? w_top16 - 0x8000u : w_top16, w_nb, key_value(lo16 << 16)};
            const uint32_t hm = window_marks<T>(sv, nv, wn.bot);
            if (w_pos) win_hits<true>(sh, sv, hm, wn);
            else win_hits<false>(sh, sv, hm, wn);
          }

        }
        __syncwarp();
        if (l == 0) mbar_arrive(&sh.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (t == 0) sh.xbits = xbits;  // read by finish_row after its first barrier
      if (fail) sh.abort = 1;        // read by finish_row after its first barrier
      const bool aborted = finish_row<T>(A, sh, x, plan, acc, w_on, w_top16, w_nb);
      acc.reset();
      if (aborted) break;
    }
    if (t == 0 && sh.abort) atomicOr(&A.hdr->error, 1u);
  }

}

template __global__ void row_stats_kernel<float>(RowArgs);
template __global__ void row_stats_kernel<__nv_bfloat16>(RowArgs);

namespace {
constexpr int kMaxDevices = 64;
constexpr size_t kRingBytes = (size_t)kStages * kChunk;
struct DeviceCache {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  DeviceInfo info{0, 0};
};
DeviceCache g_device_cache[kMaxDevices];

// Once per device (with that device current): the SM count, the row kernels' shared-memory
// attributes (all of the unified L1/shared storage as shared memory, so two CTAs fit on an
// SM) and their occupancy.  A launch then costs no attribute or occupancy query.
cudaError_t setup_device(int dev, DeviceInfo* info) {
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && sms <= 0) e = cudaErrorInvalidDevice;
  int per_sm = kRowCtasPerSm;
  const void* fns[2] = {(const void*)row_stats_kernel<__nv_bfloat16>, (const void*)row_stats_kernel<float>};
  for (const void* fn : fns) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingBytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    int n = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kRowThreads, kRingBytes);
    if (e == cudaSuccess) per_sm = min(per_sm, max(n, 1));
  }
  info->sms = sms;
  info->row_ctas_per_sm = per_sm;
  return e;
}
}  // namespace

bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  DeviceCache& c = g_device_cache[dev];
  std::call_once(c.once, [&] { c.err = setup_device(dev, &c.info); });
  if (c.err != cudaSuccess) return false;
  *out = c.info;
  return true;
}

int launch_row_stats(const RowArgs& a, int dtype, cudaStream_t stream) {
  const long long rows = a.io.total + a.io.B + a.io.total;
  if (rows <= 0) return 0;
  DeviceInfo di;
  if (!device_info(&di)) return (int)cudaErrorInvalidDevice;
  const long long grid = min(rows, (long long)di.sms * di.row_ctas_per_sm);
  if (dtype == SDCP_BF16)
    row_stats_kernel<__nv_bfloat16><<<(unsigned)grid, kRowThreads, kRingBytes, stream>>>(a);
  else
    row_stats_kernel<float><<<(unsigned)grid, kRowThreads, kRingBytes, stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp
