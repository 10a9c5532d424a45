// sdcp_device.cuh - device helpers of libsdcp (sm_103a): order keys, Philox4x32-10,
// deterministic block reductions and scans, row slicing.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sdcp.h"

namespace sdcp {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;          // threads of a group that runs a session completion
constexpr int kWarps = kThreads / 32;
constexpr int kWindowBins = 2048;      // exact bf16 keys below the row maximum
constexpr int kEpt = 8;                // ids per lane piece of the draw passes

// Internal per-row record written by the row kernel (workspace), 32 bytes.
struct RowStat {
  float lmax;        // largest logit of the row
  float s;           // sum over the kept set of exp((l - lmax) * 1000/T); 1 at T = 0
  float dlx;         // l[x] - lmax for the row's draft token (-inf: x has a -inf logit)
  int32_t argmax;    // smallest id of the largest logit (rows that need it)
  uint32_t thr_key;  // kept: key > thr_key, or key == thr_key and among the first thr_n
  int32_t thr_n;     //   tokens with that key in id order (INT_MAX: all of them)
  int32_t kept;      // size of the kept set
  uint32_t flags;    // SDCP_ROW_* plus kRowHasX
};
constexpr uint32_t kRowHasX = 16u;     // the row carries a draft token that is in range

static_assert(sizeof(RowStat) == 32, "RowStat layout");

// Workspace: a 256-byte header (cleared before every call), then one RowStat per scored
// row (target rows, then draft rows).
struct WsHeader {
  uint32_t error;                // non-zero: a bounded wait gave up
  uint32_t pad;
  unsigned long long next_slot;  // next row of the dynamic schedule
};
constexpr size_t kWsHeader = 256;

// Everything a session completion reads and writes.
struct SessIO {
  const void* target;
  const void* draft;
  int64_t V;
  int32_t B;
  const int32_t* m_offsets;
  int64_t total;
  const int32_t* tokens;
  const sdcp_session_params* params;
  const RowStat* stats;
  int32_t* accepted;
  int32_t* n_out;
  int32_t* out_tokens;
  int32_t* status;
  const uint32_t* error;  // non-zero: a bounded wait of the call gave up
  uint32_t rng;                // SDCP_RNG_*
  const uint8_t* session_ids;  // [B][16] session identifiers (SDCP_RNG_HMAC_SHA256)
  const float* q_rows;         // [total][V] q as binary32 probabilities, or null (q from logits)
};

// Arguments of the row kernel.
struct RowArgs {
  SessIO io;                  // inputs (outputs unused) and the statistics
  RowStat* stats;             // [total + B + total], writable view of io.stats
  sdcp_row_stat* pub;         // optional public copy (statistics mode)
  int stats_mode;             // 1: every row gets the full statistics
  WsHeader* hdr;
};

int launch_row_stats(const RowArgs& a, int dtype, cudaStream_t stream);
int check_common(const void* target, int dtype, int64_t V, int32_t B, const int32_t* m_offsets,
                 int64_t total, const int32_t* tokens, const sdcp_session_params* params,
                 const void* draft);

// Device facts the launches need, looked up once per device (the SM count, and the
// kernels' shared-memory attributes set once).  Returns false if the device query failed.
struct DeviceInfo {
  int sms;
  int row_ctas_per_sm;
};
bool device_info(DeviceInfo* out);
int launch_sessions(const SessIO& a, int dtype, bool pdl, cudaStream_t stream);

// ---------------------------------------------------------------------------------
// Order key of a binary32 bit pattern: unsigned order of keys = numeric order of the
// values, -0 and +0 share a key (so ties between them go to the smaller id).
// Positive x: bits | 2^31.  Negative x: -bits (two's complement), which maps -0 onto
// +0's key and keeps every other negative value below it.
// +inf -> 0xFF800000, -inf -> 0x00800000; NaNs fall outside [0x00800000, 0xFF800000].
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  uint32_t t = (uint32_t)((int32_t)bits >> 31);
  return (bits ^ (t | 0x80000000u)) - t;
}
__device__ __forceinline__ float key_value(uint32_t key) {
  uint32_t bits = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : (0u - key);
  return __uint_as_float(bits);
}
constexpr uint32_t kKeyPosInf = 0xFF800000u;
constexpr uint32_t kKeyNegInf = 0x00800000u;

// 2^x on the SFU (PTX ex2.approx, flush-to-zero; ~2 ulp relative).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max that propagates NaN (PTX max.NaN).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// The sampling profile's temperature as the kernels apply it (Section 4.1: logits / T with
// T = temperature_milli / 1000), in fp32 so no per-row step needs the slow fp64 pipe:
// c = log2(e) * 1000 / T, so that exp((l - m) / T) = 2^((l - m) c), and the inverse scale
// T / 1000 that turns nats into logit units.  Every kernel uses these two, so the row
// statistics and the draws agree bit for bit.
__device__ __forceinline__ float profile_c(uint32_t temperature_milli) {
  return __fdiv_rn(1442.6950408889634f, (float)temperature_milli);
}
__device__ __forceinline__ float profile_inv_scale(uint32_t temperature_milli) {
  return (float)temperature_milli * 0.001f;
}

// ---------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): per round the pair of 32x32->64
// products with multipliers 0xD2511F53 (of word 0) and 0xCD9E8D57 (of word 2) is mixed
// with words 1 and 3 and the key; the key advances by 0x9E3779B9 / 0xBB67AE85.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    uint32_t h0 = __umulhi(m0, c.x), l0 = m0 * c.x;
    uint32_t h1 = __umulhi(m1, c.z), l1 = m1 * c.z;
    c = make_uint4(h1 ^ c.y ^ k.x, l1, h0 ^ c.w ^ k.y, l0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}
// The verifier's uniform for (position, purpose) of one session: 53 bits / 2^53.
__device__ __forceinline__ double verifier_uniform(const sdcp_session_params& p,
                                                   uint32_t position, uint32_t purpose) {
  uint4 w = philox4x32_10(make_uint4(position, purpose, p.round, p.session_tag),
                          make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
  unsigned long long bits = ((unsigned long long)w.x << 21) | (unsigned long long)(w.y >> 11);
  return (double)bits * 0x1.0p-53;
}

// ---------------------------------------------------------------------------------
// Element access.
// ---------------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static uint32_t bits(float v) { return __float_as_uint(v); }
  __device__ __forceinline__ static void unpack(const uint4& q, uint32_t (&b)[4]) {
    b[0] = q.x; b[1] = q.y; b[2] = q.z; b[3] = q.w;
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ __forceinline__ static uint32_t bits(__nv_bfloat16 v) {
    return ((uint32_t)__bfloat16_as_ushort(v)) << 16;
  }
  __device__ __forceinline__ static void unpack(const uint4& q, uint32_t (&b)[8]) {
    b[0] = q.x << 16; b[1] = q.x & 0xFFFF0000u;
    b[2] = q.y << 16; b[3] = q.y & 0xFFFF0000u;
    b[4] = q.z << 16; b[5] = q.z & 0xFFFF0000u;
    b[6] = q.w << 16; b[7] = q.w & 0xFFFF0000u;
  }
};

template <typename T>
__device__ __forceinline__ uint32_t load_bits(const T* row, int64_t j) {
  return Elem<T>::bits(row[j]);
}


// A row split into: head (scalar elements up to the first 16-byte boundary), nvec full
// 16-byte vectors, and a scalar tail.
struct RowLayout {
  int64_t head, nvec, tail0;  // tail elements are [tail0, V)
};
template <typename T>
__device__ __forceinline__ RowLayout row_layout(const T* row, int64_t V) {
  constexpr int E = Elem<T>::kPerVec;
  uintptr_t a = (uintptr_t)row;
  int64_t head = (int64_t)(((16u - (uint32_t)(a & 15u)) & 15u) / sizeof(T));
  if (head > V) head = V;
  int64_t nvec = (V - head) / E;
  RowLayout L;
  L.head = head;
  L.nvec = nvec;
  L.tail0 = head + nvec * E;
  return L;
}

// ---------------------------------------------------------------------------------
// Deterministic reductions: fixed butterfly per warp, then warp 0 over the warp results.
// ---------------------------------------------------------------------------------
template <typename F>
__device__ __forceinline__ float warp_reduce(float v, F op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ int64_t warp_max_i64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, (int64_t)__shfl_xor_sync(0xFFFFFFFFu, (long long)v, o));
  return v;
}
__device__ __forceinline__ int64_t warp_min_i64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, (int64_t)__shfl_xor_sync(0xFFFFFFFFu, (long long)v, o));
  return v;
}
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Session of a row by a warp-cooperative 128-ary search over m_offsets: the largest b in
// [0, B) with key(b) <= r, key(b) = m_offsets[b] + (target ? b : 0).  Clamped to [0, B).
__device__ __forceinline__ int32_t find_session(const int32_t* __restrict__ m_offsets, int32_t B,
                                                int64_t r, bool target) {
  int64_t lo = 0, hi = B;
  const int l = threadIdx.x & 31;
  while (hi - lo > 1) {  // 128 candidates a round: lane l tests 4 consecutive ones
    const int64_t step = (hi - lo + 127) / 128;
    int lastc = -1;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = l * 4 + q;
      const int64_t j = lo + (int64_t)c * step;
      if (j < hi && (int64_t)__ldg(&m_offsets[j]) + (target ? j : 0) <= r) lastc = c;
    }
    const int best = max(0, (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)(lastc + 1)) - 1);
    const int64_t nlo = lo + (int64_t)best * step;
    const int64_t nhi = nlo + step;
    lo = nlo;
    hi = nhi < hi ? nhi : hi;
  }
  return (int32_t)lo;
}

// ---------------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA) primitives, PTX ISA 8.x, shared::cta addresses.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }"
               ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return done != 0;
}
// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// A waiting thread sleeps until the phase completes or kSuspendNs pass (so a waiting warp
// takes no issue slots from the warps that work); a wait gives up after kWaitNs in all.
constexpr uint32_t kSuspendNs = 100000;
#ifdef SDCP_TEST_WAIT_EXPIRY
// Test build only (the flag is never set in the library): waits give up after 20 ms, and the
// row kernel leaves one ring stage unfilled (sdcp_rows.cu), so a wait runs out on purpose.
constexpr unsigned long long kWaitNs = 20000000ull;
#else
constexpr unsigned long long kWaitNs = 2000000000ull;
#endif
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
               : "=r"(done) : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs) : "memory");
  return done != 0;
}
// Bounded wait that polls without sleeping (for a warp whose next work is the awaited data).
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}
// Bounded wait for the phase of `parity`: false after kWaitNs, or at once when *abort is set
// (another role of the block gave up; abort may be null).
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}
// Global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Named barrier 1 (the id is a literal, so a kernel reserves no other barrier for it).
__device__ __forceinline__ void named_sync1(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
// Programmatic dependent launch controls (no-ops when the launch did not enable them).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// Reductions over a group of warps 0..nw-1 that share a named barrier (fixed order).
// scratch needs 2 * 32 + 2 entries.
// ---------------------------------------------------------------------------------
// A group of warps 0 .. nthreads/32 - 1 of a CTA that synchronises on named barrier 1.
struct Group {
  int nthreads;
  int bar;  // always 1
  __device__ __forceinline__ void sync() const { named_sync1(nthreads); }
  __device__ __forceinline__ int nwarps() const { return nthreads >> 5; }
};
__device__ __forceinline__ float group_sum(const Group& g, float v, float* scratch) {
  v = warp_reduce(v, [](float a, float b) { return a + b; });
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  g.sync();
  if (l == 0) scratch[w] = v;
  g.sync();
  float r = 0.f;
  for (int i = 0; i < g.nwarps(); ++i) r += scratch[i];
  return r;
}
__device__ __forceinline__ long long group_sum_ll(const Group& g, long long v, long long* scratch) {
  v = warp_sum_ll(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  g.sync();
  if (l == 0) scratch[w] = v;
  g.sync();
  long long r = 0;
  for (int i = 0; i < g.nwarps(); ++i) r += scratch[i];
  return r;
}
__device__ __forceinline__ int64_t group_max_i64(const Group& g, int64_t v, long long* scratch) {
  v = warp_max_i64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  g.sync();
  if (l == 0) scratch[w] = v;
  g.sync();
  int64_t r = INT64_MIN;
  for (int i = 0; i < g.nwarps(); ++i) r = max(r, (int64_t)scratch[i]);
  return r;
}
__device__ __forceinline__ int64_t group_min_i64(const Group& g, int64_t v, long long* scratch) {
  v = warp_min_i64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  g.sync();
  if (l == 0) scratch[w] = v;
  g.sync();
  int64_t r = INT64_MAX;
  for (int i = 0; i < g.nwarps(); ++i) r = min(r, (int64_t)scratch[i]);
  return r;
}
// Exclusive scans over the group (fixed association); *total = group sum.
__device__ __forceinline__ float group_excl_scan(const Group& g, float v, float* scratch, float* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (l >= o) incl += t;
  }
  float ex = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (l == 0) ex = 0.f;
  g.sync();
  if (l == 31) scratch[w] = incl;
  g.sync();
  float base = 0.f, tot = 0.f;
  for (int i = 0; i < g.nwarps(); ++i) {
    if (i == w) base = tot;
    tot += scratch[i];
  }
  *total = tot;
  return base + ex;
}
__device__ __forceinline__ long long group_excl_scan_ll(const Group& g, long long v, long long* scratch,
                                                        long long* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (l >= o) incl += t;
  }
  long long ex = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (l == 0) ex = 0;
  g.sync();
  if (l == 31) scratch[w] = incl;
  g.sync();
  long long base = 0, tot = 0;
  for (int i = 0; i < g.nwarps(); ++i) {
    if (i == w) base = tot;
    tot += scratch[i];
  }
  *total = tot;
  return base + ex;
}

}  // namespace sdcp
