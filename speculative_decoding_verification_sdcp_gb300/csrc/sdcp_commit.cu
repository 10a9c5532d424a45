// sdcp_commit.cu - the commit step after acceptance (SDCP draft
// draft-li-mlc-inference-acceleration-00): Section 6.3 step "Acceptance" (truncation of the
// emitted tokens after the first stop token and at max_new), step "Commit" (n and the
// committed-prefix digest d[n] of Section 4.2) and step "Control" (Section 6.5: low rounds,
// the counters c, g, j, the fallback ladder and m_cap).
//
// One thread per session: the digest chain is sequential within a session (each link hashes
// the previous digest), and a session commits at most M + 1 <= 65 tokens, one SHA-256
// compression each.  The sessions of a batch run in parallel.
#include "sdcp_device.cuh"
#include "sdcp_sha256.cuh"

namespace sdcp {

namespace {

constexpr int kCommitThreads = 128;

struct CommitArgs {
  int32_t B;
  const int32_t* m_offsets;
  const int32_t* accepted;
  int32_t* n_out;
  int32_t* out_tokens;
  const int32_t* status;
  const sdcp_commit_params* cparams;
  const uint32_t* stop_tokens;
  sdcp_session_state* state;
  uint32_t load;
  int32_t* action;
};

__device__ __forceinline__ uint32_t load_be32(const uint8_t* p) {
  return ((uint32_t)p[0] << 24) | ((uint32_t)p[1] << 16) | ((uint32_t)p[2] << 8) | (uint32_t)p[3];
}
__device__ __forceinline__ void store_be32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)(v >> 24); p[1] = (uint8_t)(v >> 16); p[2] = (uint8_t)(v >> 8); p[3] = (uint8_t)v;
}

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(CommitArgs A) {
  const int32_t b = (int32_t)(blockIdx.x * kCommitThreads + threadIdx.x);
  if (b >= A.B) return;
  if (A.status[b] != SDCP_S_OK) {
    A.action[b] = SDCP_ACTION_NONE;
    return;
  }
  const sdcp_commit_params cp = A.cparams[b];
  sdcp_session_state st = A.state[b];
  const int64_t off0 = A.m_offsets[b], M = (int64_t)A.m_offsets[b + 1] - off0;
  const int32_t a = A.accepted[b];
  int32_t* toks = A.out_tokens + off0 + b;
  const int32_t n0 = A.n_out[b];

  // truncation after the first stop token, then at max_new
  int32_t n = n0;
  bool finished = false;
  for (int32_t k = 0; k < n; ++k) {
    const uint32_t t = (uint32_t)toks[k];
    bool stop = false;
    for (uint32_t s = 0; s < cp.stop_count; ++s) stop |= (t == A.stop_tokens[cp.stop_offset + s]);
    if (stop) { n = k + 1; finished = true; break; }
  }
  const uint32_t room = (st.committed >= cp.max_new) ? 0u : cp.max_new - st.committed;
  if ((uint32_t)n >= room) { n = (int32_t)room; finished = true; }
  for (int32_t k = n; k < n0; ++k) toks[k] = -1;
  A.n_out[b] = n;

  // commit: d[k] = SHA-256(d[k-1] || uint32(o[k])) for the tokens kept
  Sha256State d;
#pragma unroll
  for (int i = 0; i < 8; ++i) d.h[i] = load_be32(st.digest + 4 * i);
  for (int32_t k = 0; k < n; ++k) d = digest_link(d, (uint32_t)toks[k]);
#pragma unroll
  for (int i = 0; i < 8; ++i) store_be32(st.digest + 4 * i, d.h[i]);
  st.committed += (uint32_t)n;

  // control (Section 6.5)
  const uint32_t R = cp.low_rounds < 1u ? 1u : cp.low_rounds;
  const uint32_t nfb = cp.fallback_len > 8u ? 8u : cp.fallback_len;
  const bool low = (cp.low_ratio != 0u) ? (100ull * (uint32_t)a < (unsigned long long)cp.low_ratio * (uint64_t)M)
                                        : (a == 0);
  if (low) {
    st.c += 1u;
    st.g = 0u;
  } else {
    st.c = 0u;
    st.g += 1u;
    if (st.g >= R) st.j = 0u;
    const uint32_t mc = st.m_cap + cp.m_restore;
    st.m_cap = mc > cp.m_max ? cp.m_max : mc;
  }
  int32_t act = SDCP_ACTION_CONTINUE;
  if (finished) {
    act = SDCP_ACTION_FINISH;
  } else if (st.c >= R) {
    act = SDCP_ACTION_FAIL;  // unless an entry remains
    while (st.j < nfb) {
      const uint32_t e = cp.fallback[st.j];
      st.j += 1u;
      if (e == SDCP_ACTION_SELF_DECODE && !(cp.self_load <= 100u && A.load <= cp.self_load)) continue;
      act = (int32_t)e;
      break;
    }
    st.c = 0u;
    if (act == SDCP_ACTION_REDUCE) st.m_cap = st.m_cap / 2u > 1u ? st.m_cap / 2u : 1u;
  }
  A.state[b] = st;
  A.action[b] = act;
}

}  // namespace

int launch_commit(int32_t B, const int32_t* m_offsets, const int32_t* accepted, int32_t* n_out,
                  int32_t* out_tokens, const int32_t* status, const sdcp_commit_params* cparams,
                  const uint32_t* stop_tokens, sdcp_session_state* state, uint32_t load,
                  int32_t* action, cudaStream_t stream) {
  if (B <= 0) return 0;
  const CommitArgs a{B, m_offsets, accepted, n_out, out_tokens, status, cparams, stop_tokens, state,
                     load, action};
  const unsigned grid = (unsigned)((B + kCommitThreads - 1) / kCommitThreads);
  commit_kernel<<<grid, kCommitThreads, 0, stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp

extern "C" int sdcp_commit_batch(int32_t B, const int32_t* m_offsets, const int32_t* accepted,
                                 int32_t* n_out, int32_t* out_tokens, const int32_t* status,
                                 const sdcp_commit_params* cparams, const uint32_t* stop_tokens,
                                 sdcp_session_state* state, uint32_t load_percent, int32_t* action,
                                 void* stream) {
  if (B < 0) return SDCP_E_INVALID;
  if (B == 0) return SDCP_OK;
  if (!m_offsets || !accepted || !n_out || !out_tokens || !status || !cparams || !state || !action)
    return SDCP_E_INVALID;
  return sdcp::launch_commit(B, m_offsets, accepted, n_out, out_tokens, status, cparams, stop_tokens,
                             state, load_percent, action, reinterpret_cast<cudaStream_t>(stream)) != 0
             ? SDCP_E_LAUNCH
             : SDCP_OK;
}
