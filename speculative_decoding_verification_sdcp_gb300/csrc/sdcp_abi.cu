// sdcp_abi.cu - the C ABI of libsdcp (declared in include/sdcp.h): argument checks on
// the host, the workspace layout, and the launches on the caller's stream: a clear of the
// workspace header, the row kernel, then the session kernel (a programmatic dependent of
// the row kernel in sdcp_verify_batch).
#include <climits>
#include <vector>

#include "sdcp_device.cuh"

namespace sdcp {

namespace {
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

// Host-side checks every verify entry point runs first, in this order.
int check_common(const void* target, int dtype, int64_t V, int32_t B, const int32_t* m_offsets,
                 int64_t total, const int32_t* tokens, const sdcp_session_params* params,
                 const void* draft) {
  if (B < 0 || total < 0 || V < 1) return SDCP_E_INVALID;
  if (dtype != SDCP_F32 && dtype != SDCP_BF16) return SDCP_E_INVALID;
  if (V > SDCP_MAX_VOCAB) return SDCP_E_TOO_LARGE;
  if (total + B + total > (int64_t)INT32_MAX / 2) return SDCP_E_TOO_LARGE;
  if (B == 0) return SDCP_OK;
  if (!target || !m_offsets || !params || (total > 0 && !tokens)) return SDCP_E_INVALID;
  const size_t esz = dtype == SDCP_BF16 ? 2 : 4;
  if (((uintptr_t)target % esz) != 0 || (draft && ((uintptr_t)draft % esz) != 0)) return SDCP_E_ALIGN;
  return SDCP_OK;
}

namespace {
int check_workspace(void* workspace, size_t workspace_bytes, int64_t V, int32_t B, int64_t total);
}  // namespace
}  // namespace sdcp

using namespace sdcp;

extern "C" size_t sdcp_workspace_bytes(int64_t V, int32_t B, int64_t total_drafts) {
  if (B < 0 || total_drafts < 0 || V < 1 || V > SDCP_MAX_VOCAB) return 0;
  return kWsHeader + align256((size_t)(total_drafts + B + total_drafts) * sizeof(RowStat));
}

namespace sdcp {
namespace {
int check_workspace(void* workspace, size_t workspace_bytes, int64_t V, int32_t B, int64_t total) {
  if (!workspace || ((uintptr_t)workspace & 255u) != 0 ||
      workspace_bytes < sdcp_workspace_bytes(V, B, total))
    return SDCP_E_WORKSPACE;
  return SDCP_OK;
}

// The session inputs and outputs, with the workspace's statistics and error word.
SessIO make_io(const void* target, const void* draft, int64_t V, int32_t B, const int32_t* m_offsets,
               int64_t total, const int32_t* tokens, const sdcp_session_params* params,
               int32_t* accepted, int32_t* n_out, int32_t* out_tokens, int32_t* status, void* ws) {
  char* w = static_cast<char*>(ws);
  return SessIO{target, draft, V, B, m_offsets, total, tokens, params,
                reinterpret_cast<const RowStat*>(w + kWsHeader),
                accepted, n_out, out_tokens, status, reinterpret_cast<const uint32_t*>(w),
                SDCP_RNG_PHILOX4X32_10, nullptr, nullptr};
}

// Clears the header, then launches the row kernel.
int launch_rows(const SessIO& io, void* ws, sdcp_row_stat* pub, int stats_mode, int dtype, cudaStream_t s) {
  char* w = static_cast<char*>(ws);
  if (cudaMemsetAsync(w, 0, kWsHeader, s) != cudaSuccess) return SDCP_E_LAUNCH;
  RowArgs ra{io, const_cast<RowStat*>(io.stats), pub, stats_mode, reinterpret_cast<WsHeader*>(w)};
  return launch_row_stats(ra, dtype, s) != 0 ? SDCP_E_LAUNCH : SDCP_OK;
}
}  // namespace
}  // namespace sdcp

using namespace sdcp;

extern "C" {

int sdcp_abi_version(void) { return SDCP_ABI_VERSION; }

const char* sdcp_strerror(int code) {
  switch (code) {
    case SDCP_OK: return "success";
    case SDCP_E_INVALID: return "invalid argument (null pointer, negative size, V < 1 or unknown dtype)";
    case SDCP_E_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case SDCP_E_ALIGN: return "logits pointer not aligned to its element size";
    case SDCP_E_TOO_LARGE: return "vocabulary or row count above the supported maximum";
    case SDCP_E_LAUNCH: return "CUDA kernel launch failed";
    case SDCP_E_DEVICE: return "no usable CUDA device";
    case SDCP_E_SCRATCH_LIMIT:
      return "batch needs more scratch than the library's no-alloc array (SDCP_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown sdcp error code";
  }
}

int sdcp_verify_rows(const void* target_logits, const void* draft_logits, int dtype, int64_t V,
                     int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                     const int32_t* draft_tokens, const sdcp_session_params* params,
                     void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_common(target_logits, dtype, V, B, m_offsets, total_drafts, draft_tokens, params,
                        draft_logits);
  if (rc != SDCP_OK) return rc;
  if (B == 0) return SDCP_OK;
  rc = check_workspace(workspace, workspace_bytes, V, B, total_drafts);
  if (rc != SDCP_OK) return rc;
  const SessIO io = make_io(target_logits, draft_logits, V, B, m_offsets, total_drafts, draft_tokens,
                            params, nullptr, nullptr, nullptr, nullptr, workspace);
  return launch_rows(io, workspace, nullptr, 0, dtype, reinterpret_cast<cudaStream_t>(stream));
}

static int verify_sessions(const void* target_logits, const void* draft_logits, int dtype, int64_t V,
                           int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                           const int32_t* draft_tokens, const sdcp_session_params* params,
                           int32_t* accepted, int32_t* n_out, int32_t* out_tokens, int32_t* status,
                           void* workspace, size_t workspace_bytes, void* stream, bool pdl,
                           const sdcp_verify_options* opts = nullptr) {
  int rc = check_common(target_logits, dtype, V, B, m_offsets, total_drafts, draft_tokens, params,
                        draft_logits);
  if (rc != SDCP_OK) return rc;
  if (B == 0) return SDCP_OK;
  if (!accepted || !n_out || !out_tokens || !status) return SDCP_E_INVALID;
  rc = check_workspace(workspace, workspace_bytes, V, B, total_drafts);
  if (rc != SDCP_OK) return rc;
  SessIO io = make_io(target_logits, draft_logits, V, B, m_offsets, total_drafts, draft_tokens,
                      params, accepted, n_out, out_tokens, status, workspace);
  if (opts) {
    io.rng = opts->rng_id;
    io.session_ids = opts->session_ids;
    io.q_rows = opts->q_rows;
  }
  if (launch_sessions(io, dtype, pdl, reinterpret_cast<cudaStream_t>(stream)) != 0) return SDCP_E_LAUNCH;
  return SDCP_OK;
}

// Checks of the options of sdcp_verify_batch_ex (NULL: the defaults).
static int check_options(const sdcp_verify_options* opts) {
  if (!opts) return SDCP_OK;
  if (opts->struct_size < sizeof(sdcp_verify_options)) return SDCP_E_INVALID;
  if (opts->rng_id != SDCP_RNG_PHILOX4X32_10 && opts->rng_id != SDCP_RNG_HMAC_SHA256) return SDCP_E_INVALID;
  if (opts->rng_id == SDCP_RNG_HMAC_SHA256 && !opts->session_ids) return SDCP_E_INVALID;
  if (opts->q_rows && ((uintptr_t)opts->q_rows % sizeof(float)) != 0) return SDCP_E_ALIGN;
  return SDCP_OK;
}

int sdcp_verify_sessions(const void* target_logits, const void* draft_logits, int dtype, int64_t V,
                         int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                         const int32_t* draft_tokens, const sdcp_session_params* params,
                         int32_t* accepted, int32_t* n_out, int32_t* out_tokens, int32_t* status,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return verify_sessions(target_logits, draft_logits, dtype, V, B, m_offsets, total_drafts,
                         draft_tokens, params, accepted, n_out, out_tokens, status, workspace,
                         workspace_bytes, stream, false);
}

int sdcp_verify_batch(const void* target_logits, const void* draft_logits, int dtype, int64_t V,
                      int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                      const int32_t* draft_tokens, const sdcp_session_params* params,
                      int32_t* accepted, int32_t* n_out, int32_t* out_tokens, int32_t* status,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (B > 0 && (!accepted || !n_out || !out_tokens || !status)) {
    int rc = check_common(target_logits, dtype, V, B, m_offsets, total_drafts, draft_tokens,
                          params, draft_logits);
    return rc != SDCP_OK ? rc : SDCP_E_INVALID;
  }
  int rc = sdcp_verify_rows(target_logits, draft_logits, dtype, V, B, m_offsets, total_drafts,
                            draft_tokens, params, workspace, workspace_bytes, stream);
  if (rc != SDCP_OK || B == 0) return rc;
  // phase 2 is a programmatic dependent of phase 1: its launch overlaps phase 1's tail
  return verify_sessions(target_logits, draft_logits, dtype, V, B, m_offsets, total_drafts,
                         draft_tokens, params, accepted, n_out, out_tokens, status, workspace,
                         workspace_bytes, stream, true);
}

int sdcp_verify_batch_ex(const void* target_logits, const void* draft_logits, int dtype, int64_t V,
                         int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                         const int32_t* draft_tokens, const sdcp_session_params* params,
                         int32_t* accepted, int32_t* n_out, int32_t* out_tokens, int32_t* status,
                         void* workspace, size_t workspace_bytes, const sdcp_verify_options* opts,
                         void* stream) {
  int rc = check_common(target_logits, dtype, V, B, m_offsets, total_drafts, draft_tokens, params,
                        draft_logits);
  if (rc != SDCP_OK) return rc;
  rc = check_options(opts);
  if (rc != SDCP_OK) return rc;
  if (B > 0 && (!accepted || !n_out || !out_tokens || !status)) return SDCP_E_INVALID;
  if (B == 0) return SDCP_OK;
  rc = check_workspace(workspace, workspace_bytes, V, B, total_drafts);
  if (rc != SDCP_OK) return rc;
  SessIO io = make_io(target_logits, draft_logits, V, B, m_offsets, total_drafts, draft_tokens, params,
                      nullptr, nullptr, nullptr, nullptr, workspace);
  if (opts) io.q_rows = opts->q_rows;
  rc = launch_rows(io, workspace, nullptr, 0, dtype, reinterpret_cast<cudaStream_t>(stream));
  if (rc != SDCP_OK) return rc;
  return verify_sessions(target_logits, draft_logits, dtype, V, B, m_offsets, total_drafts,
                         draft_tokens, params, accepted, n_out, out_tokens, status, workspace,
                         workspace_bytes, stream, true, opts);
}

int sdcp_row_stats(const void* target_logits, const void* draft_logits, int dtype, int64_t V,
                   int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                   const int32_t* draft_tokens, const sdcp_session_params* params,
                   sdcp_row_stat* stats_out, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int rc = check_common(target_logits, dtype, V, B, m_offsets, total_drafts, draft_tokens, params,
                        draft_logits);
  if (rc != SDCP_OK) return rc;
  if (B == 0) return SDCP_OK;
  if (!stats_out) return SDCP_E_INVALID;
  if (total_drafts > 0 && !draft_logits) return SDCP_E_INVALID;
  rc = check_workspace(workspace, workspace_bytes, V, B, total_drafts);
  if (rc != SDCP_OK) return rc;
  const SessIO io = make_io(target_logits, draft_logits, V, B, m_offsets, total_drafts, draft_tokens,
                            params, nullptr, nullptr, nullptr, nullptr, workspace);
  return launch_rows(io, workspace, stats_out, 1, dtype, reinterpret_cast<cudaStream_t>(stream));
}

int sdcp_split_sessions(const int32_t* m_offsets, const sdcp_session_params* params, int32_t B,
                        int32_t n_parts, int32_t* bounds) {
  if (!m_offsets || !bounds || B < 0 || n_parts < 1) return SDCP_E_INVALID;
  if (m_offsets[0] != 0) return SDCP_E_INVALID;
  for (int32_t b = 0; b < B; ++b)
    if (m_offsets[b + 1] < m_offsets[b]) return SDCP_E_INVALID;
  // prefix of scored rows: M_b + 1 target rows, plus M_b draft rows under Rule 2
  std::vector<int64_t> pre((size_t)B + 1, 0);
  for (int32_t b = 0; b < B; ++b) {
    const int64_t M = (int64_t)m_offsets[b + 1] - m_offsets[b];
    const bool rule2 = !params || params[b].rule_id == SDCP_RULE_SPECULATIVE_SAMPLING;
    pre[(size_t)b + 1] = pre[(size_t)b] + M + 1 + (rule2 ? M : 0);
  }
  const int64_t total = pre[(size_t)B];
  bounds[0] = 0;
  int32_t cut = 0;
  for (int32_t k = 1; k < n_parts; ++k) {
    // target k * total / n_parts, compared as k * total vs pre * n_parts (exact in int64)
    const int64_t goal = (int64_t)k * total;
    int32_t best = cut;
    int64_t best_d = INT64_MAX;
    for (int32_t b = cut; b <= B; ++b) {
      const int64_t d = pre[(size_t)b] * n_parts - goal;
      const int64_t ad = d < 0 ? -d : d;
      if (ad < best_d) { best_d = ad; best = b; }
      if (d >= 0) break;  // the prefix only grows from here
    }
    cut = best;
    bounds[k] = cut;
  }
  bounds[n_parts] = B;
  return SDCP_OK;
}

}  // extern "C"
