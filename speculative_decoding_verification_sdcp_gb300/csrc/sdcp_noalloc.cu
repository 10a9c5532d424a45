// sdcp_noalloc.cu - sdcp_verify_batch_noalloc: the verify call for callers that may not
// allocate device memory.  Its scratch is a file-scope __device__ array owned by the
// library (held by every GPU that loads it, until exit); the caller passes only inputs,
// outputs and a stream.
#include <mutex>

#include "sdcp_device.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SDCP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the array on the current device, looked up once per device.  In host
// code the array's name is only a stand-in, never a device address, so it must go
// through cudaGetSymbolAddress.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDCP_E_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return SDCP_E_DEVICE;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SDCP_OK;
}

}  // namespace

extern "C" int sdcp_verify_batch_noalloc(const void* target_logits, const void* draft_logits,
                                         int dtype, int64_t V, int32_t B,
                                         const int32_t* m_offsets, int64_t total_drafts,
                                         const int32_t* draft_tokens,
                                         const sdcp_session_params* params, int32_t* accepted,
                                         int32_t* n_out, int32_t* out_tokens, int32_t* status,
                                         void* stream) {
  int rc = sdcp::check_common(target_logits, dtype, V, B, m_offsets, total_drafts, draft_tokens,
                              params, draft_logits);
  if (rc != SDCP_OK) return rc;
  if (B == 0) return SDCP_OK;
  const size_t need = sdcp_workspace_bytes(V, B, total_drafts);
  if (need == 0) return V > SDCP_MAX_VOCAB ? SDCP_E_TOO_LARGE : SDCP_E_INVALID;
  if (need > SDCP_NOALLOC_SCRATCH_BYTES) return SDCP_E_SCRATCH_LIMIT;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != SDCP_OK) return rc;
  return sdcp_verify_batch(target_logits, draft_logits, dtype, V, B, m_offsets, total_drafts,
                           draft_tokens, params, accepted, n_out, out_tokens, status, scratch,
                           SDCP_NOALLOC_SCRATCH_BYTES, stream);
}
