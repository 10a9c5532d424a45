// sdcp_sessions.cu - phase 2 of the acceptance step (SDCP draft
// draft-li-mlc-inference-acceleration-00, Section 6.3 "Preconditions of the rule" and
// Section 6.4 Rules 1 and 2): one thread-block cluster per session runs the completion of
// sdcp_session.cuh on the row statistics phase 1 left in the workspace.  Launched as a
// programmatic dependent of the row kernel, it waits for the row statistics before
// reading them.
#include <mutex>

#include "sdcp_session.cuh"

namespace sdcp {

constexpr size_t kRingBytes = (size_t)kDrawStages * 2 * kDrawHalf;

// QR: q given as rows of binary32 probabilities (a separate instantiation, so that the
// usual kernel keeps its own register allocation).
template <typename T, bool QR>
__global__ void __launch_bounds__(kThreads, 2) session_kernel(SessIO A) {
  extern __shared__ __align__(128) unsigned char ring[];  // the streamed draw's stages
  __shared__ SessSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const Group g{kThreads, 1};
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDrawStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], kWarps); }
    sm.ring_uses = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_primary();  // the row statistics and the error word are complete from here on
  complete_session<T, QR>(A, cluster, g, sm, ring, (int32_t)(blockIdx.x / cluster.num_blocks()));
}

template __global__ void session_kernel<float, false>(SessIO);
template __global__ void session_kernel<__nv_bfloat16, false>(SessIO);
template __global__ void session_kernel<float, true>(SessIO);
template __global__ void session_kernel<__nv_bfloat16, true>(SessIO);

// CTAs per session: as many as fit two CTAs per SM over the whole batch (a draw is a
// latency-bound chain, so small batches gain from splitting it), never slices under 16
// segments (4096 ids) of a row; 1 .. 8.
static int session_cluster(int sms, int64_t V, int32_t B) {
  int64_t c = (2 * (int64_t)sms) / (B > 0 ? B : 1);
  const int64_t by_size = V / 4096;
  if (c > by_size) c = by_size;
  return (int)(c < 1 ? 1 : (c > 8 ? 8 : c));
}

namespace {
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
cudaError_t g_err[kMaxDevices];

// Once per device: the session kernels' shared-memory attributes (the draw ring as dynamic
// shared memory, and all of the unified L1/shared storage as shared memory, so two CTAs fit
// on an SM).
cudaError_t session_attributes(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_once[dev], [&] {
    cudaError_t e = cudaSuccess;
    const void* fns[4] = {(const void*)session_kernel<__nv_bfloat16, false>, (const void*)session_kernel<float, false>,
                          (const void*)session_kernel<__nv_bfloat16, true>, (const void*)session_kernel<float, true>};
    for (const void* fn : fns) {
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingBytes);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    }
    g_err[dev] = e;
  });
  return g_err[dev];
}
}  // namespace

int launch_sessions(const SessIO& a, int dtype, bool pdl, cudaStream_t stream) {
  if (a.B <= 0) return 0;
  DeviceInfo di;
  int dev = 0;
  if (!device_info(&di) || cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
  cudaError_t e = session_attributes(dev);
  if (e != cudaSuccess) return (int)e;
  const int C = session_cluster(di.sms, a.V, a.B);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.B * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kRingBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const bool qr = a.q_rows != nullptr;
  if (dtype == SDCP_BF16)
    e = qr ? cudaLaunchKernelEx(&cfg, session_kernel<__nv_bfloat16, true>, a)
           : cudaLaunchKernelEx(&cfg, session_kernel<__nv_bfloat16, false>, a);
  else
    e = qr ? cudaLaunchKernelEx(&cfg, session_kernel<float, true>, a)
           : cudaLaunchKernelEx(&cfg, session_kernel<float, false>, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp
