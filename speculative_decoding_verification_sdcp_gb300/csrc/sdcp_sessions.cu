// sdcp_sessions.cu - phase 2 of the acceptance step (SDCP draft
// draft-li-mlc-inference-acceleration-00, Section 6.3 "Preconditions of the rule" and
// Section 6.4 Rules 1 and 2): one CTA per session runs the completion of sdcp_session.cuh
// on the row statistics phase 1 left in the workspace.  Launched as a programmatic
// dependent of the row kernel, it waits for the row statistics before reading them.
#include "sdcp_session.cuh"

namespace sdcp {

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) session_kernel(SessIO A) {
  __shared__ SessSmem sm;
  const Group g{kThreads, 1};
  pdl_wait_primary();  // the row statistics and the error word are complete from here on
  complete_session<T>(A, g, sm, (int32_t)blockIdx.x);
}

template __global__ void session_kernel<float>(SessIO);
template __global__ void session_kernel<__nv_bfloat16>(SessIO);

int launch_sessions(const SessIO& a, int dtype, bool pdl, cudaStream_t stream) {
  if (a.B <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.B, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (dtype == SDCP_BF16)
    e = cudaLaunchKernelEx(&cfg, session_kernel<__nv_bfloat16>, a);
  else
    e = cudaLaunchKernelEx(&cfg, session_kernel<float>, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace sdcp
