"""A bounded wait that runs out reports SDCP_S_INTERNAL and leaves the device usable.

Every wait of the kernels (on a ring stage's copy, on a stage's release, on the draw's
copies) gives up after a wall-time limit, sets the call's error word, and the session
kernel then reports SDCP_S_INTERNAL for every session.  This test builds the library once
more with the test-only flag SDCP_TEST_WAIT_EXPIRY: the limit becomes 20 ms and the row
kernel's CTA 0 leaves the ring stage of its first row unfilled (no copy is issued into it, so
nothing is in flight there when the CTA gives up).  The wait of CTA 0's consumers for that
stage then runs out on purpose.  No fault, trap or endless loop is involved: every wait is
bounded, and the test checks afterwards that the ordinary library still verifies a batch
exactly as before on the same device.
Kept in a file of its own that pytest collects last.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def waitlib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_sdcp_gb300 import build_ext
    build_ext.build()
    path = build_ext.build(extra_flags=["-DSDCP_TEST_WAIT_EXPIRY"],
                           lib=os.path.join(build_ext.PKG, "libsdcp_waittest.so"),
                           build_dir=os.path.join(build_ext.BUILD, "waittest"))
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    lib.sdcp_verify_batch.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, vp, vp, vp,
                                      vp, sz, vp]
    lib.sdcp_verify_batch.restype = ctypes.c_int
    return lib


def _batch():
    from speculative_decoding_verification_sdcp_gb300 import synth
    w = synth.custom_workload(B=24, V=32000, dtype=synth.BF16, m=("uniform", 1, 8), rules="alternate",
                              temperature_milli=(700, 1000), top_k=50, sigma=3.0, noise=1.0,
                              seed_base=700, gen_seed=31)
    return synth.make_batch(w, device=DEV)


def test_wait_that_runs_out_reports_internal(waitlib):
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    batch = _batch()
    ver = sdcp.Verifier(batch.V, batch.B, batch.total_drafts, DEV)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    for t in (ver.accepted, ver.n_out, ver.out_tokens, ver.status):
        t.fill_(-7)
    rc = waitlib.sdcp_verify_batch(P(batch.target), P(batch.draft), batch.dtype_code, batch.V, batch.B,
                                   P(batch.m_offsets), batch.total_drafts, P(batch.draft_tokens),
                                   P(batch.params_dev), P(ver.accepted), P(ver.n_out), P(ver.out_tokens),
                                   P(ver.status), P(ver.workspace), ver.workspace.numel(),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0  # SDCP_OK: the launches were accepted
    torch.cuda.synchronize()  # raises if the device had faulted
    status = ver.status.cpu().numpy()
    assert (status == sdcp.S_INTERNAL).all(), status
    # the ordinary library on the same device afterwards: every session verified, and the
    # same outputs as a second call (nothing of the failed call is left behind)
    ref = [t.clone() for t in ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens,
                                  batch.params_dev)]
    again = ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens, batch.params_dev)
    torch.cuda.synchronize()
    assert (ref[3].cpu().numpy() == sdcp.S_OK).all()
    for r, a in zip(ref, again):
        assert np.array_equal(r.cpu().numpy(), a.cpu().numpy())
