"""The verify entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (for example code that runs while someone else is
capturing a CUDA graph, or a host runtime that owns all device allocations).
sdcp_verify_batch_noalloc serves them from a scratch array compiled into the library.  This
test calls it through the C ABI and checks that it returns exactly what sdcp_verify_batch
returns with a caller-owned workspace, on two different batches in a row (the second call
finds the first call's leftovers in the shared array), and that a batch needing more
scratch than the array holds is refused before any launch.
Kept in a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_sdcp_gb300 import build_ext
    build_ext.build()


def _both(batch):
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    ver = sdcp.Verifier(batch.V, batch.B, batch.total_drafts, DEV)
    ref = [t.clone() for t in ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens,
                                  batch.params_dev)]
    out = [torch.full_like(t, -7) for t in ref]
    sdcp.sdcp_verify_batch_noalloc(batch.target, batch.draft, batch.m_offsets, batch.total_drafts,
                                   batch.draft_tokens, batch.params_dev, *out)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in ref], [t.cpu().numpy() for t in out]


def test_noalloc_matches_workspace_entry_point_twice():
    from speculative_decoding_verification_sdcp_gb300 import synth
    w1 = synth.custom_workload(B=24, V=32000, dtype=synth.BF16, m=("uniform", 1, 16), rules="alternate",
                               temperature_milli=(500, 700, 1000), top_k=50, sigma=3.0, noise=1.0,
                               seed_base=500, gen_seed=21)
    w2 = synth.custom_workload(B=9, V=50257, dtype=synth.F32, m=("uniform", 1, 64), rules="spec",
                               temperature_milli=900, top_p_milli=900, sigma=3.0, noise=0.8,
                               seed_base=900, gen_seed=22)
    for w in (w1, w2):
        batch = synth.make_batch(w, device=DEV)
        ref, out = _both(batch)
        for r, o in zip(ref, out):
            assert np.array_equal(r, o)
        assert (ref[3] == 0).all()


def test_noalloc_refuses_batches_beyond_its_scratch():
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    B, V, total = 40000, 8, 40000   # (2 * total + B) * 32 bytes of row statistics = 3.84 MB
    assert sdcp.sdcp_workspace_bytes(V, B, total) > sdcp.NOALLOC_SCRATCH_BYTES
    t = torch.zeros(total + B, V, device=DEV)
    d = torch.zeros(total, V, device=DEV)
    off = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    x = torch.zeros(total, dtype=torch.int32, device=DEV)
    prm = torch.zeros(B * 32, dtype=torch.uint8, device=DEV)
    outs = [torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV),
            torch.empty(total + B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)]
    with pytest.raises(sdcp.SdcpError, match="no-alloc array"):
        sdcp.sdcp_verify_batch_noalloc(t, d, off, total, x, prm, *outs)
