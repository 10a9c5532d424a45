"""GPU parity of the q_rows input form: q given as the drafter's rows of binary32
probabilities (SDCP draft Section 5.2 q_rows; Section 6.4 Rule 2 takes q[i] as the row of
q_rows for position i), used as given, against the oracle's q-rows mode.

The rows are the stand-in drafter's own distributions (the rows it samples its tokens from).
The first phase then reads target rows only.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from speculative_decoding_verification_sdcp_gb300 import synth  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_sdcp_gb300 import build_ext
    build_ext.build()
    import oracle
    oracle.build()


def _q_rows(batch):
    off = batch.m_offsets.cpu().numpy()
    rows = torch.empty(batch.draft.shape, dtype=torch.float32, device=batch.draft.device)
    for b in range(batch.B):
        d0, d1 = int(off[b]), int(off[b + 1])
        pb = batch.params[b]
        rows[d0:d1] = synth.drafter_rows(batch.draft[d0:d1], int(pb["temperature_milli"]), int(pb["top_k"]),
                                         int(pb["top_p_milli"]))
    return rows


def _run(batch, q_rows, with_draft=False):
    from speculative_decoding_verification_sdcp_gb300.sdcp import Verifier
    ver = Verifier(batch.V, batch.B, batch.total_drafts, DEV)
    out = ver(batch.target, batch.draft if with_draft else None, batch.m_offsets, batch.draft_tokens,
              batch.params_dev, q_rows=q_rows)
    torch.cuda.synchronize()
    return {k: t.cpu().numpy() for k, t in zip(("accepted", "n_out", "out_tokens", "status"), out)}


CASES = [
    # dtype, V, M, T, top_k, top_p
    (synth.BF16, 32000, 8, 700, 50, 1000),       # p has a cut: the kept-set draw
    (synth.BF16, 32000, ("uniform", 1, 12), 800, 0, 900),
    (synth.F32, 50257, 4, 1000, 0, 1000),        # no cut: the global-memory draw
    (synth.BF16, 128256, 6, 800, 0, 900),        # long rows, a top-p cut
    (synth.F32, 4099, 5, 0, 0, 1000),            # temperature 0
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "dt%d-V%d-T%d-k%d-p%d" % (c[0], c[1], c[3], c[4], c[5]))
def test_q_rows_parity(case):
    import oracle
    import parity
    dt, V, m, T, k, p = case
    w = synth.custom_workload(B=12, V=V, dtype=dt, m=m, rules="spec", temperature_milli=T, top_k=k,
                              top_p_milli=p, sigma=3.0, noise=1.0, seed_base=650,
                              gen_seed=600 + CASES.index(case))
    batch = synth.make_batch(w, device=DEV)
    q_rows = _q_rows(batch)
    got = _run(batch, q_rows)
    Tn, Dn, off, x = parity.host_arrays(batch)
    qn = q_rows.cpu().numpy()
    ref = oracle.verify_batch(Tn, None, off, x, batch.params, nthreads=parity.ORACLE_THREADS, q_rows=qn)
    gs = parity.gpu_row_stats(batch)
    counts = parity.compare_verdicts(got, ref, Tn, Dn, off, x, batch.params, gs=gs, q_rows=qn)
    parity.check_invariants(got, off, x, batch.params, batch.V)
    parity.report("q_rows_%d" % CASES.index(case), counts)
    assert (got["status"] == 0).all(), got["status"]
    assert counts["exact"] >= batch.B - 2, counts
    # the draft logits, if also given, are not read
    got2 = _run(batch, q_rows, with_draft=True)
    for key in got:
        assert np.array_equal(got[key], got2[key]), key


def test_q_rows_statuses():
    """q(x) = 0 is a bad proposal; NaN, infinite or negative q(x) has no distribution."""
    import oracle
    import parity
    w = synth.custom_workload(B=6, V=64, dtype=synth.F32, m=2, rules="spec", temperature_milli=1000,
                              gen_seed=77)
    batch = synth.make_batch(w, device=DEV)
    q_rows = _q_rows(batch)
    off = batch.m_offsets.cpu().numpy()
    x = batch.draft_tokens.cpu().numpy()
    for b, val in ((1, 0.0), (2, float("nan")), (3, -0.5), (4, float("inf"))):
        q_rows[int(off[b]), int(x[off[b]])] = val
    got = _run(batch, q_rows)
    Tn, Dn, offn, xn = parity.host_arrays(batch)
    ref = oracle.verify_batch(Tn, None, offn, xn, batch.params, q_rows=q_rows.cpu().numpy())
    assert np.array_equal(got["status"], ref["status"]), (got["status"], ref["status"])
    S = oracle
    assert list(got["status"][:5]) == [S.S_OK, S.S_BAD_PROPOSAL, S.S_BAD_PARAMS, S.S_BAD_PARAMS, S.S_BAD_PARAMS]
