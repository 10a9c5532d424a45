"""GPU path (libsdcp through its C ABI) against the CPU oracle, element by element.

Every batch is compared whole with the oracle: every session's outputs and every row's
statistics, including the four large workloads of the benchmark at full size in the
benchmark's launch configuration.  Boundary cases (decisions within 1e-5 of their
boundary) are counted per case and printed; with SDCP_PARITY_REPORT set they are also
appended to that file.
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


def _parity(batch, rows=True, with_draft=True, name=None):
    import oracle
    import parity
    got = parity.run_gpu(batch, with_draft=with_draft)
    T, D, off, x = parity.host_arrays(batch)
    ref = oracle.verify_batch(T, D if with_draft else None, off, x, batch.params,
                              nthreads=parity.ORACLE_THREADS)
    gs = parity.gpu_row_stats(batch) if rows else None
    counts = parity.compare_verdicts(got, ref, T, D, off, x, batch.params, gs=gs)
    parity.check_invariants(got, off, x, batch.params, batch.V)
    if rows:
        counts["rows"] = parity.compare_row_stats(gs, T, D, off, x, batch.params, batch.dtype_code)
    if name is not None:
        parity.report(name, counts)
    return got, counts


@pytest.mark.parametrize("name", ["tiny", "tiny_greedy"])
def test_tiny_workloads(name):
    batch = synth.make_batch(synth.WORKLOADS[name], device=DEV)
    _, counts = _parity(batch)
    assert counts["exact"] == batch.B, counts


CASES = [
    # dtype, V, M, rules, T, top_k, top_p, sigma, noise
    (synth.F32, 1, 3, "spec", 1000, 0, 1000, 1.0, 0.5),
    (synth.F32, 7, 5, "alternate", 1000, 0, 1000, 1.0, 0.5),
    (synth.BF16, 7, 5, "alternate", 700, 3, 1000, 1.0, 0.5),
    (synth.F32, 64, ("uniform", 1, 12), "spec", 600, 0, 900, 2.0, 1.0),
    (synth.BF16, 1000, ("uniform", 1, 64), "alternate", 1000, 0, 1000, 2.0, 0.5),
    (synth.BF16, 4099, 6, "spec", 800, 50, 1000, 3.0, 1.0),       # ragged rows (unaligned)
    (synth.BF16, 4099, 6, "spec", 800, 0, 900, 3.0, 1.0),
    (synth.BF16, 4099, 6, "spec", 1300, 40, 700, 3.0, 1.0),
    (synth.F32, 4099, 6, "spec", 800, 50, 900, 3.0, 1.0),          # fp32 filters: generic search
    (synth.BF16, 32000, 8, "spec", 700, 50, 1000, 3.0, 1.0),
    (synth.BF16, 32000, 4, "spec", 0, 0, 1000, 3.0, 1.0),          # temperature 0 under Rule 2
    (synth.BF16, 50257, ("uniform", 1, 9), "spec", 1000, 1, 1000, 3.0, 1.0),
    (synth.F32, 50257, 3, "alternate", 1700, 0, 1000, 3.0, 1.0),
    (synth.BF16, 65536, 3, "spec", 900, 0, 1, 3.0, 1.0),           # top-p keeps only the argmax
    (synth.BF16, 65536, 3, "spec", 900, 0, 999, 3.0, 1.0),
    (synth.BF16, 32000, 6, "spec", 800, 1000, 1000, 3.0, 1.0),     # top-k above 256: 8-nat window
    (synth.BF16, 32000, 6, "spec", 800, 256, 950, 3.0, 1.0),       # top-k bound at k = 256, top-p
    (synth.F32, 32000, 6, "spec", 800, 0, 900, 3.0, 1.0),          # fp32 top-p: generic search
    (synth.F32, 50257, 4, "spec", 700, 40, 950, 3.0, 1.0),         # fp32 top-k + top-p
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "dt%d-V%d-T%d-k%d-p%d-%s" % (c[0], c[1], c[4], c[5], c[6], c[3]))
def test_small_matrix(case):
    dt, V, m, rules, T, k, p, sigma, noise = case
    w = synth.custom_workload(B=12, V=V, dtype=dt, m=m, rules=rules, temperature_milli=T, top_k=k,
                              top_p_milli=p, sigma=sigma, noise=noise, seed_base=77,
                              gen_seed=100 + CASES.index(case))
    batch = synth.make_batch(w, device=DEV)
    _, counts = _parity(batch, name="small_%d" % CASES.index(case))
    assert counts["exact"] >= batch.B - 2, counts


@pytest.mark.parametrize("top_p", [1000, 900])
def test_long_slice_global_draw(top_p):
    """160 sessions of one draft token over V = 600000: one CTA per session, a slice of
    2344 segments (more than the 2048 segment sums a CTA holds), so the draw runs from
    global memory with grouped segments (no cut on p), or with the cut-value lists
    (a top-p cut inside a bf16 value)."""
    w = synth.custom_workload(B=160, V=600000, dtype=synth.BF16, m=1, rules="spec",
                              temperature_milli=900, top_p_milli=top_p, sigma=3.0, noise=1.0,
                              seed_base=60, gen_seed=61 + top_p)
    batch = synth.make_batch(w, device=DEV)
    _, counts = _parity(batch, name="long_slice_p%d" % top_p)
    assert counts["exact"] >= batch.B - 3, counts


def test_ties_and_tie_overflow():
    """Integer logits (many equal values) and a cut value shared by ~30000 tokens."""
    B, V, M = 6, 32000, 3
    w = synth.custom_workload(B=B, V=V, dtype=synth.BF16, m=M, rules="spec", temperature_milli=1000,
                              top_k=100, top_p_milli=950, gen_seed=5)
    batch = synth.make_batch(w, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(3)
    t = torch.randint(-3, 4, batch.target.shape, generator=g, device=DEV).float()
    t[:3] = 0.0
    t[:3, :5] = 2.0
    batch.target.copy_(t.to(torch.bfloat16))
    batch.draft.copy_(batch.target[: batch.total_drafts].clone())
    _parity(batch)


@pytest.mark.parametrize("top_k,top_p", [(50, 1000), (0, 900), (200, 950)])
def test_cut_value_ties_in_both_rows(top_k, top_p):
    """Logits on a 0.5 grid: the cut of p and the cut of q both fall inside a value shared
    by tens of tokens, so the residual draw must rank the tokens of both cut values (the
    single-pass draw); the drafter samples its tokens from the quantised q."""
    B, V, M = 10, 32000, 4
    w = synth.custom_workload(B=B, V=V, dtype=synth.BF16, m=M, rules="spec", temperature_milli=800,
                              top_k=top_k, top_p_milli=top_p, gen_seed=21)
    batch = synth.make_batch(w, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    t = torch.round(torch.randn(batch.target.shape, generator=g, device=DEV) * 6.0) / 2.0
    d = torch.round((t[: batch.total_drafts] + torch.randn(batch.draft.shape, generator=g, device=DEV))
                    * 2.0) / 2.0
    batch.target.copy_(t.to(torch.bfloat16))
    batch.draft.copy_(d.to(torch.bfloat16))
    batch.draft_tokens.copy_(synth.drafter_sample(batch.draft, 800, top_k, top_p, g))
    got, counts = _parity(batch)
    assert (got["status"] == 0).all(), got["status"]
    assert counts["exact"] >= B - 2, counts


def test_flat_distribution_window_fallback():
    """Logits within +-0.05 straddle zero: the nucleus spans many binades below the max
    and the window cannot hold it, so the generic search decides."""
    w = synth.custom_workload(B=4, V=8192, dtype=synth.BF16, m=3, rules="spec", temperature_milli=1000,
                              top_p_milli=900, sigma=0.02, noise=0.01, gen_seed=9)
    batch = synth.make_batch(w, device=DEV)
    _, counts = _parity(batch)
    assert counts["rows"]["fallback"] > 0


def test_statuses_and_degenerate_rows():
    import oracle
    import parity
    B, V, M = 9, 40, 2
    w = synth.custom_workload(B=B, V=V, dtype=synth.F32, m=M, rules="spec", gen_seed=11)
    batch = synth.make_batch(w, device=DEV)
    off = batch.m_offsets.cpu().numpy()
    prm = batch.params.copy()
    prm["rule_id"][0] = 0
    prm["rule_id"][1] = 3
    prm["top_p_milli"][2] = 1001
    x = batch.draft_tokens.cpu().numpy().copy()
    x[off[3]] = V                                   # token out of range
    prm["top_k"][4] = 1                             # q(x) = 0 unless x is the draft argmax
    dargs = batch.draft.cpu().numpy()
    x[off[4] + 1] = (int(np.argmax(dargs[off[4] + 1])) + 1) % V
    batch.draft[off[5], int(x[off[5]])] = -float("inf")   # q(x) = 0 through -inf
    batch.target[off[6] + 6 + 1, 3] = float("nan")         # NaN in a scored row
    batch.target[off[7] + 7 + 2, :] = -float("inf")        # a row without a finite logit
    batch.draft_tokens.copy_(torch.from_numpy(x))
    batch.params = prm
    batch.params_dev = synth.params_to_device(prm, DEV)
    got, _ = _parity(batch, rows=False)
    S = oracle
    assert list(got["status"]) == [S.S_BAD_PARAMS, S.S_BAD_PARAMS, S.S_BAD_PARAMS, S.S_BAD_PROPOSAL,
                                   S.S_BAD_PROPOSAL, S.S_BAD_PROPOSAL, S.S_BAD_PARAMS,
                                   S.S_BAD_PARAMS, S.S_OK]
    # Rule 2 without draft logits, and greedy sessions without them
    got2 = parity.run_gpu(batch, with_draft=False)
    ref2 = oracle.verify_batch(*parity.host_arrays(batch)[:1], None, off, x, prm)
    assert np.array_equal(got2["status"], ref2["status"])


def test_limits_on_m():
    import oracle
    import parity
    V = 16
    Ms = [0, 65, 64, 1]
    off = np.zeros(len(Ms) + 1, np.int32)
    off[1:] = np.cumsum(Ms)
    tot = int(off[-1])
    g = torch.Generator(device=DEV).manual_seed(1)
    T = torch.randn(tot + len(Ms), V, generator=g, device=DEV)
    D = torch.randn(tot, V, generator=g, device=DEV)
    x = torch.randint(0, V, (tot,), generator=g, device=DEV, dtype=torch.int32)
    prm = np.zeros(len(Ms), dtype=synth.PARAMS_DTYPE)
    prm["rule_id"] = 1
    prm["temperature_milli"] = 1000
    prm["top_p_milli"] = 1000
    w = synth.custom_workload(B=len(Ms), V=V)
    batch = synth.Batch(w, T, D, torch.from_numpy(off).to(DEV), x, prm, synth.params_to_device(prm, DEV))
    got = parity.run_gpu(batch)
    ref = oracle.verify_batch(T.cpu().numpy(), D.cpu().numpy(), off, x.cpu().numpy(), prm)
    for k in ("status", "accepted", "n_out", "out_tokens"):
        assert np.array_equal(got[k], ref[k]), k
    assert list(got["status"][:2]) == [oracle.S_LIMIT, oracle.S_LIMIT]


def test_empty_batch():
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    z = torch.empty(0, dtype=torch.int32, device=DEV)
    t = torch.empty(0, 8, dtype=torch.float32, device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    sdcp.sdcp_verify_batch(t, t, torch.zeros(1, dtype=torch.int32, device=DEV), 0, z,
                           torch.empty(0, dtype=torch.uint8, device=DEV), z, z, z, z, ws)


def test_reproducible_bit_for_bit():
    import parity
    batch = synth.make_batch(synth.custom_workload(B=16, V=32000, dtype=synth.BF16, m=("uniform", 1, 16),
                                                   rules="spec", temperature_milli=800, top_p_milli=900,
                                                   sigma=3.0, noise=0.8, gen_seed=4), device=DEV)
    a = parity.run_gpu(batch)
    b = parity.run_gpu(batch)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_large_vocabulary():
    batch = synth.make_batch(synth.custom_workload(B=3, V=1 << 20, dtype=synth.BF16, m=2, rules="spec",
                                                   temperature_milli=1000, top_k=1000, sigma=3.0,
                                                   noise=1.0, gen_seed=6), device=DEV)
    _parity(batch)


@pytest.mark.parametrize("name", ["topk50", "topp90_ragged", "large_batch_mixed", "mmax_stress"])
def test_full_size_workloads(name):
    """The whole batch on the GPU in the benchmark's call, compared whole with the oracle:
    every session's outputs and every row's statistics."""
    batch = synth.make_batch(synth.WORKLOADS[name], device=DEV)
    got, counts = _parity(batch, name=name)
    assert (got["status"] == 0).all(), np.unique(got["status"], return_counts=True)
    assert counts["rows"]["fallback"] == 0, counts


@pytest.mark.parametrize("name", ["topk50", "large_batch_mixed"])
def test_two_phase_path(name):
    """sdcp_verify_rows then sdcp_verify_sessions (the separate completion kernel, thread-block
    clusters and streamed draws) against the oracle, like the one-call path above."""
    import oracle
    import parity
    from speculative_decoding_verification_sdcp_gb300.sdcp import Verifier
    batch = synth.make_batch(synth.WORKLOADS[name], device=DEV)
    ver = Verifier(batch.V, batch.B, batch.total_drafts, DEV)
    out = ver.phases(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens, batch.params_dev)
    torch.cuda.synchronize()
    got = {k: t.cpu().numpy() for k, t in zip(("accepted", "n_out", "out_tokens", "status"), out)}
    T, D, off, x = parity.host_arrays(batch)
    ref = oracle.verify_batch(T, D, off, x, batch.params, nthreads=parity.ORACLE_THREADS)
    gs = parity.gpu_row_stats(batch)
    counts = parity.compare_verdicts(got, ref, T, D, off, x, batch.params, gs=gs)
    parity.check_invariants(got, off, x, batch.params, batch.V)
    parity.report("two_phase_" + name, counts)
    assert counts["exact"] >= batch.B - 2, counts


RELAXED = [
    # dtype, V, M, T, top_k, top_p
    (synth.BF16, 32000, 6, 700, 50, 1000),
    (synth.F32, 4099, ("uniform", 1, 9), 1000, 3, 900),
    (synth.BF16, 50257, 4, 0, 0, 1000),        # temperature 0: the greedy rule
    (synth.BF16, 32000, 5, 800, 0, 900),       # the kept set of a top-p cut
    (synth.BF16, 65536, 3, 900, 1, 1000),      # top-1: the greedy rule again
]


@pytest.mark.parametrize("case", RELAXED, ids=lambda c: "dt%d-V%d-T%d-k%d-p%d" % (c[0], c[1], c[3], c[4], c[5]))
def test_relaxed_rule(case):
    """The private-use relaxed rule (id 192): accept while x is in p's kept set, then a draw
    from p; it reads no draft rows, so the call also runs without draft logits."""
    import oracle
    import parity
    dt, V, m, T, k, p = case
    w = synth.custom_workload(B=16, V=V, dtype=dt, m=m, rules="relaxed", temperature_milli=T, top_k=k,
                              top_p_milli=p, sigma=3.0, noise=1.0, seed_base=321,
                              gen_seed=500 + RELAXED.index(case))
    batch = synth.make_batch(w, device=DEV)
    got, counts = _parity(batch, name="relaxed_%d" % RELAXED.index(case))
    assert (got["status"] == 0).all()
    assert counts["exact"] >= batch.B - 2, counts
    got2 = parity.run_gpu(batch, with_draft=False)
    for key in got:
        assert np.array_equal(got[key], got2[key]), key
