"""Seeded random batches: the GPU path against the oracle on many small shapes at once.

Each case draws a vocabulary size (aligned and unaligned rows, from 1 token up), a dtype,
a rule mix, a temperature, top-k and top-p, ragged draft lengths and logit scales from one
fixed seed, and some cases make one session invalid (an unknown rule id or top_p_milli above
1000: its target rows are then copied before the session is known to need nothing, and
handed back unread).  Every batch is compared whole with the oracle under the rules of
tests/parity.py, with the row statistics of every batch without a rejected session.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from speculative_decoding_verification_sdcp_gb300 import synth  # noqa: E402

DEV = "cuda:0"
N_CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_sdcp_gb300 import build_ext
    build_ext.build()
    import oracle
    oracle.build()


def _case(i):
    rng = np.random.default_rng(9000 + i)
    V = int(rng.choice([1, 2, 7, 31, 64, 257, 1000, 4099, 8192, 12345, 32000, 50257]))
    dt = synth.BF16 if rng.random() < 0.6 else synth.F32
    m = int(rng.integers(1, 9)) if rng.random() < 0.5 else ("uniform", 1, int(rng.integers(2, 17)))
    rules = str(rng.choice(["spec", "spec", "alternate", "greedy", "relaxed"]))
    T = int(rng.choice([0, 500, 700, 1000, 1300]))
    k = int(rng.choice([0, 0, 1, 5, 50, 300]))
    p = int(rng.choice([1000, 1000, 999, 950, 900, 500]))
    sigma = float(rng.choice([1.0, 2.0, 3.0, 4.0]))
    noise = float(rng.choice([0.3, 1.0]))
    B = int(rng.integers(1, 25))
    bad = rng.random() < 0.3
    return dict(B=B, V=V, dtype=dt, m=m, rules=rules, temperature_milli=T, top_k=k, top_p_milli=p,
                sigma=sigma, noise=noise, seed_base=300 + 17 * i, gen_seed=4000 + i), bad, int(rng.integers(0, B))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_batch(i):
    import oracle
    import parity
    kw, bad, which = _case(i)
    batch = synth.make_batch(synth.custom_workload(**kw), device=DEV)
    if bad:  # one session with parameters the call rejects
        prm = batch.params.copy()
        if which % 2 == 0:
            prm["rule_id"][which] = 0
        else:
            prm["top_p_milli"][which] = 1001
        batch.params = prm
        batch.params_dev = synth.params_to_device(prm, DEV)
    got = parity.run_gpu(batch)
    T, D, off, x = parity.host_arrays(batch)
    ref = oracle.verify_batch(T, D, off, x, batch.params, nthreads=parity.ORACLE_THREADS)
    gs = parity.gpu_row_stats(batch)
    counts = parity.compare_verdicts(got, ref, T, D, off, x, batch.params, gs=gs)
    parity.check_invariants(got, off, x, batch.params, batch.V)
    if not bad:  # (row statistics of a rejected session are not compared)
        counts["rows"] = parity.compare_row_stats(gs, T, D, off, x, batch.params, batch.dtype_code)
    parity.report("fuzz_%d" % i, counts)
    if bad:
        assert got["status"][which] == oracle.S_BAD_PARAMS
    assert counts["exact"] >= batch.B - 2, counts
