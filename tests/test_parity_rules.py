"""The comparison rules of the parity tests, checked on CPU with the oracle's own outputs
(mistakes are planted in a copy of those outputs, never in a GPU run).

A differing draw is accepted only where the GPU's token has positive weight and u * W lies
within 1e-5 * W of that token's cumulative interval (so whatever lies between the two
tokens weighs less than 1e-5 * W); a differing greedy session, or a draw far from u * W,
must fail.
"""
import numpy as np
import pytest

import parity


def _cdf(weights):
    C = np.cumsum(np.asarray(weights, dtype=np.float64))
    return C, float(C[-1])


def test_draw_boundary_accepts_tokens_within_the_window():
    C, W = _cdf([0.2, 0.0, 0.3, 0.5])
    # edge between token 0 and token 2 (token 1 has no weight) is at 0.2
    u = 0.2 / W
    parity._check_draw_boundary(C, W, u + 3e-6, 0, 2, 0)
    parity._check_draw_boundary(C, W, u - 3e-6, 2, 0, 0)
    # tokens of negligible weight between the two: still within the boundary window
    C, W = _cdf([0.2, 1e-12, 2e-12, 0.3, 0.5])
    parity._check_draw_boundary(C, W, (0.2 - 3e-6) / W, 3, 0, 0)


@pytest.mark.parametrize("tg,to,u", [
    (0, 2, 0.25),     # far from the shared edge
    (3, 0, 0.19),     # token 2's weight lies between them
    (1, 2, 0.2),      # the GPU token has no weight
    (3, 2, 0.3),      # u*W inside token 2, far from token 3
])
def test_draw_boundary_rejects(tg, to, u):
    C, W = _cdf([0.2, 0.0, 0.3, 0.5])
    with pytest.raises(AssertionError):
        parity._check_draw_boundary(C, W, u, tg, to, 0)


def _batch(oracle_mod, rule):
    rng = np.random.default_rng(4)
    B, V, M = 8, 40, 3
    off = np.arange(B + 1, dtype=np.int32) * M
    T = rng.normal(0, 2, size=(B * M + B, V)).astype(np.float32)
    D = (T[np.arange(B * M) + np.repeat(np.arange(B), M)] + rng.normal(0, 1, size=(B * M, V))).astype(np.float32)
    x = rng.integers(0, V, size=B * M).astype(np.int32)
    prm = np.zeros(B, dtype=oracle_mod.PARAMS_DTYPE)
    prm["rule_id"] = rule
    prm["temperature_milli"] = 1000
    prm["top_p_milli"] = 1000
    prm["seed"] = np.arange(B) + 1
    prm["round"] = 1
    prm["session_tag"] = np.arange(B)
    ref = oracle_mod.verify_batch(T, D, off, x, prm)
    return T, D, off, x, prm, ref


def _outputs(ref):
    return {k: ref[k].copy() for k in ("accepted", "n_out", "out_tokens", "status")}


def test_identical_outputs_pass(oracle_mod):
    T, D, off, x, prm, ref = _batch(oracle_mod, 2)
    c = parity.compare_verdicts(_outputs(ref), ref, T, D, off, x, prm)
    assert c["exact"] == len(prm)


def test_planted_far_token_fails(oracle_mod):
    T, D, off, x, prm, ref = _batch(oracle_mod, 2)
    got = _outputs(ref)
    b = 0
    a = int(ref["accepted"][b])
    slot = int(off[b]) + b + a
    V = T.shape[1]
    # a token of positive weight far from u * W: the last token with weight, or the first
    C, W = parity._draw_cdf(T, D, off, b, a, prm[b], ref["detail"]["extra_mode"][b])
    pos = np.nonzero(np.diff(np.concatenate([[0.0], C])) > 0)[0]
    tok = int(ref["out_tokens"][slot])
    far = int(pos[-1]) if abs(int(pos[-1]) - tok) > 1 else int(pos[0])
    assert far != tok
    got["out_tokens"][slot] = far
    with pytest.raises(AssertionError):
        parity.compare_verdicts(got, ref, T, D, off, x, prm)


def test_planted_greedy_difference_fails(oracle_mod):
    T, D, off, x, prm, ref = _batch(oracle_mod, 1)
    got = _outputs(ref)
    slot = int(off[2]) + 2 + int(ref["accepted"][2])
    got["out_tokens"][slot] = (got["out_tokens"][slot] + 1) % T.shape[1]
    with pytest.raises(AssertionError, match="greedy"):
        parity.compare_verdicts(got, ref, T, D, off, x, prm)


def test_planted_acceptance_far_from_boundary_fails(oracle_mod):
    T, D, off, x, prm, ref = _batch(oracle_mod, 2)
    got = _outputs(ref)
    det = ref["detail"]
    for b in range(len(prm)):
        a = int(ref["accepted"][b])
        M = int(off[b + 1] - off[b])
        if a < M and abs(det["u0"][b][a] - det["ratio"][b][a]) > 1e-3:
            # claim one more accepted token than the oracle
            o0 = int(off[b])
            got["accepted"][b] = a + 1
            got["n_out"][b] = a + 2
            got["out_tokens"][o0 + b + a] = x[o0 + a]
            if a + 1 <= M:
                got["out_tokens"][o0 + b + a + 1] = 0
            break
    else:
        pytest.skip("no rejection far from its boundary in this batch")
    with pytest.raises(AssertionError, match="acceptance"):
        parity.compare_verdicts(got, ref, T, D, off, x, prm)
