"""GPU parity of the draft's own random derivation and of the commit step.

* sdcp_verify_batch_ex with the HMAC-SHA-256 generator (SDCP draft Section 6.4, last
  paragraph) against the oracle with the same session identifiers, under the parity rules of
  tests/parity.py.
* sdcp_commit_batch (Section 6.3 truncation and commit, Section 4.2 digest chain, Section 6.5
  control) against the oracle's commit of the same verify outputs, bit for bit (tokens,
  counts, state bytes, actions), over two rounds in a row; and the Appendix A vectors on the
  GPU: the worked greedy round (n 2 -> 5, continue) and the digests d[1], d[2].
"""
import json

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from conftest import golden_path  # noqa: E402
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


def _session_ids(B, seed):
    return np.random.default_rng(seed).integers(0, 256, size=(B, 16), dtype=np.uint8)


HMAC_CASES = [
    dict(B=12, V=1000, dtype=synth.F32, m=4, rules="alternate", temperature_milli=1000),
    dict(B=16, V=32000, dtype=synth.BF16, m=8, rules="spec", temperature_milli=700, top_k=50, sigma=3.0, noise=1.0),
    dict(B=16, V=50257, dtype=synth.BF16, m=("uniform", 1, 16), rules="spec", temperature_milli=800,
         top_p_milli=900, sigma=3.0, noise=0.8),
    dict(B=8, V=65536, dtype=synth.F32, m=("uniform", 1, 64), rules="spec", temperature_milli=1000,
         sigma=4.0, noise=0.5, draft_scale=1.5),
]


@pytest.mark.parametrize("ci", range(len(HMAC_CASES)))
def test_hmac_generator_parity(ci):
    import oracle
    import parity
    from speculative_decoding_verification_sdcp_gb300.sdcp import RNG_HMAC_SHA256, Verifier
    w = synth.custom_workload(seed_base=900 + ci, gen_seed=300 + ci, **HMAC_CASES[ci])
    batch = synth.make_batch(w, device=DEV)
    sids = _session_ids(batch.B, ci)
    ver = Verifier(batch.V, batch.B, batch.total_drafts, DEV)
    out = ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens, batch.params_dev,
              rng_id=RNG_HMAC_SHA256, session_ids=torch.from_numpy(sids).to(DEV))
    torch.cuda.synchronize()
    got = {k: t.cpu().numpy() for k, t in zip(("accepted", "n_out", "out_tokens", "status"), out)}
    T, D, off, x = parity.host_arrays(batch)
    ref = oracle.verify_batch(T, D, off, x, batch.params, nthreads=parity.ORACLE_THREADS, session_ids=sids)
    gs = parity.gpu_row_stats(batch)
    counts = parity.compare_verdicts(got, ref, T, D, off, x, batch.params, gs=gs, session_ids=sids)
    parity.check_invariants(got, off, x, batch.params, batch.V)
    parity.report("hmac_%d" % ci, counts)
    assert counts["exact"] >= batch.B - 2, counts
    # a different generator gives different draws somewhere
    philox = parity.run_gpu(batch)
    assert not all(np.array_equal(philox[k], got[k]) for k in got)


def _contracts(B, rng, V):
    import oracle
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    assert oracle.COMMIT_PARAMS_DTYPE.itemsize == sdcp.COMMIT_PARAMS_DTYPE.itemsize
    cp = np.zeros(B, dtype=oracle.COMMIT_PARAMS_DTYPE)
    stops = []
    for b in range(B):
        ns = int(rng.integers(0, 4))
        cp["stop_offset"][b] = len(stops)
        cp["stop_count"][b] = ns
        stops.extend(int(v) for v in rng.integers(0, V, size=ns))
        cp["max_new"][b] = int(rng.integers(1, 40))
        cp["m_max"][b] = 64
        cp["low_rounds"][b] = int(rng.integers(1, 4))
        cp["low_ratio"][b] = int(rng.choice([0, 0, 25, 50, 100]))
        cp["self_load"][b] = int(rng.choice([0xFFFFFFFF, 30, 90]))
        fl = int(rng.integers(1, 5))
        cp["fallback_len"][b] = fl
        cp["fallback"][b, :fl] = rng.choice([1, 2, 3, 5], size=fl)
        cp["m_restore"][b] = int(rng.integers(0, 3))
    return cp, np.asarray(stops if stops else [0], np.uint32)


def _states(B, rng):
    import oracle
    st = np.zeros(B, dtype=oracle.STATE_DTYPE)
    st["digest"] = rng.integers(0, 256, size=(B, 32), dtype=np.uint8)
    st["committed"] = rng.integers(0, 40, size=B)
    st["c"] = rng.integers(0, 3, size=B)
    st["g"] = rng.integers(0, 3, size=B)
    st["j"] = rng.integers(0, 3, size=B)
    st["m_cap"] = rng.integers(1, 65, size=B)
    return st


def _to_dev(arr):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).copy()).to(DEV)


def test_commit_matches_oracle_two_rounds():
    import oracle
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    rng = np.random.default_rng(17)
    w = synth.custom_workload(B=96, V=300, dtype=synth.BF16, m=("uniform", 1, 12), rules="alternate",
                              temperature_milli=(0, 700, 1000), top_k=60, sigma=2.0, noise=0.3, gen_seed=41,
                              seed_base=70)
    batch = synth.make_batch(w, device=DEV)
    B, V = batch.B, batch.V
    cp, stops = _contracts(B, rng, V)
    st = _states(B, rng)
    # one status that is not OK: nothing is committed for it
    x = batch.draft_tokens.cpu().numpy()
    off = batch.m_offsets.cpu().numpy()
    x[off[5]] = V + 1
    batch.draft_tokens.copy_(torch.from_numpy(x))
    cp_dev, stop_dev, st_dev = _to_dev(cp), torch.from_numpy(stops.view(np.int32)).to(DEV), _to_dev(st)
    ver = sdcp.Verifier(V, B, batch.total_drafts, DEV)
    action = torch.empty(B, dtype=torch.int32, device=DEV)
    for rnd in range(2):
        batch.params["round"] += 1
        batch.params_dev = synth.params_to_device(batch.params, DEV)
        acc, nout, toks, status = ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens,
                                      batch.params_dev)
        torch.cuda.synchronize()
        pre = {k: t.cpu().numpy().copy() for k, t in zip(("accepted", "n_out", "out_tokens", "status"),
                                                          (acc, nout, toks, status))}
        load = 40 + 30 * rnd
        sdcp.sdcp_commit_batch(batch.m_offsets, acc, nout, toks, status, cp_dev, stop_dev, st_dev, load, action)
        torch.cuda.synchronize()
        g_n, g_t = nout.cpu().numpy(), toks.cpu().numpy()
        g_st = st_dev.cpu().numpy().view(st.dtype)
        g_act = action.cpu().numpy()
        for b in range(B):
            o0, M = int(off[b]), int(off[b + 1] - off[b])
            sl = slice(o0 + b, o0 + b + M + 1)
            if pre["status"][b] != 0:
                assert g_act[b] == sdcp.ACTION_NONE
                assert g_st[b].tobytes() == st[b].tobytes() and g_n[b] == pre["n_out"][b]
                continue
            s1 = st[b:b + 1].copy()
            act, em = oracle.commit_round(cp[b], stops, s1, int(pre["accepted"][b]), M,
                                          pre["out_tokens"][o0 + b:o0 + b + pre["n_out"][b]], load)
            assert g_act[b] == act, (b, g_act[b], act)
            assert g_n[b] == len(em), (b, g_n[b], em)
            assert list(g_t[sl][:len(em)]) == em and (g_t[sl][len(em):] == -1).all(), b
            assert g_st[b].tobytes() == s1[0].tobytes(), (b, g_st[b], s1[0])
            st[b] = s1[0]
        assert (g_act == sdcp.ACTION_FINISH).any() and (g_act == sdcp.ACTION_CONTINUE).any()


def _greedy_batch(rows_argmax, proposal, V=64):
    """One greedy session whose target rows have the given argmax tokens."""
    M = len(proposal)
    T = torch.zeros(M + 1, V, dtype=torch.float32)
    for i, tok in enumerate(rows_argmax):
        T[i, tok] = 5.0
    prm = np.zeros(1, dtype=synth.PARAMS_DTYPE)
    prm["rule_id"] = 1
    prm["temperature_milli"] = 1000
    prm["top_p_milli"] = 1000
    w = synth.custom_workload(B=1, V=V)
    return synth.Batch(w, T.to(DEV), torch.zeros(M, V, device=DEV),
                       torch.tensor([0, M], dtype=torch.int32, device=DEV),
                       torch.tensor(proposal, dtype=torch.int32, device=DEV), prm,
                       synth.params_to_device(prm, DEV))


def _commit_one(batch, cp, st, stops=(2,)):
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    ver = sdcp.Verifier(batch.V, 1, batch.total_drafts, DEV)
    acc, nout, toks, status = ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens,
                                  batch.params_dev)
    st_dev = _to_dev(st)
    action = torch.empty(1, dtype=torch.int32, device=DEV)
    sdcp.sdcp_commit_batch(batch.m_offsets, acc, nout, toks, status, _to_dev(cp),
                           torch.tensor(list(stops), dtype=torch.int32, device=DEV), st_dev, 0, action)
    torch.cuda.synchronize()
    n = int(nout.item())
    return int(acc.item()), toks.cpu().numpy()[:n].tolist(), st_dev.cpu().numpy().view(st.dtype)[0], int(action.item())


def _appendix_contract():
    rng = np.random.default_rng(0)
    cp, _ = _contracts(1, rng, 64)
    cp["max_new"] = 256
    cp["stop_offset"] = 0
    cp["stop_count"] = 1
    cp["m_max"] = 8
    cp["low_rounds"] = 3
    cp["low_ratio"] = 0
    cp["self_load"] = 0xFFFFFFFF
    cp["fallback_len"] = 4
    cp["fallback"][0, :4] = [1, 2, 3, 5]
    cp["m_restore"] = 0
    return cp


def test_appendix_a_worked_round_on_gpu():
    fx = json.load(open(golden_path("appendix_a_greedy_round.json")))
    batch = _greedy_batch(fx["target_argmax_per_position"], fx["proposal"])
    st = _states(1, np.random.default_rng(1))
    st["committed"] = fx["committed_before"]
    st["c"] = 2
    a, em, s2, act = _commit_one(batch, _appendix_contract(), st)
    assert a == fx["expected_accepted"] and em == fx["expected_emitted"]
    assert int(s2["committed"]) == fx["expected_committed_after"]
    assert act == 0 and int(s2["c"]) == 0  # not low: c reset, continue


def test_appendix_a_digest_chain_on_gpu():
    """From d[0] of the prompt [1, 2, 3, 4], committing 17 then 42 gives the draft's d[2]
    (and committing 17 alone its d[1])."""
    fx = json.load(open(golden_path("appendix_a_digests.json")))
    st = _states(1, np.random.default_rng(2))
    st["digest"][0] = np.frombuffer(bytes.fromhex(fx["d"][0]), np.uint8)
    st["committed"] = 0
    batch = _greedy_batch([17, 42], [17])
    a, em, s2, act = _commit_one(batch, _appendix_contract(), st)
    assert em == [17, 42]
    assert s2["digest"].tobytes().hex() == fx["d"][2]
    assert int(s2["committed"]) == 2
    batch = _greedy_batch([17, 3], [5])  # rejected at once: emits 17 alone
    a, em, s1, act = _commit_one(batch, _appendix_contract(), st)
    assert em == [17] and s1["digest"].tobytes().hex() == fx["d"][1]
