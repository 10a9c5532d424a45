"""Pins of the oracle's digests, random derivation, truncation and control (no GPU needed).

Each test checks the oracle against something fixed outside it:
  * SHA-256 and HMAC-SHA-256 against Python's hashlib and hmac (library routines);
  * the SDCP draft's Appendix A vectors: the contract digest of the 143-octet sample
    contract and the committed-prefix digests d[0], d[1], d[2] (Sections 4.1, 4.2);
  * the random values of Section 6.4 (last paragraph) rebuilt here from the text with
    hmac and struct: key, message layout, and the first 53 bits;
  * the Appendix A worked round after acceptance (not low, action continue, n = 5);
  * truncation after the first stop token and at max_new (Section 6.3, "Acceptance");
  * the low-round counters and fallback ladder (Section 6.5.2), traced by hand from the
    text.
"""
import hashlib
import hmac
import json
import struct

import numpy as np
import pytest

from conftest import golden_path


@pytest.mark.parametrize("n", [0, 1, 3, 32, 36, 55, 56, 57, 63, 64, 65, 100, 119, 120, 128, 1000])
def test_sha256_matches_library(oracle_mod, n):
    msg = bytes((7 * i + 3) & 0xFF for i in range(n))
    assert oracle_mod.sha256(msg) == hashlib.sha256(msg).digest()


@pytest.mark.parametrize("klen", [0, 8, 32, 63, 64, 65, 100])
@pytest.mark.parametrize("mlen", [0, 39, 100])
def test_hmac_sha256_matches_library(oracle_mod, klen, mlen):
    key = bytes((11 * i + 1) & 0xFF for i in range(klen))
    msg = bytes((5 * i + 2) & 0xFF for i in range(mlen))
    assert oracle_mod.hmac_sha256(key, msg) == hmac.new(key, msg, hashlib.sha256).digest()


def test_appendix_a_contract_and_prefix_digests(oracle_mod):
    fx = json.load(open(golden_path("appendix_a_digests.json")))
    cbor = bytes.fromhex(fx["contract_cbor_hex"])
    assert len(cbor) == fx["contract_cbor_octets"] == 143
    cd = oracle_mod.contract_digest(cbor)
    assert cd.hex() == fx["contract_digest"]
    d0 = oracle_mod.prefix_digest(cd, fx["prompt"])
    assert d0.hex() == fx["d"][0]
    d1 = oracle_mod.digest_extend(d0, fx["outputs"][:1])
    assert d1.hex() == fx["d"][1]
    d2 = oracle_mod.digest_extend(d1, fx["outputs"][1:])
    assert d2.hex() == fx["d"][2]
    assert oracle_mod.digest_extend(d0, fx["outputs"]).hex() == fx["d"][2]
    assert oracle_mod.digest_extend(d0, []) == d0


def _hmac_u(seed, session, round_, i, purpose):
    msg = b"SDCP-VERIFY-1" + b"\x00" + session + struct.pack(">IIB", round_, i, purpose)
    mac = hmac.new(struct.pack(">Q", seed), msg, hashlib.sha256).digest()
    return (int.from_bytes(mac[:8], "big") >> 11) / float(2 ** 53)


def test_hmac_uniform_is_the_drafts_derivation(oracle_mod):
    rng = np.random.default_rng(5)
    for _ in range(50):
        seed = int(rng.integers(0, 2 ** 63)) * 2 + int(rng.integers(0, 2))
        session = bytes(rng.integers(0, 256, size=16, dtype=np.uint8))
        r, i, p = int(rng.integers(0, 2 ** 32)), int(rng.integers(0, 66)), int(rng.integers(0, 2))
        assert oracle_mod.hmac_uniform(seed, session, r, i, p) == _hmac_u(seed, session, r, i, p)


def test_hmac_uniform_range_and_uniformity(oracle_mod):
    sid = bytes(range(16))
    u = np.array([oracle_mod.hmac_uniform(99, sid, 7, i, i & 1) for i in range(20000)])
    assert (u >= 0).all() and (u < 1).all()
    h, _ = np.histogram(u, bins=32, range=(0, 1))
    e = len(u) / 32
    assert ((h - e) ** 2 / e).sum() < 70  # 31 dof, p ~ 1e-4


def test_verify_with_hmac_uses_one_based_positions(oracle_mod):
    """Under the HMAC derivation, the acceptance test of 0-based position k uses i = k + 1
    and the additional token after a accepted tokens uses i = a + 1 (the pages number the
    positions 1 .. M+1)."""
    rng = np.random.default_rng(9)
    B, V, M = 6, 50, 5
    off = np.arange(B + 1, dtype=np.int32) * M
    T = rng.normal(0, 2, size=(B * M + B, V)).astype(np.float32)
    D = (T[np.arange(B * M) + np.repeat(np.arange(B), M)] + rng.normal(0, 1, size=(B * M, V))).astype(np.float32)
    x = rng.integers(0, V, size=B * M).astype(np.int32)
    prm = np.zeros(B, dtype=oracle_mod.PARAMS_DTYPE)
    prm["rule_id"] = 2
    prm["temperature_milli"] = 1000
    prm["top_p_milli"] = 1000
    prm["seed"] = np.arange(B) * 7919 + 3
    prm["round"] = 4
    sids = rng.integers(0, 256, size=(B, 16), dtype=np.uint8)
    r = oracle_mod.verify_batch(T, D, off, x, prm, session_ids=sids)
    det = r["detail"]
    for b in range(B):
        a = int(r["accepted"][b])
        sid = sids[b].tobytes()
        for k in range(a + (1 if a < M else 0)):
            assert det["u0"][b][k] == _hmac_u(int(prm["seed"][b]), sid, 4, k + 1, 0)
        assert det["u1"][b] == _hmac_u(int(prm["seed"][b]), sid, 4, a + 1, 1)
    # and the two generators give different streams
    r2 = oracle_mod.verify_batch(T, D, off, x, prm)
    assert not np.array_equal(r["detail"]["u1"], r2["detail"]["u1"])


# ---------------------------------------------------------------------------------------
# truncation, commit and control
# ---------------------------------------------------------------------------------------
def _contract(oracle_mod, max_new=256, stop=(2,), m_max=8, R=3, low_ratio=0, self_load=255,
              fallback=(1, 2, 3, 5), m_restore=0):
    cp = np.zeros(1, dtype=oracle_mod.COMMIT_PARAMS_DTYPE)
    cp["max_new"] = max_new
    cp["stop_offset"] = 0
    cp["stop_count"] = len(stop)
    cp["m_max"] = m_max
    cp["low_rounds"] = R
    cp["low_ratio"] = low_ratio
    cp["self_load"] = self_load
    cp["fallback_len"] = len(fallback)
    cp["fallback"][0, :len(fallback)] = fallback
    cp["m_restore"] = m_restore
    return cp, list(stop)


def _state(oracle_mod, committed=0, m_cap=8, digest=b"\x00" * 32):
    st = np.zeros(1, dtype=oracle_mod.STATE_DTYPE)
    st["committed"] = committed
    st["m_cap"] = m_cap
    st["digest"][0] = np.frombuffer(digest, np.uint8)
    return st


def test_appendix_a_worked_round_after_acceptance(oracle_mod):
    """Committed n = 2, proposal [7, 9, 11], a = 2, emitted [7, 9, 13]: the new committed
    length is 5, the round is not low, c is reset and the action is continue."""
    fx = json.load(open(golden_path("appendix_a_greedy_round.json")))
    cp, stop = _contract(oracle_mod)
    d = bytes(range(32))
    st = _state(oracle_mod, committed=fx["committed_before"], digest=d)
    st["c"] = 2
    act, em = oracle_mod.commit_round(cp, stop, st, fx["expected_accepted"], len(fx["proposal"]),
                                      fx["expected_emitted"])
    assert act == oracle_mod.ACT_CONTINUE
    assert em == fx["expected_emitted"]
    assert int(st["committed"][0]) == fx["expected_committed_after"]
    assert int(st["c"][0]) == 0 and int(st["g"][0]) == 1
    assert st["digest"][0].tobytes() == oracle_mod.digest_extend(d, fx["expected_emitted"])


@pytest.mark.parametrize("emitted,committed,max_new,stop,expect,finish", [
    ([5, 2, 9], 0, 256, [2], [5, 2], True),        # truncated after the first stop token
    ([2, 7], 10, 256, [2], [2], True),             # a stop token first
    ([5, 6, 7], 0, 256, [2, 3], [5, 6, 7], False),  # no stop token, room enough
    ([5, 6, 7], 254, 256, [2], [5, 6], True),       # at max_new
    ([5, 6, 7], 253, 256, [2], [5, 6, 7], True),    # exactly reaches max_new
    ([5, 6, 7], 256, 256, [2], [], True),           # nothing left to emit
    ([5, 3, 2], 254, 256, [2, 3], [5, 3], True),    # both cuts agree
    ([5, 6, 7], 0, 256, [], [5, 6, 7], False),      # no stop tokens in the contract
])
def test_truncation(oracle_mod, emitted, committed, max_new, stop, expect, finish):
    cp, _ = _contract(oracle_mod, max_new=max_new, stop=stop)
    st = _state(oracle_mod, committed=committed)
    act, em = oracle_mod.commit_round(cp, stop, st, len(emitted) - 1, len(emitted) - 1 or 1, emitted)
    assert em == expect
    assert int(st["committed"][0]) == committed + len(expect)
    assert (act == oracle_mod.ACT_FINISH) == finish
    assert st["digest"][0].tobytes() == oracle_mod.digest_extend(b"\x00" * 32, expect)


def _run(oracle_mod, cp, stop, st, rounds, load=0):
    """rounds: list of (a, M); returns the actions and the m_cap after each round."""
    acts, caps = [], []
    for a, M in rounds:
        act, _ = oracle_mod.commit_round(cp, stop, st, a, M, [7] * (a + 1), load)
        acts.append(act)
        caps.append(int(st["m_cap"][0]))
    return acts, caps


def test_escalation_ladder(oracle_mod):
    """R = 3, fallback [reduce, switch, self_decode, fail], low_ratio absent (low iff a = 0).
    Every third consecutive low round applies the next entry; self_decode is skipped without
    self_load; when no entry remains the action is fail."""
    C, R_, S, SD, F, FI = (oracle_mod.ACT_CONTINUE, oracle_mod.ACT_REDUCE, oracle_mod.ACT_SWITCH,
                           oracle_mod.ACT_SELF_DECODE, oracle_mod.ACT_FAIL, oracle_mod.ACT_FINISH)
    cp, stop = _contract(oracle_mod, max_new=10 ** 6, stop=[])
    st = _state(oracle_mod, m_cap=8)
    acts, caps = _run(oracle_mod, cp, stop, st, [(0, 4)] * 12)
    assert acts == [C, C, R_, C, C, S, C, C, F, C, C, F]
    assert caps == [8, 8, 4, 4, 4, 4, 4, 4, 4, 4, 4, 4]
    assert int(st["j"][0]) == 4 and int(st["c"][0]) == 0
    # self_load present and the load within it: self_decode is applied
    st = _state(oracle_mod, m_cap=8)
    cp2, _ = _contract(oracle_mod, max_new=10 ** 6, stop=[], self_load=50)
    acts, _ = _run(oracle_mod, cp2, stop, st, [(0, 4)] * 12, load=30)
    assert acts == [C, C, R_, C, C, S, C, C, SD, C, C, F]
    # load above self_load: skipped again
    st = _state(oracle_mod, m_cap=8)
    acts, _ = _run(oracle_mod, cp2, stop, st, [(0, 4)] * 9, load=80)
    assert acts == [C, C, R_, C, C, S, C, C, F]


def test_counters_reset(oracle_mod):
    """A round that is not low resets c; R rounds that are not low in a row reset j."""
    C, R_, S = oracle_mod.ACT_CONTINUE, oracle_mod.ACT_REDUCE, oracle_mod.ACT_SWITCH
    cp, stop = _contract(oracle_mod, max_new=10 ** 6, stop=[])
    st = _state(oracle_mod, m_cap=8)
    seq = [(0, 4), (0, 4), (1, 4), (0, 4), (0, 4), (0, 4)]  # the not-low round breaks the run
    acts, caps = _run(oracle_mod, cp, stop, st, seq)
    assert acts == [C, C, C, C, C, R_]
    assert int(st["j"][0]) == 1
    # two rounds that are not low: j stays; the third (g = R) resets j to zero
    acts, _ = _run(oracle_mod, cp, stop, st, [(2, 4), (2, 4)])
    assert int(st["j"][0]) == 1 and int(st["g"][0]) == 2
    acts, _ = _run(oracle_mod, cp, stop, st, [(2, 4)])
    assert int(st["j"][0]) == 0
    acts, caps = _run(oracle_mod, cp, stop, st, [(0, 4)] * 3)
    assert acts == [C, C, R_] and caps[-1] == 2  # 4 -> 2: reduce applied again from entry 0


def test_low_ratio_and_restore(oracle_mod):
    """low_ratio 50: a round is low iff 100 a < 50 M.  m_cap halves (floor, at least 1) on
    reduce and grows by m_restore, up to m_max, after rounds that are not low."""
    C, R_ = oracle_mod.ACT_CONTINUE, oracle_mod.ACT_REDUCE
    cp, stop = _contract(oracle_mod, max_new=10 ** 6, stop=[], low_ratio=50, R=1, fallback=(1,),
                         m_restore=1, m_max=8)
    st = _state(oracle_mod, m_cap=3)
    acts, caps = _run(oracle_mod, cp, stop, st, [(1, 4)])   # 100 < 200: low, R = 1 -> reduce
    assert acts == [R_] and caps == [1]
    acts, caps = _run(oracle_mod, cp, stop, st, [(2, 4)])   # 200 < 200 is false: not low
    assert acts == [C] and caps == [2]
    acts, caps = _run(oracle_mod, cp, stop, st, [(4, 4)] * 8)
    assert caps == [3, 4, 5, 6, 7, 8, 8, 8]
    # the rounds that were not low reset j (g reached R = 1): entry 0 applies again; the
    # ladder has one entry, so the escalation right after it finds none and fails
    acts, caps = _run(oracle_mod, cp, stop, st, [(0, 4), (0, 4)])
    assert acts == [R_, oracle_mod.ACT_FAIL] and caps == [4, 4]


def test_finish_takes_precedence(oracle_mod):
    cp, stop = _contract(oracle_mod, max_new=10 ** 6, stop=[2], R=1, fallback=(1,))
    st = _state(oracle_mod, m_cap=8)
    act, em = oracle_mod.commit_round(cp, stop, st, 0, 4, [2])
    assert act == oracle_mod.ACT_FINISH and em == [2]
    assert int(st["m_cap"][0]) == 8  # no ladder entry applied
