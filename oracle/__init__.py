"""CPU oracle of the SDCP verifier's acceptance step (test infrastructure).

The oracle is the plain fp64 C program in ``sdcp_oracle.c`` (see its header for the
definitions it follows: the sampling profile of SDCP Section 4.1, the precondition of
Section 6.3 and Rules 1 and 2 of Section 6.4 of the SDCP draft
draft-li-mlc-inference-acceleration-00).  This module only builds it with gcc and
marshals numpy arrays into it.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and
its ``--impl reference`` arm) may import this package.  It shares no code with the CUDA
path and imports nothing from it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "sdcp_oracle.c"), os.path.join(_HERE, "sdcp_oracle_commit.c")]
_LIB_PATH = os.path.join(_HERE, "libsdcp_oracle.so")

F32, BF16 = 0, 1
S_OK, S_BAD_PROPOSAL, S_LIMIT, S_BAD_PARAMS, S_Q_UNAVAILABLE = 0, 1, 2, 3, 4
MMAX = 64

# Same 32-byte layout as one session's parameters in the C ABI (rule, temperature x1000,
# top_k, top_p x1000, seed, round, session tag).
PARAMS_DTYPE = np.dtype([("rule_id", "<u4"), ("temperature_milli", "<u4"), ("top_k", "<u4"),
                         ("top_p_milli", "<u4"), ("seed", "<u8"), ("round", "<u4"),
                         ("session_tag", "<u4")])


class RowInfo(ctypes.Structure):
    _fields_ = [("lmax", ctypes.c_double), ("log_s", ctypes.c_double),
                ("argmax", ctypes.c_int32), ("kept", ctypes.c_int32), ("k1", ctypes.c_int32),
                ("invalid", ctypes.c_int32), ("topp_cum_before", ctypes.c_double),
                ("topp_cum_at", ctypes.c_double), ("topp_target", ctypes.c_double)]


DETAIL_DTYPE = np.dtype([
    ("status", "<i4"), ("a", "<i4"), ("n_out", "<i4"), ("extra_mode", "<i4"),
    ("extra_token", "<i4"), ("extra_pos", "<i4"), ("m", "<i4"), ("pad", "<i4"),
    ("u1", "<f8"), ("W", "<f8"), ("c_lo", "<f8"), ("c_hi", "<f8"),
    ("u0", "<f8", (MMAX,)), ("ratio", "<f8", (MMAX,)), ("log_p", "<f8", (MMAX,)),
    ("log_q", "<f8", (MMAX,)), ("topp_margin", "<f8")])

EXTRA_ARGMAX, EXTRA_RESIDUAL, EXTRA_BONUS, EXTRA_RESIDUAL_AS_P, EXTRA_FROM_P = 1, 2, 3, 4, 5
RULE_GREEDY, RULE_SPECULATIVE_SAMPLING, RULE_RELAXED_TOP_K = 1, 2, 192

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, OpenMP, -O2, no -ffast-math) in place; return its path."""
    newest = max(os.path.getmtime(f) for f in _SRCS)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp] + _SRCS + ["-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64
        L.oracle_philox4x32_10.argtypes = [vp, vp, vp]
        L.oracle_philox4x32_10.restype = None
        L.oracle_uniform.argtypes = [u64, u32, u32, u32, u32]
        L.oracle_uniform.restype = ctypes.c_double
        L.oracle_row_dist.argtypes = [vp, ctypes.c_int, i64, u32, u32, u32, vp, vp, ctypes.POINTER(RowInfo)]
        L.oracle_row_dist.restype = ctypes.c_int
        L.oracle_draw_cdf.argtypes = [vp, vp, i64, vp]
        L.oracle_draw_cdf.restype = ctypes.c_double
        L.oracle_draw.argtypes = [vp, vp, i64, ctypes.c_double]
        L.oracle_draw.restype = ctypes.c_int32
        L.oracle_verify_batch.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp,
                                          vp, vp, vp, vp, vp, ctypes.c_int]
        L.oracle_verify_batch.restype = ctypes.c_int
        L.oracle_row_stats_batch.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, vp,
                                             vp, ctypes.c_int]
        L.oracle_row_stats_batch.restype = ctypes.c_int
        L.oracle_set_topp_shift.argtypes = [ctypes.c_double]
        L.oracle_set_topp_shift.restype = None
        L.oracle_verify_batch_rng.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp,
                                              vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
        L.oracle_row_dist_forced.argtypes = [vp, ctypes.c_int, i64, u32, u32, u32, vp, vp,
                                             ctypes.POINTER(RowInfo), i64]
        L.oracle_row_dist_forced.restype = ctypes.c_int
        L.oracle_verify_batch_rng.restype = ctypes.c_int
        L.oracle_sha256.argtypes = [vp, ctypes.c_size_t, vp]
        L.oracle_sha256.restype = None
        L.oracle_hmac_sha256.argtypes = [vp, ctypes.c_size_t, vp, ctypes.c_size_t, vp]
        L.oracle_hmac_sha256.restype = None
        L.oracle_hmac_uniform.argtypes = [u64, vp, u32, u32, u32]
        L.oracle_hmac_uniform.restype = ctypes.c_double
        L.oracle_contract_digest.argtypes = [vp, ctypes.c_size_t, vp]
        L.oracle_contract_digest.restype = None
        L.oracle_prefix_digest.argtypes = [vp, vp, u32, vp]
        L.oracle_prefix_digest.restype = None
        L.oracle_digest_extend.argtypes = [vp, vp, i32, vp]
        L.oracle_digest_extend.restype = None
        L.oracle_commit_round.argtypes = [vp, vp, vp, i32, i32, vp, vp, u32]
        L.oracle_commit_round.restype = i32
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(arr: np.ndarray) -> int:
    """float32 arrays are binary32 logits; uint16 arrays hold raw bfloat16 bits."""
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("logits must be float32 or uint16 (raw bfloat16 bits), got %s" % arr.dtype)


def philox4x32_10(counter, key):
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, round_: int, position: int, purpose: int, tag: int) -> float:
    return lib().oracle_uniform(seed, round_, position, purpose, tag)


def row_dist(row: np.ndarray, temperature_milli: int = 1000, top_k: int = 0,
             top_p_milli: int = 1000, want_dist: bool = True, want_kept: bool = False,
             force_kept: int = -1):
    """The sampling profile of SDCP Section 4.1 on one row.  Returns (dist, kept, info, rc).
    force_kept >= 1 places the top-p crossing at that many tokens (parity-test hook)."""
    row = np.ascontiguousarray(row)
    V = row.shape[0]
    dist = np.zeros(V, dtype=np.float64) if want_dist else None
    kept = np.zeros(V, dtype=np.uint8) if want_kept else None
    info = RowInfo()
    rc = lib().oracle_row_dist_forced(_ptr(row), _dtype_code(row), V, temperature_milli, top_k,
                                      top_p_milli, _ptr(dist), _ptr(kept), ctypes.byref(info),
                                      int(force_kept))
    return dist, kept, info, rc


def draw_cdf(p: np.ndarray, q: np.ndarray | None = None):
    """Cumulative weights of a draw, ids ascending (residual max(0,p-q) if q is given)."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = None if q is None else np.ascontiguousarray(q, dtype=np.float64)
    C = np.zeros_like(p)
    W = lib().oracle_draw_cdf(_ptr(p), _ptr(q), p.shape[0], _ptr(C))
    return C, W


def draw(p: np.ndarray, q: np.ndarray | None, u: float) -> int:
    """Inverse-CDF draw of the additional token for one uniform u."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = None if q is None else np.ascontiguousarray(q, dtype=np.float64)
    return int(lib().oracle_draw(_ptr(p), _ptr(q), p.shape[0], float(u)))


def verify_batch(target: np.ndarray, draft: np.ndarray | None, m_offsets: np.ndarray,
                 draft_tokens: np.ndarray, params: np.ndarray, nthreads: int = 1,
                 want_detail: bool = True, session_ids: np.ndarray | None = None,
                 force_kept: np.ndarray | None = None, q_rows: np.ndarray | None = None):
    """Rules 1 and 2 of SDCP Section 6.4 over a ragged batch (layout of the C ABI).

    target: [total_drafts + B, V], draft: [total_drafts, V] or None (float32 or raw bf16
    bits as uint16).  session_ids ([B, 16] uint8) selects the draft's HMAC-SHA-256 random
    values (Section 6.4) instead of Philox.  force_kept ([2 total + B] int32, row order of
    the C ABI's row statistics, -1 = as defined) places top-p crossings (a parity-test
    hook).  q_rows ([total, V] float32) gives q as rows of probabilities (SDCP Section 5.2)
    instead of the draft logits.  Returns a dict of numpy arrays (accepted, n_out,
    out_tokens, status, detail).
    """
    target = np.ascontiguousarray(target)
    dcode = _dtype_code(target)
    if draft is not None:
        draft = np.ascontiguousarray(draft)
        if draft.dtype != target.dtype:
            raise TypeError("target and draft logits must share a dtype")
    m_offsets = np.ascontiguousarray(m_offsets, dtype=np.int32)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    params = np.ascontiguousarray(params, dtype=PARAMS_DTYPE)
    B = params.shape[0]
    V = target.shape[1]
    total = int(draft_tokens.shape[0])
    acc = np.zeros(B, np.int32)
    nout = np.zeros(B, np.int32)
    toks = np.full(total + B, -1, np.int32)
    st = np.zeros(B, np.int32)
    det = np.zeros(B, DETAIL_DTYPE) if want_detail else None
    sid = None
    if session_ids is not None:
        sid = np.ascontiguousarray(session_ids, dtype=np.uint8).reshape(B, 16)
    fk = None
    if force_kept is not None:
        fk = np.ascontiguousarray(force_kept, dtype=np.int32)
        assert fk.shape == (2 * total + B,)
    qr = None
    if q_rows is not None:
        qr = np.ascontiguousarray(q_rows, dtype=np.float32)
        assert qr.shape == (total, V)
    rc = lib().oracle_verify_batch_rng(_ptr(target), _ptr(draft), dcode, V, B, _ptr(m_offsets),
                                       total, _ptr(draft_tokens), _ptr(params), _ptr(sid), _ptr(fk),
                                       _ptr(qr), _ptr(acc), _ptr(nout), _ptr(toks), _ptr(st), _ptr(det),
                                       int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify_batch rejected its arguments (rc=%d)" % rc)
    return {"accepted": acc, "n_out": nout, "out_tokens": toks, "status": st, "detail": det}


ROW_INFO_DTYPE = np.dtype([("lmax", "<f8"), ("log_s", "<f8"), ("argmax", "<i4"), ("kept", "<i4"),
                           ("k1", "<i4"), ("invalid", "<i4"), ("topp_cum_before", "<f8"),
                           ("topp_cum_at", "<f8"), ("topp_target", "<f8")])
assert ROW_INFO_DTYPE.itemsize == ctypes.sizeof(RowInfo)


def row_stats_batch(target: np.ndarray, draft: np.ndarray, m_offsets: np.ndarray,
                    draft_tokens: np.ndarray, params: np.ndarray, nthreads: int = 1):
    """The sampling profile (SDCP Section 4.1) of every scored row of a ragged batch, in the
    row order of the C ABI's row-statistics call (target rows, then draft rows).

    Returns (info [R] ROW_INFO_DTYPE, lpx [R] float64, skipped [R] bool)."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    dcode = _dtype_code(target)
    m_offsets = np.ascontiguousarray(m_offsets, dtype=np.int32)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    params = np.ascontiguousarray(params, dtype=PARAMS_DTYPE)
    B = params.shape[0]
    total = int(draft_tokens.shape[0])
    R = 2 * total + B
    info = np.zeros(R, ROW_INFO_DTYPE)
    lpx = np.zeros(R, np.float64)
    skipped = np.zeros(R, np.int32)
    rc = lib().oracle_row_stats_batch(_ptr(target), _ptr(draft), dcode, target.shape[1], B,
                                      _ptr(m_offsets), total, _ptr(draft_tokens), _ptr(params),
                                      _ptr(info), _ptr(lpx), _ptr(skipped), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_row_stats_batch rejected its arguments (rc=%d)" % rc)
    return info, lpx, skipped.astype(bool)


class topp_shift:
    """Context manager: the oracle's top-p target times (1 + rel) inside the block (the two
    readings of a top-p crossing that lies within rounding of P)."""

    def __init__(self, rel: float):
        self.rel = float(rel)

    def __enter__(self):
        lib().oracle_set_topp_shift(self.rel)
        return self

    def __exit__(self, *exc):
        lib().oracle_set_topp_shift(0.0)
        return False


# ---------------------------------------------------------------------------------------
# SHA-256, HMAC, digests, truncation and control (sdcp_oracle_commit.c)
# ---------------------------------------------------------------------------------------
ACT_CONTINUE, ACT_REDUCE, ACT_SWITCH, ACT_SELF_DECODE, ACT_FINISH, ACT_FAIL = 0, 1, 2, 3, 4, 5

# contract terms of one session and the verifier's per-session state (layouts of
# orc_commit_params and orc_session_state)
COMMIT_PARAMS_DTYPE = np.dtype([("max_new", "<u4"), ("stop_offset", "<u4"), ("stop_count", "<u4"),
                                ("m_max", "<u4"), ("low_rounds", "<u4"), ("low_ratio", "<u4"),
                                ("self_load", "<u4"), ("fallback_len", "<u4"), ("fallback", "u1", (8,)),
                                ("m_restore", "<u4"), ("pad", "<u4")])
STATE_DTYPE = np.dtype([("digest", "u1", (32,)), ("committed", "<u4"), ("c", "<u4"), ("g", "<u4"),
                        ("j", "<u4"), ("m_cap", "<u4"), ("pad", "<u4", (3,))])


def _bytes_in(b: bytes):
    a = np.frombuffer(bytes(b), dtype=np.uint8).copy()
    return a, (a.ctypes.data_as(ctypes.c_void_p) if a.size else None)


def sha256(msg: bytes) -> bytes:
    a, p = _bytes_in(msg)
    out = np.zeros(32, np.uint8)
    lib().oracle_sha256(p, len(msg), _ptr(out))
    return out.tobytes()


def hmac_sha256(key: bytes, msg: bytes) -> bytes:
    k, kp = _bytes_in(key)
    m, mp = _bytes_in(msg)
    out = np.zeros(32, np.uint8)
    lib().oracle_hmac_sha256(kp, len(key), mp, len(msg), _ptr(out))
    return out.tobytes()


def hmac_uniform(seed: int, session: bytes, round_: int, i: int, purpose: int) -> float:
    s, sp = _bytes_in(session)
    assert len(session) == 16
    return lib().oracle_hmac_uniform(seed, sp, round_, i, purpose)


def contract_digest(cbor: bytes) -> bytes:
    c, cp = _bytes_in(cbor)
    out = np.zeros(32, np.uint8)
    lib().oracle_contract_digest(cp, len(cbor), _ptr(out))
    return out.tobytes()


def prefix_digest(contract_dig: bytes, prompt) -> bytes:
    c, cp = _bytes_in(contract_dig)
    t = np.ascontiguousarray(np.asarray(prompt, dtype=np.uint32))
    out = np.zeros(32, np.uint8)
    lib().oracle_prefix_digest(cp, _ptr(t) if t.size else None, len(t), _ptr(out))
    return out.tobytes()


def digest_extend(d: bytes, tokens) -> bytes:
    c, cp = _bytes_in(d)
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    out = np.zeros(32, np.uint8)
    lib().oracle_digest_extend(cp, _ptr(t) if t.size else None, len(t), _ptr(out))
    return out.tobytes()


def commit_round(cparams: np.ndarray, stop_tokens, state: np.ndarray, a: int, M: int,
                 emitted, load: int = 0):
    """One session's round after acceptance (SDCP Sections 6.3 and 6.5): truncation, commit,
    control.  state ([1] STATE_DTYPE) is updated in place; returns (action, emitted)."""
    cp = np.ascontiguousarray(cparams, dtype=COMMIT_PARAMS_DTYPE).reshape(1)
    st = np.asarray([0] if stop_tokens is None or len(stop_tokens) == 0 else stop_tokens, dtype=np.uint32)
    st = np.ascontiguousarray(st)
    toks = np.ascontiguousarray(np.asarray(emitted, dtype=np.int32)).copy()
    n = np.asarray([len(toks)], np.int32)
    assert state.dtype == STATE_DTYPE and state.flags["C_CONTIGUOUS"]
    act = lib().oracle_commit_round(_ptr(cp), _ptr(st), _ptr(state), int(a), int(M), _ptr(n),
                                    _ptr(toks) if toks.size else None, int(load))
    return int(act), [int(v) for v in toks[:int(n[0])]]


def max_threads() -> int:
    return lib().oracle_max_threads()
