"""Thin Python binding of libsdcp (C ABI in include/sdcp.h): argument marshalling only.

Every step of the acceptance step runs in the library's CUDA kernels; this module turns
torch tensors into pointers, sizes and the current CUDA stream, and raises on a non-zero
return code.  There is no fallback: if libsdcp.so is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsdcp.so")

SDCP_F32, SDCP_BF16 = 0, 1
SDCP_RULE_GREEDY, SDCP_RULE_SPECULATIVE_SAMPLING = 1, 2
S_OK, S_BAD_PROPOSAL, S_LIMIT, S_BAD_PARAMS, S_Q_UNAVAILABLE, S_INTERNAL = 0, 1, 2, 3, 4, 5
ROW_INVALID, ROW_X_KEPT, ROW_SKIPPED, ROW_FALLBACK = 1, 2, 4, 8
MAX_M = 64

# sdcp_session_params (32 bytes) and sdcp_row_stat (32 bytes) as numpy records.
PARAMS_DTYPE = np.dtype([("rule_id", "<u4"), ("temperature_milli", "<u4"), ("top_k", "<u4"),
                         ("top_p_milli", "<u4"), ("seed", "<u8"), ("round", "<u4"),
                         ("session_tag", "<u4")])
ROW_STAT_DTYPE = np.dtype([("lmax", "<f4"), ("log_s", "<f4"), ("lp_x", "<f4"), ("argmax", "<i4"),
                           ("kept", "<i4"), ("thr_key", "<u4"), ("thr_n", "<i4"), ("flags", "<u4")])

# random generators of the acceptance step
RNG_PHILOX4X32_10, RNG_HMAC_SHA256 = 0, 1
# actions of a verdict, and the contract's "no self_load"
ACTION_NONE, ACTION_CONTINUE, ACTION_REDUCE, ACTION_SWITCH = -1, 0, 1, 2
ACTION_SELF_DECODE, ACTION_FINISH, ACTION_FAIL = 3, 4, 5
NO_SELF_LOAD = 0xFFFFFFFF
# sdcp_commit_params (48 bytes) and sdcp_session_state (64 bytes)
COMMIT_PARAMS_DTYPE = np.dtype([("max_new", "<u4"), ("stop_offset", "<u4"), ("stop_count", "<u4"),
                                ("m_max", "<u4"), ("low_rounds", "<u4"), ("low_ratio", "<u4"),
                                ("self_load", "<u4"), ("fallback_len", "<u4"), ("fallback", "u1", (8,)),
                                ("m_restore", "<u4"), ("reserved", "<u4")])
STATE_DTYPE = np.dtype([("digest", "u1", (32,)), ("committed", "<u4"), ("c", "<u4"), ("g", "<u4"),
                        ("j", "<u4"), ("m_cap", "<u4"), ("reserved", "<u4", (3,))])
assert COMMIT_PARAMS_DTYPE.itemsize == 48 and STATE_DTYPE.itemsize == 64


class VerifyOptions(ctypes.Structure):
    """sdcp_verify_options."""
    _fields_ = [("struct_size", ctypes.c_uint32), ("rng_id", ctypes.c_uint32),
                ("session_ids", ctypes.c_void_p), ("q_rows", ctypes.c_void_p)]


class SdcpError(RuntimeError):
    pass


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libsdcp.so is not built; run "
                          "`python -m speculative_decoding_verification_sdcp_gb300.build_ext` "
                          "(or __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    L.sdcp_workspace_bytes.argtypes = [i64, i32, i64]
    L.sdcp_workspace_bytes.restype = sz
    L.sdcp_verify_batch.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, vp, vp,
                                    vp, vp, sz, vp]
    L.sdcp_verify_batch.restype = ctypes.c_int
    L.sdcp_verify_rows.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, sz, vp]
    L.sdcp_verify_rows.restype = ctypes.c_int
    L.sdcp_verify_sessions.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, vp, vp,
                                       vp, vp, sz, vp]
    L.sdcp_verify_sessions.restype = ctypes.c_int
    L.sdcp_verify_batch_noalloc.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp,
                                            vp, vp, vp, vp]
    L.sdcp_verify_batch_noalloc.restype = ctypes.c_int
    L.sdcp_row_stats.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, vp, sz, vp]
    L.sdcp_row_stats.restype = ctypes.c_int
    L.sdcp_verify_batch_ex.argtypes = [vp, vp, ctypes.c_int, i64, i32, vp, i64, vp, vp, vp, vp, vp,
                                       vp, vp, sz, ctypes.POINTER(VerifyOptions), vp]
    L.sdcp_verify_batch_ex.restype = ctypes.c_int
    L.sdcp_commit_batch.argtypes = [i32, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_uint32, vp, vp]
    L.sdcp_commit_batch.restype = ctypes.c_int
    L.sdcp_split_sessions.argtypes = [vp, vp, i32, i32, vp]
    L.sdcp_split_sessions.restype = ctypes.c_int
    L.sdcp_strerror.argtypes = [ctypes.c_int]
    L.sdcp_strerror.restype = ctypes.c_char_p
    L.sdcp_abi_version.argtypes = []
    L.sdcp_abi_version.restype = ctypes.c_int
    return L


lib = _load()


def sdcp_strerror(code: int) -> str:
    return lib.sdcp_strerror(code).decode()


def sdcp_abi_version() -> int:
    return lib.sdcp_abi_version()


def sdcp_workspace_bytes(V: int, B: int, total_drafts: int) -> int:
    return int(lib.sdcp_workspace_bytes(V, B, total_drafts))


def _check(rc: int, what: str):
    if rc != 0:
        raise SdcpError("%s failed: %s (code %d)" % (what, sdcp_strerror(rc), rc))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SDCP_BF16
    if t.dtype == torch.float32:
        return SDCP_F32
    raise TypeError("logits must be torch.float32 or torch.bfloat16, got %s" % t.dtype)


def params_tensor(params: np.ndarray, device) -> torch.Tensor:
    raw = np.ascontiguousarray(params, dtype=PARAMS_DTYPE).view(np.uint8)
    return torch.from_numpy(raw.copy()).to(device)


def alloc_workspace(V: int, B: int, total_drafts: int, device) -> torch.Tensor:
    n = sdcp_workspace_bytes(V, B, total_drafts)
    if n == 0:
        raise SdcpError("invalid sizes for the workspace (V=%d, B=%d, total=%d)" % (V, B, total_drafts))
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(n, dtype=torch.uint8, device=device)


def _stream_handle(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _on(t: torch.Tensor):
    """The library launches on the current CUDA device: make the tensors' device current."""
    return torch.cuda.device(t.device)


def sdcp_verify_batch(target_logits, draft_logits, m_offsets, total_drafts, draft_tokens,
                      params_dev, accepted, n_out, out_tokens, status, workspace,
                      stream=None):
    """Device tensors in, device tensors out; enqueued on ``stream`` (default: current)."""
    V = target_logits.shape[1]
    B = accepted.shape[0]
    s = _stream_handle(target_logits.device) if stream is None else ctypes.c_void_p(stream)
    with _on(target_logits):
        rc = lib.sdcp_verify_batch(_ptr(target_logits), _ptr(draft_logits), dtype_code(target_logits),
                                   V, B, _ptr(m_offsets), int(total_drafts), _ptr(draft_tokens),
                                   _ptr(params_dev), _ptr(accepted), _ptr(n_out), _ptr(out_tokens),
                                   _ptr(status), _ptr(workspace), workspace.numel(), s)
    _check(rc, "sdcp_verify_batch")


def sdcp_verify_batch_ex(target_logits, draft_logits, m_offsets, total_drafts, draft_tokens,
                         params_dev, accepted, n_out, out_tokens, status, workspace,
                         rng_id=RNG_PHILOX4X32_10, session_ids=None, q_rows=None, stream=None):
    """sdcp_verify_batch with the random generator chosen by rng_id (session_ids: a device
    uint8 tensor [B, 16] of session identifiers, for the HMAC-SHA-256 generator), and q from
    the draft logits or from q_rows (a device float32 tensor [total_drafts, V] of the
    drafter's probabilities)."""
    V = target_logits.shape[1]
    B = accepted.shape[0]
    s = _stream_handle(target_logits.device) if stream is None else ctypes.c_void_p(stream)
    if q_rows is not None and q_rows.dtype != torch.float32:
        raise TypeError("q_rows must be torch.float32 probabilities")
    opts = VerifyOptions(ctypes.sizeof(VerifyOptions), int(rng_id),
                         None if session_ids is None else session_ids.data_ptr(),
                         None if q_rows is None else q_rows.data_ptr())
    with _on(target_logits):
        rc = lib.sdcp_verify_batch_ex(_ptr(target_logits), _ptr(draft_logits), dtype_code(target_logits),
                                      V, B, _ptr(m_offsets), int(total_drafts), _ptr(draft_tokens),
                                      _ptr(params_dev), _ptr(accepted), _ptr(n_out), _ptr(out_tokens),
                                      _ptr(status), _ptr(workspace), workspace.numel(),
                                      ctypes.byref(opts), s)
    _check(rc, "sdcp_verify_batch_ex")


def sdcp_commit_batch(m_offsets, accepted, n_out, out_tokens, status, cparams_dev, stop_tokens,
                      state_dev, load_percent, action, stream=None):
    """The commit step after acceptance (truncation, digest chain, control) on device tensors:
    cparams_dev / state_dev are uint8 tensors holding COMMIT_PARAMS_DTYPE / STATE_DTYPE
    records; n_out, out_tokens and state_dev are updated in place."""
    B = accepted.shape[0]
    s = _stream_handle(accepted.device) if stream is None else ctypes.c_void_p(stream)
    with _on(accepted):
        rc = lib.sdcp_commit_batch(B, _ptr(m_offsets), _ptr(accepted), _ptr(n_out), _ptr(out_tokens),
                                   _ptr(status), _ptr(cparams_dev), _ptr(stop_tokens), _ptr(state_dev),
                                   int(load_percent), _ptr(action), s)
    _check(rc, "sdcp_commit_batch")


NOALLOC_SCRATCH_BYTES = 2 << 20


def sdcp_verify_batch_noalloc(target_logits, draft_logits, m_offsets, total_drafts, draft_tokens,
                              params_dev, accepted, n_out, out_tokens, status, stream=None):
    """sdcp_verify_batch without a workspace argument: the library's own scratch array is
    used (for callers that cannot allocate device memory; calls must not overlap)."""
    V = target_logits.shape[1]
    B = accepted.shape[0]
    s = _stream_handle(target_logits.device) if stream is None else ctypes.c_void_p(stream)
    with _on(target_logits):
        rc = lib.sdcp_verify_batch_noalloc(_ptr(target_logits), _ptr(draft_logits),
                                           dtype_code(target_logits), V, B, _ptr(m_offsets),
                                           int(total_drafts), _ptr(draft_tokens), _ptr(params_dev),
                                           _ptr(accepted), _ptr(n_out), _ptr(out_tokens), _ptr(status), s)
    _check(rc, "sdcp_verify_batch_noalloc")


def sdcp_verify_rows(target_logits, draft_logits, m_offsets, total_drafts, draft_tokens,
                     params_dev, workspace, B, stream=None):
    V = target_logits.shape[1]
    s = _stream_handle(target_logits.device) if stream is None else ctypes.c_void_p(stream)
    with _on(target_logits):
        rc = lib.sdcp_verify_rows(_ptr(target_logits), _ptr(draft_logits), dtype_code(target_logits), V,
                                  B, _ptr(m_offsets), int(total_drafts), _ptr(draft_tokens),
                                  _ptr(params_dev), _ptr(workspace), workspace.numel(), s)
    _check(rc, "sdcp_verify_rows")


def sdcp_verify_sessions(target_logits, draft_logits, m_offsets, total_drafts, draft_tokens,
                         params_dev, accepted, n_out, out_tokens, status, workspace, stream=None):
    V = target_logits.shape[1]
    B = accepted.shape[0]
    s = _stream_handle(target_logits.device) if stream is None else ctypes.c_void_p(stream)
    with _on(target_logits):
        rc = lib.sdcp_verify_sessions(_ptr(target_logits), _ptr(draft_logits), dtype_code(target_logits),
                                      V, B, _ptr(m_offsets), int(total_drafts), _ptr(draft_tokens),
                                      _ptr(params_dev), _ptr(accepted), _ptr(n_out), _ptr(out_tokens),
                                      _ptr(status), _ptr(workspace), workspace.numel(), s)
    _check(rc, "sdcp_verify_sessions")


def sdcp_row_stats(target_logits, draft_logits, m_offsets, total_drafts, draft_tokens, params_dev,
                   stats_out, workspace, stream=None):
    V = target_logits.shape[1]
    B = m_offsets.shape[0] - 1
    s = _stream_handle(target_logits.device) if stream is None else ctypes.c_void_p(stream)
    with _on(target_logits):
        rc = lib.sdcp_row_stats(_ptr(target_logits), _ptr(draft_logits), dtype_code(target_logits), V, B,
                                _ptr(m_offsets), int(total_drafts), _ptr(draft_tokens), _ptr(params_dev),
                                _ptr(stats_out), _ptr(workspace), workspace.numel(), s)
    _check(rc, "sdcp_row_stats")


def sdcp_split_sessions(m_offsets: np.ndarray, params: np.ndarray | None, n_parts: int) -> np.ndarray:
    """Contiguous session blocks for n_parts GPUs (host arrays in, [n_parts+1] bounds out)."""
    off = np.ascontiguousarray(m_offsets, dtype=np.int32)
    B = off.shape[0] - 1
    prm = None if params is None else np.ascontiguousarray(params, dtype=PARAMS_DTYPE)
    bounds = np.zeros(n_parts + 1, dtype=np.int32)
    rc = lib.sdcp_split_sessions(off.ctypes.data_as(ctypes.c_void_p),
                                 None if prm is None else prm.ctypes.data_as(ctypes.c_void_p),
                                 B, int(n_parts), bounds.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "sdcp_split_sessions")
    return bounds


class Verifier:
    """Owns the output and workspace buffers of one batch shape on one device."""

    def __init__(self, V: int, B: int, total_drafts: int, device):
        self.V, self.B, self.total = V, B, int(total_drafts)
        self.device = torch.device(device)
        self.accepted = torch.empty(B, dtype=torch.int32, device=self.device)
        self.n_out = torch.empty(B, dtype=torch.int32, device=self.device)
        self.out_tokens = torch.empty(self.total + B, dtype=torch.int32, device=self.device)
        self.status = torch.empty(B, dtype=torch.int32, device=self.device)
        self.workspace = alloc_workspace(V, B, self.total, self.device)

    def __call__(self, target, draft, m_offsets, draft_tokens, params_dev, stream=None,
                 rng_id=RNG_PHILOX4X32_10, session_ids=None, q_rows=None):
        if rng_id == RNG_PHILOX4X32_10 and session_ids is None and q_rows is None:
            sdcp_verify_batch(target, draft, m_offsets, self.total, draft_tokens, params_dev,
                              self.accepted, self.n_out, self.out_tokens, self.status,
                              self.workspace, stream)
        else:
            sdcp_verify_batch_ex(target, draft, m_offsets, self.total, draft_tokens, params_dev,
                                 self.accepted, self.n_out, self.out_tokens, self.status,
                                 self.workspace, rng_id, session_ids, q_rows, stream)
        return self.accepted, self.n_out, self.out_tokens, self.status

    def phases(self, target, draft, m_offsets, draft_tokens, params_dev, ev_mid=None):
        """Phase 1 then phase 2 (identical to __call__), optionally recording ev_mid between."""
        sdcp_verify_rows(target, draft, m_offsets, self.total, draft_tokens, params_dev,
                         self.workspace, self.B)
        if ev_mid is not None:
            ev_mid.record()
        sdcp_verify_sessions(target, draft, m_offsets, self.total, draft_tokens, params_dev,
                             self.accepted, self.n_out, self.out_tokens, self.status,
                             self.workspace)
        return self.accepted, self.n_out, self.out_tokens, self.status

    def row_stats(self, target, draft, m_offsets, draft_tokens, params_dev):
        out = torch.empty((2 * self.total + self.B) * 32, dtype=torch.uint8, device=self.device)
        sdcp_row_stats(target, draft, m_offsets, self.total, draft_tokens, params_dev, out,
                       self.workspace)
        return out
