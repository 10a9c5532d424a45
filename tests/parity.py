"""Comparison of the CUDA path with the CPU oracle on the same seeded inputs.

Rule 1 (greedy) outcomes must be bit-exact.  Rule 2 outcomes must be bit-exact except
where a decision lies within 1e-5 (relative) of its boundary in the oracle's own fp64
arithmetic: an acceptance uniform within 1e-5 of min(1, p/q), a draw whose uniform lies
within 1e-5 * W of the edge of the drawn token's cumulative interval, or a top-p crossing
within 1e-5 of P.  Such cases are counted and returned, never silently accepted.
Row statistics: lmax, argmax and the kept count exactly (kept count except at a top-p
boundary), log S and log p(x) within 1e-5 (fp32 logits) or 2e-3 (bf16 logits).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_verification_sdcp_gb300 import synth
from speculative_decoding_verification_sdcp_gb300.sdcp import (ROW_STAT_DTYPE, ROW_FALLBACK,
                                                              Verifier)

BOUNDARY = 1e-5
ROW_TOL = {synth.F32: 1e-5, synth.BF16: 2e-3}


def run_gpu(batch: synth.Batch, with_draft=True):
    ver = Verifier(batch.V, batch.B, batch.total_drafts, batch.target.device)
    acc, nout, toks, st = ver(batch.target, batch.draft if with_draft else None, batch.m_offsets,
                              batch.draft_tokens, batch.params_dev)
    torch.cuda.synchronize()
    return {"accepted": acc.cpu().numpy(), "n_out": nout.cpu().numpy(),
            "out_tokens": toks.cpu().numpy(), "status": st.cpu().numpy()}


def gpu_row_stats(batch: synth.Batch):
    ver = Verifier(batch.V, batch.B, batch.total_drafts, batch.target.device)
    raw = ver.row_stats(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens,
                        batch.params_dev)
    torch.cuda.synchronize()
    return raw.cpu().numpy().view(ROW_STAT_DTYPE)


def host_arrays(batch: synth.Batch):
    return (synth.to_numpy_logits(batch.target), synth.to_numpy_logits(batch.draft),
            batch.m_offsets.detach().cpu().numpy(), batch.draft_tokens.detach().cpu().numpy())


def sub_batch(batch: synth.Batch, sessions):
    """Host arrays of a subset of sessions, re-laid out as a batch of their own (rows are
    gathered on the device, so only the sampled rows cross to the host)."""
    off = batch.m_offsets.detach().cpu().numpy().astype(np.int64)
    trows, drows, offs = [], [], [0]
    for b in sessions:
        o0, o1 = int(off[b]), int(off[b + 1])
        trows.extend(range(o0 + b, o1 + b + 1))
        drows.extend(range(o0, o1))
        offs.append(offs[-1] + (o1 - o0))
    dev = batch.target.device
    ti = torch.as_tensor(trows, dtype=torch.long, device=dev)
    di = torch.as_tensor(drows, dtype=torch.long, device=dev)
    T = synth.to_numpy_logits(batch.target.index_select(0, ti))
    D = synth.to_numpy_logits(batch.draft.index_select(0, di))
    x = batch.draft_tokens.index_select(0, di).cpu().numpy().astype(np.int32)
    return T, D, np.asarray(offs, np.int32), x, batch.params[list(sessions)]


def _draw_interval(T, D, off, b, a, prm, token, mode):
    """Oracle cumulative interval [C_{j-1}, C_j] of `token` for the draw of session b."""
    s = int(off[b]) + b + a
    tm, k, p = int(prm["temperature_milli"]), int(prm["top_k"]), int(prm["top_p_milli"])
    pa = oracle.row_dist(T[s], tm, k, p)[0]
    qa = oracle.row_dist(D[int(off[b]) + a], tm, k, p)[0] if mode == oracle.EXTRA_RESIDUAL else None
    C, W = oracle.draw_cdf(pa, qa)
    lo = C[token - 1] if token > 0 else 0.0
    return lo, C[token], W


def compare_verdicts(got, ref, T, D, off, x, params):
    """Returns a dict of counts; raises AssertionError on a real disagreement."""
    det = ref["detail"]
    B = params.shape[0]
    counts = {"sessions": B, "exact": 0, "accept_boundary": 0, "draw_boundary": 0,
              "topp_boundary": 0}
    assert np.array_equal(got["status"], ref["status"]), (got["status"], ref["status"])
    for b in range(B):
        o0, o1 = int(off[b]), int(off[b + 1])
        M = o1 - o0
        slot = slice(o0 + b, o1 + b + 1) if 0 <= o0 <= o1 else slice(0, 0)
        same = (got["accepted"][b] == ref["accepted"][b] and got["n_out"][b] == ref["n_out"][b]
                and np.array_equal(got["out_tokens"][slot], ref["out_tokens"][slot]))
        if same:
            counts["exact"] += 1
            continue
        rule = int(params["rule_id"][b])
        assert rule == 2, "greedy session %d differs: gpu a=%d tokens=%s, oracle a=%d tokens=%s" % (
            b, got["accepted"][b], got["out_tokens"][slot], ref["accepted"][b], ref["out_tokens"][slot])
        tmargin = det["topp_margin"][b]
        if tmargin <= BOUNDARY:
            counts["topp_boundary"] += 1
            continue
        ag, ao = int(got["accepted"][b]), int(ref["accepted"][b])
        if ag != ao:
            i = min(ag, ao)
            u, r = det["u0"][b][i], det["ratio"][b][i]
            assert not np.isnan(r), (b, i)
            margin = abs(u - r) / max(r, 1e-300)
            assert margin <= BOUNDARY, "session %d: acceptance at position %d differs, u=%r ratio=%r" % (b, i, u, r)
            counts["accept_boundary"] += 1
            continue
        # same a: the prefix must match exactly, only the drawn token may differ
        a = ag
        gt = got["out_tokens"][o0 + b:o0 + b + a + 1]
        rt = ref["out_tokens"][o0 + b:o0 + b + a + 1]
        assert np.array_equal(gt[:a], rt[:a]) and got["n_out"][b] == a + 1
        mode = int(det["extra_mode"][b])
        assert mode in (oracle.EXTRA_RESIDUAL, oracle.EXTRA_BONUS, oracle.EXTRA_RESIDUAL_AS_P), mode
        tok = int(gt[a])
        assert 0 <= tok < T.shape[1], tok
        m2 = oracle.EXTRA_RESIDUAL if mode == oracle.EXTRA_RESIDUAL else oracle.EXTRA_BONUS
        lo, hi, W = _draw_interval(T, D, off, b, a, params[b], tok, m2)
        target = det["u1"][b] * W
        assert hi > lo, "session %d: GPU drew token %d of zero weight" % (b, tok)
        assert lo - BOUNDARY * W <= target <= hi + BOUNDARY * W, (
            "session %d: GPU token %d interval [%r, %r] far from u*W=%r (W=%r), oracle token %d" % (
                b, tok, lo, hi, target, W, int(rt[a])))
        counts["draw_boundary"] += 1
        # only the last slot may differ
        assert np.array_equal(got["out_tokens"][o0 + b + a + 1:o1 + b + 1],
                              ref["out_tokens"][o0 + b + a + 1:o1 + b + 1])
    return counts


def check_invariants(got, off, x, params, V):
    """Properties that hold at any size (SDCP Sections 5.2 and 6.4)."""
    B = params.shape[0]
    for b in range(B):
        o0, o1 = int(off[b]), int(off[b + 1])
        M = o1 - o0
        if got["status"][b] != 0:
            assert got["accepted"][b] == 0 and got["n_out"][b] == 0
            continue
        a, n = int(got["accepted"][b]), int(got["n_out"][b])
        assert 0 <= a <= M and n == a + 1
        toks = got["out_tokens"][o0 + b:o1 + b + 1]
        assert np.array_equal(toks[:a], x[o0:o0 + a])
        assert 0 <= toks[a] < V
        assert (toks[a + 1:] == -1).all()


def compare_row_stats(gs, T, D, off, x, params, dtype_code, rows=None):
    """GPU sdcp_row_stats against oracle.row_dist on the listed rows (default: all)."""
    B = params.shape[0]
    total = int(off[-1])
    R_T = total + B
    tol = ROW_TOL[dtype_code]
    sess_t = np.repeat(np.arange(B), np.diff(off) + 1)
    sess_d = np.repeat(np.arange(B), np.diff(off))
    rows = range(R_T + total) if rows is None else rows
    n_topp_boundary = 0
    n_fallback = 0
    for r in rows:
        if r < R_T:
            b = int(sess_t[r]); logits = T[r]; pos = r - int(off[b]) - b
            xi = int(x[r - b]) if pos < int(off[b + 1]) - int(off[b]) else None
        else:
            d = r - R_T; b = int(sess_d[d]); logits = D[d]; xi = int(x[d])
        prm = params[b]
        tm, k, p = int(prm["temperature_milli"]), int(prm["top_k"]), int(prm["top_p_milli"])
        dist, kept, info, rc = oracle.row_dist(logits, tm, k, p, want_kept=True)
        g = gs[r]
        if g["flags"] & ROW_FALLBACK:
            n_fallback += 1
        if rc != 0:
            assert g["flags"] & 1, (r, "oracle says invalid row")
            continue
        assert not (g["flags"] & 1), (r, "gpu says invalid row")
        assert float(g["lmax"]) == float(info.lmax), (r, g["lmax"], info.lmax)
        assert int(g["argmax"]) == int(info.argmax), (r, g["argmax"], info.argmax)
        topp_b = info.topp_target >= 0 and min(abs(info.topp_cum_at - info.topp_target),
                                               abs(info.topp_cum_before - info.topp_target)) <= BOUNDARY * info.topp_target
        if topp_b:
            n_topp_boundary += 1
            continue
        assert int(g["kept"]) == int(info.kept), (r, g["kept"], info.kept)
        assert abs(float(g["log_s"]) - info.log_s) <= tol * max(1.0, abs(info.log_s)), (r, g["log_s"], info.log_s)
        if xi is not None and 0 <= xi < len(dist):
            px = dist[xi]
            if kept[xi] and px > 0:
                lp = np.log(px)
                assert abs(float(g["lp_x"]) - lp) <= tol * max(1.0, abs(lp)), (r, g["lp_x"], lp)
            elif not kept[xi]:
                assert float(g["lp_x"]) == -np.inf, (r, g["lp_x"])
    return {"rows": len(rows), "topp_boundary": n_topp_boundary, "fallback": n_fallback}
