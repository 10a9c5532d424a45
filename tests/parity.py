"""Comparison of the CUDA path with the CPU oracle on the same seeded inputs.

Rule 1 (greedy) outcomes must be bit-exact.  Rule 2 outcomes must be bit-exact except
where a decision lies within 1e-5 (relative) of its boundary in the oracle's own fp64
arithmetic, and then the GPU's outcome must be the one on the other side of that boundary:
  * acceptance: the uniform within 1e-5 of min(1, p/q) at the first position where the
    two accepted counts part;
  * draw: the GPU's token has positive weight and u * W lies within 1e-5 * W of its
    cumulative interval (ids ascending), so the tokens between it and the oracle's token
    weigh less than 1e-5 * W in all;
  * top-p crossing (SDCP Section 4.1): where a row's cumulative mass lies within 1e-5 of
    P, any crossing between the oracle's crossings for P (1 - 1e-5) and P (1 + 1e-5) is a
    faithful reading; the GPU's crossing must lie in that band, and the session must then
    match the oracle run with the GPU's crossing (under the rules above).
Such cases are counted and returned, never silently accepted.
Row statistics: lmax, argmax and the kept count exactly, log S and log p(x) within 1e-5
(fp32 logits) or 2e-3 (bf16 logits); a row at a top-p boundary must keep a count inside
the band, and its log S and log p(x) must match the oracle's at that count.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from speculative_decoding_verification_sdcp_gb300 import synth
from speculative_decoding_verification_sdcp_gb300.sdcp import (ROW_STAT_DTYPE, ROW_FALLBACK,
                                                              ROW_INVALID, ROW_SKIPPED, Verifier)

BOUNDARY = 1e-5
ROW_TOL = {synth.F32: 1e-5, synth.BF16: 2e-3}
ORACLE_THREADS = max(1, min(64, len(os.sched_getaffinity(0))))


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


def session_arrays(T, D, off, x, params, b):
    """Host arrays of session b alone, laid out as a batch of one."""
    o0, o1 = int(off[b]), int(off[b + 1])
    return (T[o0 + b:o1 + b + 1], D[o0:o1], np.asarray([0, o1 - o0], np.int32),
            np.ascontiguousarray(x[o0:o1], dtype=np.int32), params[b:b + 1])


def _sid(session_ids, b):
    return None if session_ids is None else session_ids[b:b + 1]


def _qr(q_rows, off, b):
    return None if q_rows is None else q_rows[int(off[b]):int(off[b + 1])]


def session_outputs(got, off, b):
    o0, o1 = int(off[b]), int(off[b + 1])
    return {"status": got["status"][b:b + 1], "accepted": got["accepted"][b:b + 1],
            "n_out": got["n_out"][b:b + 1], "out_tokens": got["out_tokens"][o0 + b:o1 + b + 1]}


def _draw_cdf(T, D, off, b, a, prm, mode, force=None, q_rows=None):
    """Oracle cumulative weights (ids ascending) of the draw of session b at position a
    (force: top-p crossings per row, in the row order of the C ABI's row statistics; q_rows:
    q given as probability rows)."""
    s = int(off[b]) + b + a
    d = int(off[b]) + a
    R_T = int(off[-1]) + (off.shape[0] - 1)
    tm, k, p = int(prm["temperature_milli"]), int(prm["top_k"]), int(prm["top_p_milli"])
    fp = -1 if force is None else int(force[s])
    fq = -1 if force is None else int(force[R_T + d])
    pa = oracle.row_dist(T[s], tm, k, p, force_kept=fp)[0]
    qa = None
    if mode == oracle.EXTRA_RESIDUAL:
        qa = q_rows[d].astype(np.float64) if q_rows is not None else oracle.row_dist(D[d], tm, k, p, force_kept=fq)[0]
    return oracle.draw_cdf(pa, qa)


def _check_draw_boundary(C, W, u1, tg, to, b):
    """A draw that differs is a boundary case when u * W lies within BOUNDARY * W of the
    GPU token's own cumulative interval (ids ascending) and that token has positive weight:
    every token between the two then carries less than BOUNDARY * W in all."""
    V = C.shape[0]
    assert 0 <= tg < V, "session %d: GPU token %d out of range" % (b, tg)
    lo_g = C[tg - 1] if tg > 0 else 0.0
    hi_g = C[tg]
    assert hi_g > lo_g, "session %d: GPU drew token %d of zero weight" % (b, tg)
    target = u1 * W
    lo_o = C[to - 1] if to > 0 else 0.0
    assert lo_o <= target < C[to] or target >= W, (b, to, target)  # the oracle's own token
    gap = 0.0 if lo_g <= target < hi_g else min(abs(target - lo_g), abs(target - hi_g))
    assert gap <= BOUNDARY * W, (
        "session %d: GPU token %d, oracle token %d: u*W=%r is %r from the GPU token's interval "
        "[%r, %r) (W=%r)" % (b, tg, to, target, gap, lo_g, hi_g, W))


def topp_band(logits, tm, k, p):
    """Kept counts of the oracle's top-p crossing for P (1 - 1e-5) and P (1 + 1e-5)."""
    with oracle.topp_shift(-BOUNDARY):
        lo = oracle.row_dist(logits, tm, k, p, want_dist=False)[2].kept
    with oracle.topp_shift(BOUNDARY):
        hi = oracle.row_dist(logits, tm, k, p, want_dist=False)[2].kept
    return int(lo), int(hi)


def _row_margin(info):
    if info.topp_target < 0:
        return np.inf
    return min(abs(info.topp_cum_at - info.topp_target),
               abs(info.topp_cum_before - info.topp_target)) / info.topp_target


def _forced_session(T, D, off, x, params, b, gs, session_ids=None, q_rows=None):
    """The oracle on session b alone with the GPU's top-p crossings at the session's
    boundary rows (each checked to lie in its band)."""
    B = params.shape[0]
    total = int(off[-1])
    R_T = total + B
    args = session_arrays(T, D, off, x, params, b)
    Ts, Ds = args[0], args[1]
    M = Ts.shape[0] - 1
    prm = params[b]
    tm, k, p = int(prm["temperature_milli"]), int(prm["top_k"]), int(prm["top_p_milli"])
    force = np.full(2 * M + 1, -1, np.int32)
    o0 = int(off[b])
    rows = [(i, Ts[i], o0 + b + i) for i in range(M + 1)] + [(M + 1 + i, Ds[i], R_T + o0 + i) for i in range(M)]
    for j, logits, r in rows:
        info = oracle.row_dist(logits, tm, k, p, want_dist=False)[2]
        if info.invalid or _row_margin(info) > BOUNDARY:
            continue
        n = int(gs[r]["kept"])
        lo, hi = topp_band(logits, tm, k, p)
        assert lo <= n <= hi, ("session %d row %d: GPU crossing %d outside the band [%d, %d]" % (b, r, n, lo, hi))
        force[j] = n
    return args, force, oracle.verify_batch(*args, force_kept=force, session_ids=_sid(session_ids, b),
                                            q_rows=_qr(q_rows, off, b))


def _draw_diagnostics(T, D, off, params, b, a, mode, gs, det, force):
    """What the GPU and the oracle each made of the draw's rows (for a failure message)."""
    B = params.shape[0]
    R_T = int(off[-1]) + B
    prm = params[b]
    tm, k, p = int(prm["temperature_milli"]), int(prm["top_k"]), int(prm["top_p_milli"])
    rows = [("p", int(off[b]) + b + a, T[int(off[b]) + b + a])]
    if mode == oracle.EXTRA_RESIDUAL:
        rows.append(("q", R_T + int(off[b]) + a, D[int(off[b]) + a]))
    lines = ["draw of session %d at position %d (mode %d), u1=%r" % (b, a, mode, float(det["u1"][b]))]
    for name, r, logits in rows:
        info = oracle.row_dist(logits, tm, k, p, want_dist=False)[2]
        band = topp_band(logits, tm, k, p) if info.topp_target >= 0 else None
        g = "n/a" if gs is None else "kept=%d log_s=%.9g thr_n=%d flags=%d" % (
            int(gs[r]["kept"]), float(gs[r]["log_s"]), int(gs[r]["thr_n"]), int(gs[r]["flags"]))
        lines.append("  %s row %d: oracle kept=%d log_s=%.9g margin=%.3g band=%s | gpu %s" % (
            name, r, info.kept, info.log_s, _row_margin(info), band, g))
    if gs is not None:
        u1 = float(det["u1"][b])
        fp = int(gs[rows[0][1]]["kept"])
        fq = int(gs[rows[1][1]]["kept"]) if len(rows) > 1 else -1
        pa, kp = oracle.row_dist(rows[0][2], tm, k, p, want_kept=True, force_kept=fp)[:2]
        qa, kq = oracle.row_dist(rows[1][2], tm, k, p, want_kept=True, force_kept=fq)[:2] if len(rows) > 1 else (None, None)
        C2, W2 = oracle.draw_cdf(pa, qa)
        tok = int(np.searchsorted(C2, u1 * W2, side="right"))
        lines.append("  oracle draw with the GPU's kept counts: token %d (W=%r)" % (tok, W2))

        # and with the GPU's normalisers too: p_j = exp((l_j - lmax)/T) / S_gpu on the kept set
        def with_gpu_s(logits, kept, r):
            l = logits.astype(np.float64) if logits.dtype == np.float32 else \
                (logits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            z = (l - l.max()) / (tm / 1000.0)
            return np.where(kept.astype(bool), np.exp(z - float(gs[r]["log_s"])), 0.0)
        pg = with_gpu_s(rows[0][2], kp, rows[0][1])
        qg = with_gpu_s(rows[1][2], kq, rows[1][1]) if len(rows) > 1 else None
        C3, W3 = oracle.draw_cdf(pg, qg)
        tok3 = int(np.searchsorted(C3, u1 * W3, side="right"))
        lines.append("  oracle draw with the GPU's kept counts and log S: token %d (W=%r)" % (tok3, W3))
    return "\n".join(lines)


def _compare_session(got, ref, T, D, off, x, params, b, counts, topp_ok, gs=None, force=None,
                     session_ids=None, q_rows=None):
    """One session; adds to counts; raises AssertionError on a real disagreement.  force:
    the top-p crossings ref was computed with (None: as defined)."""
    det = ref["detail"]
    o0, o1 = int(off[b]), int(off[b + 1])
    slot = slice(o0 + b, o1 + b + 1) if 0 <= o0 <= o1 else slice(0, 0)
    assert got["status"][b] == ref["status"][b], (b, got["status"][b], ref["status"][b])
    same = (got["accepted"][b] == ref["accepted"][b] and got["n_out"][b] == ref["n_out"][b]
            and np.array_equal(got["out_tokens"][slot], ref["out_tokens"][slot]))
    if same:
        counts["exact"] += 1
        return
    rule = int(params["rule_id"][b])
    assert rule in (2, 192), "greedy session %d differs: gpu a=%d tokens=%s, oracle a=%d tokens=%s" % (
        b, got["accepted"][b], got["out_tokens"][slot], ref["accepted"][b], ref["out_tokens"][slot])
    if topp_ok and det["topp_margin"][b] <= BOUNDARY:
        # a top-p crossing within rounding of P: the session must match the oracle run with
        # the GPU's crossings (each inside its band), or, without the GPU's row statistics,
        # the oracle under one of the band's two ends
        mine = session_outputs(got, off, b)
        if gs is not None:
            args, force2, r2 = _forced_session(T, D, off, x, params, b, gs, session_ids, q_rows)
            c2 = {"exact": 0, "accept_boundary": 0, "draw_boundary": 0, "topp_boundary": 0}
            try:
                _compare_session(mine, r2, *args, 0, c2, topp_ok=False, force=force2,
                                 session_ids=_sid(session_ids, b), q_rows=_qr(q_rows, off, b))
            except AssertionError as e:
                a = int(got["accepted"][b])
                mode = int(r2["detail"]["extra_mode"][0])
                raise AssertionError("%s\n(full batch) %s" % (
                    e, _draw_diagnostics(T, D, off, params, b, a, mode, gs, det, None)))
            counts["topp_boundary"] += 1
            return
        args = session_arrays(T, D, off, x, params, b)
        errs = []
        for shift in (-BOUNDARY, BOUNDARY):
            c2 = {"exact": 0, "accept_boundary": 0, "draw_boundary": 0, "topp_boundary": 0}
            with oracle.topp_shift(shift):
                r2 = oracle.verify_batch(*args, session_ids=_sid(session_ids, b), q_rows=_qr(q_rows, off, b))
                try:
                    _compare_session(mine, r2, *args, 0, c2, topp_ok=False,
                                     session_ids=_sid(session_ids, b), q_rows=_qr(q_rows, off, b))
                except AssertionError as e:
                    errs.append(str(e))
                    continue
            counts["topp_boundary"] += 1
            return
        raise AssertionError("session %d matches neither end of its top-p band: %s" % (b, errs))
    ag, ao = int(got["accepted"][b]), int(ref["accepted"][b])
    if ag != ao:
        i = min(ag, ao)
        u, r = det["u0"][b][i], det["ratio"][b][i]
        assert not np.isnan(r), (b, i)
        margin = abs(u - r) / max(r, 1e-300)
        assert margin <= BOUNDARY, "session %d: acceptance at position %d differs, u=%r ratio=%r" % (b, i, u, r)
        counts["accept_boundary"] += 1
        return
    # same a: the prefix must match exactly, only the drawn token may differ
    a = ag
    gt = got["out_tokens"][o0 + b:o0 + b + a + 1]
    rt = ref["out_tokens"][o0 + b:o0 + b + a + 1]
    assert np.array_equal(gt[:a], rt[:a]) and got["n_out"][b] == a + 1
    mode = int(det["extra_mode"][b])
    assert mode in (oracle.EXTRA_RESIDUAL, oracle.EXTRA_BONUS, oracle.EXTRA_RESIDUAL_AS_P,
                    oracle.EXTRA_FROM_P), mode
    m2 = oracle.EXTRA_RESIDUAL if mode == oracle.EXTRA_RESIDUAL else oracle.EXTRA_BONUS
    C, W = _draw_cdf(T, D, off, b, a, params[b], m2, force, q_rows)
    try:
        _check_draw_boundary(C, W, float(det["u1"][b]), int(gt[a]), int(rt[a]), b)
    except AssertionError as e:
        raise AssertionError(str(e) + "\n" + _draw_diagnostics(T, D, off, params, b, a, m2, gs, det, force))
    counts["draw_boundary"] += 1
    # only the drawn slot may differ
    assert np.array_equal(got["out_tokens"][o0 + b + a + 1:o1 + b + 1],
                          ref["out_tokens"][o0 + b + a + 1:o1 + b + 1])


def compare_verdicts(got, ref, T, D, off, x, params, gs=None, session_ids=None, q_rows=None):
    """Returns a dict of counts; raises AssertionError on a real disagreement.  gs: the
    GPU's row statistics of the same batch (sdcp_row_stats), used where a top-p crossing
    lies within rounding of P."""
    B = params.shape[0]
    counts = {"sessions": B, "exact": 0, "accept_boundary": 0, "draw_boundary": 0,
              "topp_boundary": 0}
    assert np.array_equal(got["status"], ref["status"]), (got["status"], ref["status"])
    for b in range(B):
        _compare_session(got, ref, T, D, off, x, params, b, counts, topp_ok=True, gs=gs,
                         session_ids=session_ids, q_rows=q_rows)
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


def _row_logits(T, D, R_T, r):
    return T[r] if r < R_T else D[r - R_T]


def _row_session(off, B, total, r):
    R_T = total + B
    if r < R_T:
        b = int(np.searchsorted(off + np.arange(B + 1), r, side="right") - 1)
        pos = r - int(off[b]) - b
        xi = r - b if pos < int(off[b + 1]) - int(off[b]) else None
    else:
        d = r - R_T
        b = int(np.searchsorted(off, d, side="right") - 1)
        xi = d
    return b, xi


def compare_row_stats(gs, T, D, off, x, params, dtype_code, rows=None):
    """GPU sdcp_row_stats against the oracle's row statistics on the listed rows (default:
    all), element by element."""
    B = params.shape[0]
    total = int(off[-1])
    R_T = total + B
    tol = ROW_TOL[dtype_code]
    info, lpx, skipped = oracle.row_stats_batch(T, D, off, x, params, nthreads=ORACLE_THREADS)
    sel = np.arange(R_T + total) if rows is None else np.asarray(list(rows), dtype=np.int64)
    g = gs[sel]
    o = info[sel]
    lp = lpx[sel]
    sk = skipped[sel]
    flags = g["flags"].astype(np.int64)
    assert np.array_equal((flags & ROW_SKIPPED) != 0, sk), "skipped rows differ"
    inv_g = (flags & ROW_INVALID) != 0
    inv_o = o["invalid"] != 0
    live = ~sk
    bad = np.nonzero(live & (inv_g != inv_o))[0]
    assert bad.size == 0, ("invalid flags differ", sel[bad[:5]])
    ok = live & ~inv_o
    bad = np.nonzero(ok & (g["lmax"].astype(np.float64) != o["lmax"]))[0]
    assert bad.size == 0, ("lmax differs", sel[bad[:5]], g["lmax"][bad[:5]], o["lmax"][bad[:5]])
    bad = np.nonzero(ok & (g["argmax"] != o["argmax"]))[0]
    assert bad.size == 0, ("argmax differs", sel[bad[:5]], g["argmax"][bad[:5]], o["argmax"][bad[:5]])
    tgt = o["topp_target"]
    tmargin = np.minimum(np.abs(o["topp_cum_at"] - tgt), np.abs(o["topp_cum_before"] - tgt))
    topp_b = ok & (tgt >= 0) & (tmargin <= BOUNDARY * np.maximum(tgt, 0))
    nb = ok & ~topp_b
    bad = np.nonzero(nb & (g["kept"] != o["kept"]))[0]
    assert bad.size == 0, ("kept differs", sel[bad[:5]], g["kept"][bad[:5]], o["kept"][bad[:5]])
    gls = g["log_s"].astype(np.float64)
    bad = np.nonzero(nb & ~(np.abs(gls - o["log_s"]) <= tol * np.maximum(1.0, np.abs(o["log_s"]))))[0]
    assert bad.size == 0, ("log S differs", sel[bad[:5]], gls[bad[:5]], o["log_s"][bad[:5]])
    glp = g["lp_x"].astype(np.float64)
    fin = nb & np.isfinite(lp)
    with np.errstate(invalid="ignore"):
        bad = np.nonzero(fin & ~(np.abs(glp - lp) <= tol * np.maximum(1.0, np.abs(lp))))[0]
    assert bad.size == 0, ("log p(x) differs", sel[bad[:5]], glp[bad[:5]], lp[bad[:5]])
    ninf = nb & np.isneginf(lp)
    bad = np.nonzero(ninf & ~np.isneginf(glp))[0]
    assert bad.size == 0, ("log p(x) should be -inf", sel[bad[:5]], glp[bad[:5]])
    nan = nb & np.isnan(lp)
    bad = np.nonzero(nan & ~np.isnan(glp))[0]
    assert bad.size == 0, ("log p(x) should be NaN (no draft token)", sel[bad[:5]], glp[bad[:5]])
    # rows at a top-p boundary: the GPU's crossing must lie in the band, and the row's
    # statistics must match the oracle's with that crossing
    for i in np.nonzero(topp_b)[0]:
        r = int(sel[i])
        b, xi = _row_session(off, B, total, r)
        prm = params[b]
        tm, k, p = int(prm["temperature_milli"]), int(prm["top_k"]), int(prm["top_p_milli"])
        logits = _row_logits(T, D, R_T, r)
        n = int(g["kept"][i])
        lo, hi = topp_band(logits, tm, k, p)
        assert lo <= n <= hi, ("row %d: GPU crossing %d outside the band [%d, %d]" % (r, n, lo, hi))
        dist, kept, inf2, rc = oracle.row_dist(logits, tm, k, p, want_kept=True, force_kept=n)
        assert int(inf2.kept) == n
        assert abs(gls[i] - inf2.log_s) <= tol * max(1.0, abs(inf2.log_s)), (r, gls[i], inf2.log_s)
        if xi is not None and 0 <= int(x[xi]) < len(dist):
            xv = int(x[xi])
            if kept[xv] and dist[xv] > 0:
                lpv = np.log(dist[xv])
                assert abs(glp[i] - lpv) <= tol * max(1.0, abs(lpv)), (r, glp[i], lpv)
            else:
                assert np.isneginf(glp[i]), (r, glp[i])
    return {"rows": int(sel.size), "topp_boundary": int(topp_b.sum()),
            "fallback": int(((flags & ROW_FALLBACK) != 0).sum())}


def report(name, counts):
    """Prints the boundary counts of a workload and, when SDCP_PARITY_REPORT names a file,
    appends them to it as one JSON line."""
    line = json.dumps({"case": name, **counts})
    print("parity", line)
    path = os.environ.get("SDCP_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")
