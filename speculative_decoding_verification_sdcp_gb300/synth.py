"""Seeded synthetic verify batches shaped like the workloads the SDCP pages describe.

There are no trained weights or real logits here.  A batch is made of
  * target logits: i.i.d. Normal(0, sigma^2) per element (the scores of M+1 positions per
    session), rounded to the batch dtype;
  * draft logits: ``draft_scale * target + Normal(0, noise^2)`` (a drafter that agrees with
    the target up to noise), rounded to the dtype;
  * draft tokens: a stand-in drafter samples each proposed token from its own row after
    the session's sampling profile, because a drafter "MUST sample each proposed token
    from exactly the row it publishes" (SDCP draft, Section 5.2, the q_rows object);
  * per-session parameters (rule, temperature, top-k, top-p, seed, round, tag).

This module is shared by the tests, the benchmark and the smoke check.  It computes no
part of the verifier's acceptance step; the stand-in drafter below is the party that
*proposes* tokens, outside the method under test, written with plain torch operations.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np
import torch

F32, BF16 = 0, 1

# 32-byte per-session parameter record, the layout of sdcp_session_params.
PARAMS_DTYPE = np.dtype([("rule_id", "<u4"), ("temperature_milli", "<u4"), ("top_k", "<u4"),
                         ("top_p_milli", "<u4"), ("seed", "<u8"), ("round", "<u4"),
                         ("session_tag", "<u4")])


@dataclass
class Workload:
    """Recipe of one synthetic verify batch."""
    name: str
    B: int
    V: int
    dtype: int                     # F32 or BF16
    m: int | tuple = 4             # constant M, or ("uniform", lo, hi) per session
    sigma: float = 2.0             # std of the target logits
    noise: float = 0.5             # std of the drafter's disagreement
    draft_scale: float = 1.0       # drafter logits = draft_scale * target + noise
    rules: str = "spec"            # "greedy", "spec", "relaxed" (private rule 192), or
                                   # "alternate" (even greedy, odd spec)
    temperature_milli: int | tuple = 1000   # constant, or a tuple drawn from per session
    top_k: int = 0
    top_p_milli: int = 1000
    seed_base: int = 0             # session b gets seed seed_base + b (seed_same: all equal)
    seed_same: bool = False
    gen_seed: int = 0              # seed of the generator itself
    note: str = ""


# The five workloads of the verifier's acceptance step (sizes of the benchmark configs).
WORKLOADS = {
    "tiny": Workload("tiny", B=4, V=1000, dtype=F32, m=4, sigma=2.0, noise=0.5, rules="spec",
                     temperature_milli=1000, seed_base=0, seed_same=True, gen_seed=0,
                     note="B=4, M=4, V=1000, fp32 N(0,2^2), draft +N(0,0.5^2), T=1, seed 0"),
    "tiny_greedy": Workload("tiny_greedy", B=4, V=1000, dtype=F32, m=4, sigma=2.0, noise=0.5,
                            rules="greedy", temperature_milli=1000, seed_base=0,
                            seed_same=True, gen_seed=0,
                            note="as tiny, greedy rule"),
    "topk50": Workload("topk50", B=64, V=32000, dtype=BF16, m=8, sigma=3.0, noise=1.0,
                       rules="spec", temperature_milli=700, top_k=50, seed_base=1000,
                       gen_seed=2,
                       note="B=64, M=8, V=32000, bf16 N(0,3^2), draft +N(0,1), T=0.7, top_k=50"),
    "topp90_ragged": Workload("topp90_ragged", B=256, V=128256, dtype=BF16, m=("uniform", 1, 16),
                              sigma=3.0, noise=0.8, rules="spec", temperature_milli=800,
                              top_p_milli=900, seed_base=3000, gen_seed=3,
                              note="B=256, M~U{1..16}, V=128256, bf16 N(0,3^2), draft +N(0,0.8^2), T=0.8, top_p=0.9"),
    "large_batch_mixed": Workload("large_batch_mixed", B=1024, V=152064, dtype=BF16, m=4,
                                  sigma=3.0, noise=1.2, rules="alternate",
                                  temperature_milli=(500, 700, 1000), seed_base=4000, gen_seed=4,
                                  note="B=1024, M=4, V=152064, bf16 N(0,3^2), draft +N(0,1.2^2), half greedy, T in {0.5,0.7,1.0}"),
    "mmax_stress": Workload("mmax_stress", B=32, V=262144, dtype=F32, m=64, sigma=4.0, noise=0.5,
                            draft_scale=1.5, rules="spec", temperature_milli=1000, seed_base=5000,
                            gen_seed=5,
                            note="B=32, M=64, V=262144, fp32 N(0,4^2), draft 1.5x target +N(0,0.5^2), full distribution"),
}


@dataclass
class Batch:
    """Device (or host) tensors of one verify batch, in the C ABI's ragged layout."""
    workload: Workload
    target: torch.Tensor           # [total_drafts + B, V]
    draft: torch.Tensor            # [total_drafts, V]
    m_offsets: torch.Tensor        # [B+1] int32
    draft_tokens: torch.Tensor     # [total_drafts] int32
    params: np.ndarray             # [B] PARAMS_DTYPE (host)
    params_dev: torch.Tensor       # [B*32] uint8 on the batch device
    extras: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.params.shape[0]

    @property
    def V(self):
        return self.target.shape[1]

    @property
    def total_drafts(self):
        return int(self.draft_tokens.shape[0])

    @property
    def dtype_code(self):
        return BF16 if self.target.dtype == torch.bfloat16 else F32


def torch_dtype(code: int):
    return torch.bfloat16 if code == BF16 else torch.float32


def to_numpy_logits(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of logits: float32 as is, bfloat16 as its raw uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def params_to_device(params: np.ndarray, device) -> torch.Tensor:
    raw = np.ascontiguousarray(params, dtype=PARAMS_DTYPE).view(np.uint8)
    return torch.from_numpy(raw.copy()).to(device)


def _draft_lengths(w: Workload, gen: np.random.Generator) -> np.ndarray:
    if isinstance(w.m, tuple):
        _, lo, hi = w.m
        return gen.integers(lo, hi + 1, size=w.B).astype(np.int64)
    return np.full(w.B, int(w.m), dtype=np.int64)


def make_params(w: Workload, gen: np.random.Generator) -> np.ndarray:
    p = np.zeros(w.B, dtype=PARAMS_DTYPE)
    b = np.arange(w.B)
    if w.rules == "greedy":
        p["rule_id"] = 1
    elif w.rules == "spec":
        p["rule_id"] = 2
    elif w.rules == "relaxed":
        p["rule_id"] = 192
    else:
        p["rule_id"] = np.where(b % 2 == 0, 1, 2)
    if isinstance(w.temperature_milli, tuple):
        p["temperature_milli"] = gen.choice(np.asarray(w.temperature_milli), size=w.B)
    else:
        p["temperature_milli"] = w.temperature_milli
    p["top_k"] = w.top_k
    p["top_p_milli"] = w.top_p_milli
    p["seed"] = w.seed_base if w.seed_same else (w.seed_base + b).astype(np.uint64)
    p["round"] = 1 + (b % 7)
    # a 32-bit session name that is not the batch slot (golden-ratio hash of b)
    p["session_tag"] = ((b.astype(np.uint64) + 1) * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)
    if w.name.startswith("tiny"):
        p["session_tag"] = b
    return p


def drafter_sample(draft_rows: torch.Tensor, temperature_milli: int, top_k: int,
                   top_p_milli: int, gen: torch.Generator) -> torch.Tensor:
    """Stand-in drafter: one token per row, drawn from the row after its sampling profile.

    Runs in float64 torch ops on the rows' device; the ranking is (logit desc, id asc).
    """
    V = draft_rows.shape[1]
    l = draft_rows.double()
    if temperature_milli == 0:
        return torch.argmax(l, dim=1).to(torch.int32)
    srt, idx = torch.sort(l, dim=1, descending=True, stable=True)
    k = V if (top_k == 0 or top_k >= V) else top_k
    srt, idx = srt[:, :k], idx[:, :k]
    z = srt / (temperature_milli / 1000.0)
    prob = torch.softmax(z, dim=1)
    if top_p_milli < 1000:
        cum = torch.cumsum(prob, dim=1)
        reach = cum >= (top_p_milli / 1000.0)
        # keep the minimal prefix whose cumulative reaches P (the crossing token included)
        first = torch.where(reach.any(dim=1), reach.int().argmax(dim=1),
                            torch.full_like(reach[:, 0], k - 1, dtype=torch.long))
        keep = torch.arange(k, device=l.device)[None, :] <= first[:, None]
        prob = torch.where(keep, prob, torch.zeros_like(prob))
        prob = prob / prob.sum(dim=1, keepdim=True)
    pick = torch.multinomial(prob, 1, generator=gen).squeeze(1)
    return idx.gather(1, pick[:, None]).squeeze(1).to(torch.int32)


def drafter_rows(draft_rows: torch.Tensor, temperature_milli: int, top_k: int,
                 top_p_milli: int) -> torch.Tensor:
    """The stand-in drafter's distributions over the whole vocabulary, as the binary32 rows it
    would publish (SDCP Section 5.2 q_rows): the same profile as drafter_sample, in float64,
    rounded to float32 at the end."""
    V = draft_rows.shape[1]
    l = draft_rows.double()
    out = torch.zeros_like(l)
    if temperature_milli == 0:
        out.scatter_(1, torch.argmax(l, dim=1, keepdim=True), 1.0)
        return out.float()
    srt, idx = torch.sort(l, dim=1, descending=True, stable=True)
    k = V if (top_k == 0 or top_k >= V) else top_k
    srt, idx = srt[:, :k], idx[:, :k]
    prob = torch.softmax(srt / (temperature_milli / 1000.0), dim=1)
    if top_p_milli < 1000:
        cum = torch.cumsum(prob, dim=1)
        reach = cum >= (top_p_milli / 1000.0)
        first = torch.where(reach.any(dim=1), reach.int().argmax(dim=1),
                            torch.full_like(reach[:, 0], k - 1, dtype=torch.long))
        keep = torch.arange(k, device=l.device)[None, :] <= first[:, None]
        prob = torch.where(keep, prob, torch.zeros_like(prob))
        prob = prob / prob.sum(dim=1, keepdim=True)
    out.scatter_(1, idx, prob)
    return out.float()


def make_batch(w: Workload, device="cpu", max_sessions: int | None = None,
               chunk_rows: int = 256) -> Batch:
    """Build the seeded batch of workload ``w`` on ``device`` (``max_sessions`` trims B)."""
    if max_sessions is not None and max_sessions < w.B:
        w = Workload(**{**w.__dict__, "B": max_sessions})
    gen_np = np.random.default_rng(w.gen_seed)
    lengths = _draft_lengths(w, gen_np)
    offs = np.zeros(w.B + 1, dtype=np.int64)
    offs[1:] = np.cumsum(lengths)
    total = int(offs[-1])
    params = make_params(w, gen_np)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1_000_003 * (w.gen_seed + 1))
    tdt = torch_dtype(w.dtype)
    V = w.V

    target = torch.empty(total + w.B, V, dtype=tdt, device=dev)
    draft = torch.empty(total, V, dtype=tdt, device=dev)
    for r0 in range(0, total + w.B, chunk_rows):
        r1 = min(total + w.B, r0 + chunk_rows)
        x = torch.randn(r1 - r0, V, generator=gen, device=dev, dtype=torch.float32) * w.sigma
        target[r0:r1] = x.to(tdt)
    # draft row of session b, position i <-> target row offs[b] + b + i
    sess_of_draft = np.repeat(np.arange(w.B), lengths)
    trow_of_draft = np.arange(total) + sess_of_draft
    trow_t = torch.from_numpy(trow_of_draft).to(dev)
    for d0 in range(0, total, chunk_rows):
        d1 = min(total, d0 + chunk_rows)
        base = target[trow_t[d0:d1]].float() * w.draft_scale
        nz = torch.randn(d1 - d0, V, generator=gen, device=dev, dtype=torch.float32) * w.noise
        draft[d0:d1] = (base + nz).to(tdt)

    tokens = torch.empty(total, dtype=torch.int32, device=dev)
    for b in range(w.B):
        d0, d1 = int(offs[b]), int(offs[b + 1])
        pb = params[b]
        tokens[d0:d1] = drafter_sample(draft[d0:d1], int(pb["temperature_milli"]),
                                       int(pb["top_k"]), int(pb["top_p_milli"]), gen)
    m_off = torch.from_numpy(offs.astype(np.int32)).to(dev)
    return Batch(w, target, draft, m_off, tokens, params, params_to_device(params, dev))


def shard_batch(batch: Batch, lo: int, hi: int) -> Batch:
    """Sessions lo .. hi-1 of a batch as a batch of their own: views of the same row buffers
    (the sessions' rows are contiguous in the ragged layout), offsets rebased to 0."""
    offs = batch.m_offsets.detach().cpu().numpy().astype(np.int64)
    o0, o1 = int(offs[lo]), int(offs[hi])
    target = batch.target[o0 + lo:o1 + hi]
    draft = batch.draft[o0:o1]
    m_off = torch.from_numpy((offs[lo:hi + 1] - o0).astype(np.int32)).to(batch.target.device)
    tokens = batch.draft_tokens[o0:o1]
    params = batch.params[lo:hi].copy()
    w = Workload(**{**batch.workload.__dict__, "B": hi - lo})
    return Batch(w, target, draft, m_off, tokens, params, batch.params_dev[lo * 32:hi * 32])


def custom_workload(**kw) -> Workload:
    """A workload with explicit fields (for small parity and edge cases)."""
    base = dict(name="custom", B=4, V=64, dtype=F32)
    base.update(kw)
    return Workload(**base)


def algorithmic_bytes(batch: Batch) -> dict:
    """One read of every scored row: the target rows of every session, plus the draft rows
    of Rule 2 sessions (Rule 1 needs no q), at the element size of the batch."""
    esz = 2 if batch.dtype_code == BF16 else 4
    offs = batch.m_offsets.detach().cpu().numpy().astype(np.int64)
    M = offs[1:] - offs[:-1]
    rule2 = batch.params["rule_id"] == 2
    rows_t = int((M + 1).sum())
    rows_d = int(M[rule2].sum())
    return {"rows_target": rows_t, "rows_draft": rows_d, "rule2_sessions": int(rule2.sum()),
            "bytes_rows": (rows_t + rows_d) * batch.V * esz,
            "bytes_extra_row_per_session": batch.B * batch.V * esz}
