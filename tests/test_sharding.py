"""The multi-GPU split of one verify batch, on CPU (no GPU work).

Sessions are independent (SDCP Section 6.3, "Scoring": a verifier may batch the proposals of
many sessions), so one batch splits into contiguous blocks of sessions, one per GPU, with no
collective on the data path.  sdcp_split_sessions (C ABI, host code) chooses the blocks; the
tests check its bounds, its balance, and that verifying the blocks separately and
concatenating the outputs gives the whole batch's outputs bit for bit (the oracle stands in
for each rank's GPU; two gloo ranks on 127.0.0.1).
"""
import os
import sys

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def binding():
    from speculative_decoding_verification_sdcp_gb300 import build_ext
    build_ext.build()
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    return sdcp


def _rows(off, params):
    M = np.diff(off.astype(np.int64))
    return (M + 1) + np.where(params["rule_id"] == 2, M, 0)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
def test_split_bounds_are_contiguous_and_balanced(binding, n):
    rng = np.random.default_rng(n)
    B = 257
    M = rng.integers(1, 65, size=B)
    off = np.zeros(B + 1, np.int32)
    off[1:] = np.cumsum(M)
    prm = np.zeros(B, dtype=binding.PARAMS_DTYPE)
    prm["rule_id"] = rng.choice([1, 2], size=B)
    bounds = binding.sdcp_split_sessions(off, prm, n)
    assert bounds[0] == 0 and bounds[-1] == B and (np.diff(bounds) >= 0).all()
    w = _rows(off, prm)
    pre = np.concatenate([[0], np.cumsum(w)])
    total = pre[-1]
    for k in range(1, n):
        # boundary k is the session prefix closest to k/n of the rows
        goal = k * total / n
        best = np.min(np.abs(pre[bounds[k - 1]:] - goal))
        assert abs(pre[bounds[k]] - goal) == best
    # no block exceeds its share by more than one session's rows
    blocks = np.diff(pre[bounds])
    assert blocks.max() <= total / n + w.max()


def test_split_edge_cases(binding):
    off = np.zeros(1, np.int32)
    assert list(binding.sdcp_split_sessions(off, None, 4)) == [0, 0, 0, 0, 0]
    off = np.array([0, 3], np.int32)
    assert list(binding.sdcp_split_sessions(off, None, 3)) in ([0, 0, 1, 1], [0, 1, 1, 1], [0, 0, 0, 1])
    with pytest.raises(binding.SdcpError):
        binding.sdcp_split_sessions(np.array([0, 3, 2], np.int32), None, 2)
    with pytest.raises(binding.SdcpError):
        binding.sdcp_split_sessions(np.array([0, 3], np.int32), None, 0)


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    import oracle
    from speculative_decoding_verification_sdcp_gb300 import synth
    from speculative_decoding_verification_sdcp_gb300 import sdcp
    dist.init_process_group("gloo")
    w = synth.custom_workload(B=23, V=300, dtype=synth.BF16, m=("uniform", 1, 12), rules="alternate",
                              temperature_milli=(0, 700, 1000), top_k=40, top_p_milli=950,
                              sigma=2.0, noise=0.7, seed_base=11, gen_seed=31)
    batch = synth.make_batch(w, device="cpu")
    bounds = sdcp.sdcp_split_sessions(batch.m_offsets.numpy(), batch.params, world)
    lo, hi = int(bounds[rank]), int(bounds[rank + 1])
    shard = synth.shard_batch(batch, lo, hi)
    r = oracle.verify_batch(synth.to_numpy_logits(shard.target), synth.to_numpy_logits(shard.draft),
                            shard.m_offsets.numpy(), shard.draft_tokens.numpy(), shard.params,
                            want_detail=False)
    mine = {k: r[k] for k in ("accepted", "n_out", "out_tokens", "status")}
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        whole = oracle.verify_batch(synth.to_numpy_logits(batch.target), synth.to_numpy_logits(batch.draft),
                                    batch.m_offsets.numpy(), batch.draft_tokens.numpy(), batch.params,
                                    want_detail=False)
        ok = all(np.array_equal(np.concatenate([g[k] for g in gathered]), whole[k])
                 for k in ("accepted", "n_out", "out_tokens", "status"))
        q.put((ok, [int(v) for v in bounds]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_concatenate_to_the_whole_batch(binding):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29100 + (os.getpid() % 800)
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(300)
        assert p.exitcode == 0
    ok, bounds = q.get(timeout=10)
    assert 0 < bounds[1] < 23, bounds
    assert ok, bounds
