"""Multi-rank host logic on CPU ranks (gloo, world size 2).

Head sharding needs no exchange; split-KV needs one all-gather + merge.  Both
must reproduce the unsplit oracle result.  Partial results are computed with
the oracle (CPU); the plans and the merge are the library's host code.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from exact_attention_63_gb300 import dist as adist
from exact_attention_63_gb300 import inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, fn, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    except Exception as e:  # report, do not hang the parent
        q.put((rank, e))
    finally:
        dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    for r, v in res.items():
        if isinstance(v, Exception):
            raise v
    return res


W = inputs.custom(2, 3, 200, 300, 64, True, sigma_qk=2.0, seed=61)


def _heads_worker(rank, world):
    q, k, v = inputs.make_inputs(W)
    units = adist.shard_heads(W.B, W.H, world, rank)
    out = {}
    for b, h in units:
        O, L = oracle.attention_rows(q, k, v, W.scale, W.causal, b, h, np.arange(W.Sq))
        out[(b, h)] = (O, L)
    # gather every rank's heads (object collective; no tensor exchange needed on the data path)
    allp = [None] * world
    dist.all_gather_object(allp, out)
    merged = {}
    for part in allp:
        merged.update(part)
    return merged


def test_head_sharding_matches_unsplit():
    res = _run(_heads_worker)
    q, k, v = inputs.make_inputs(W)
    O, L = oracle.attention_forward(q, k, v, W.scale, W.causal)
    for rank, merged in res.items():
        assert sorted(merged) == [(b, h) for b in range(W.B) for h in range(W.H)]
        for (b, h), (Ob, Lb) in merged.items():
            assert np.array_equal(Ob, O[b, :, h, :]) and np.array_equal(Lb, L[b, h])


def _splitkv_worker(rank, world):
    q, k, v = inputs.make_inputs(W)
    a, b_ = adist.split_keys(W.Sk, world, rank)
    q64, k64, v64 = (oracle.to_f64(t) for t in (q, k, v))
    O = np.zeros((W.B, W.H, W.Sq, W.d))
    L = np.full((W.B, W.H, W.Sq), -np.inf)
    rows = np.arange(W.Sq)
    for bb in range(W.B):
        for h in range(W.H):
            mask = oracle.visible_mask(rows, W.Sk, W.causal)[:, a:b_]
            s = oracle.head_scores(q64[bb, :, h], k64[bb, a:b_, h], W.scale)
            P, M, Ls = oracle.head_probabilities(s, mask)
            O[bb, h] = P @ v64[bb, a:b_, h]
            with np.errstate(divide="ignore"):
                L[bb, h] = np.where(np.isfinite(M), M + np.log(np.where(Ls > 0, Ls, 1.0)), -np.inf)
    o_m, l_m = adist.gather_merge(torch.from_numpy(O), torch.from_numpy(L))
    t = torch.tensor([float(rank + 1)])
    return o_m.numpy(), l_m.numpy(), adist.max_over_ranks(float(rank + 1))


def test_split_kv_exchange_matches_unsplit():
    res = _run(_splitkv_worker)
    q, k, v = inputs.make_inputs(W)
    O, L = oracle.attention_forward(q, k, v, W.scale, W.causal)
    O_bhsd = O.transpose(0, 2, 1, 3)
    for rank, (o_m, l_m, mx) in res.items():
        assert np.max(np.abs(o_m - O_bhsd)) <= 1e-12
        assert np.max(np.abs(l_m - L)) <= 1e-12
        assert mx == 2.0


def test_plans():
    assert adist.shard_range(10, 3, 0) == (0, 4) and adist.shard_range(10, 3, 2) == (7, 10)
    seen = [u for r in range(4) for u in adist.shard_heads(3, 5, 4, r)]
    assert seen == [(b, h) for b in range(3) for h in range(5)]
    ranges = [adist.split_keys(1000, 3, r) for r in range(3)]
    assert ranges[0][0] == 0 and ranges[-1][1] == 1000
    assert all(x[1] == y[0] for x, y in zip(ranges, ranges[1:]))
    assert all(a % 128 == 0 for a, _ in ranges)
    assert adist.rank_seed(5, 0) == 5 and adist.rank_seed(5, 1) != 5
    with pytest.raises(ValueError):
        adist.shard_range(4, 2, 2)
