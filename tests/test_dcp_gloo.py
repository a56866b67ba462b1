"""DCP (KV sharded round-robin by token over G ranks) on CPU ranks over gloo.

Each spawned rank holds only its own positions (p % G == rank) of every
request, runs the DCP exchange of ``dsa_sparse_mla_topk_gb300.dcp`` with the
fp64 oracle as its compute steps, and must reproduce the single-rank result:
the same global top-k selection bit for bit, and the same attention output
and log-sum-exp (fp64 on both sides, so to rounding).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    from dsa_sparse_mla_topk_gb300 import workloads as wl
    # 3 requests x 3 query tokens, the tiny 16-head shape, ties in the scores
    return wl.Workload("dcp_h16", 3, 3, 16, 64, 16, 700, 0, 16, 64, seed=8, tie_frac=0.05,
                       ctx_per_req=(700, 333, 129))


def _local_pool(inp, w, rank, world):
    """This rank's positions of every request: local index j holds global
    position j * G + rank; identity pages, request-major."""
    P = w.page_size
    rows, scales, tables = [], [], []
    npages = 0
    for r, ctx in enumerate(w.contexts()):
        b, s = inp.logical[r]
        pos = np.arange(rank, ctx, world)
        n = len(pos)
        pages = -(-n // P)
        pad = pages * P - n
        rows.append(np.concatenate([b[pos], np.zeros((pad, w.dqk), np.uint8)]))
        scales.append(np.concatenate([s[pos], np.ones(pad, np.float32)]))
        tables.append(np.arange(npages, npages + pages, dtype=np.int32))
        npages += pages
    width = max(len(t) for t in tables)
    bt = np.full((len(tables), width), -1, dtype=np.int32)
    for r, t in enumerate(tables):
        bt[r, :len(t)] = t
    return np.concatenate(rows), np.concatenate(scales), bt


def _oracle_compute(inp, w, kv, sc, bt):
    import oracle
    from dsa_sparse_mla_topk_gb300.dcp import Compute

    q_bits = inp.q.view(torch.int16).numpy()
    q_req = inp.q_req.numpy()

    def topk(scores, q_pos, k):
        s, qp = scores.numpy(), q_pos.numpy()
        out = np.full((s.shape[0], k), -1, dtype=np.int32)
        rows = np.nonzero(qp >= 0)[0]
        if len(rows):
            out[rows] = oracle.topk(s[rows], qp[rows], k)
        return torch.from_numpy(out)

    def partial(idx):
        _, _, op, lp = oracle.sparse_mla(q_bits, kv, sc, bt, q_req, idx.numpy(), d_latent=w.d_latent,
                                         d_rope=w.d_rope, page_size=w.page_size, softmax_scale=w.scale,
                                         num_splits=2, return_partials=True)
        return torch.from_numpy(op), torch.from_numpy(lp)

    def combine(op, lp):
        out, lse = oracle.combine(op.numpy(), lp.numpy())
        return torch.from_numpy(out), torch.from_numpy(lse)

    return Compute(topk, partial, combine)


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from dsa_sparse_mla_topk_gb300 import dcp
    from dsa_sparse_mla_topk_gb300 import workloads as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _workload()
        inp = wl.make_inputs(w, device="cpu", keep_logical=True)
        kv, sc, bt = _local_pool(inp, w, rank, world)
        cols = dcp.owned_positions(inp.scores.shape[1], rank, world)
        scores_local = inp.scores[:, cols].contiguous()
        out, lse, idx = dcp.dcp_sparse_mla_topk(scores_local, inp.q_pos, w.k, _oracle_compute(inp, w, kv, sc, bt))
        results[rank] = (out.numpy(), lse.numpy(), idx.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dcp_matches_the_single_rank_result(world):
    import oracle
    from dsa_sparse_mla_topk_gb300 import workloads as wl
    oracle.build()
    w = _workload()
    inp = wl.make_inputs(w, device="cpu")
    ref_idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), w.k)
    ref_out, ref_lse = oracle.sparse_mla(inp.q.view(torch.int16).numpy(), inp.kv.numpy(), inp.kv_scale.numpy(),
                                         inp.block_table.numpy(), inp.q_req.numpy(), ref_idx, d_latent=w.d_latent,
                                         d_rope=w.d_rope, page_size=w.page_size, softmax_scale=w.scale)
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, start_method="spawn",
                           join=True)
        got = dict(results)
    assert sorted(got) == list(range(world))
    for r in range(world):
        out, lse, idx = got[r]
        assert np.array_equal(idx, ref_idx)
        np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_local_views():
    sys.path.insert(0, ROOT)
    from dsa_sparse_mla_topk_gb300 import dcp
    assert dcp.owned_positions(10, 1, 3).tolist() == [1, 4, 7]
    qp = torch.tensor([0, 1, 2, 5, 6], dtype=torch.int32)
    assert dcp.local_q_pos(qp, 0, 3).tolist() == [0, 0, 0, 1, 2]
    assert dcp.local_q_pos(qp, 2, 3).tolist() == [-1, -1, 0, 1, 1]
