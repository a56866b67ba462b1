"""Host-side layout checks of the synthetic workloads (no GPU)."""
import torch

from dsa_sparse_mla_topk_gb300 import workloads as wl


def test_prefix_sharing_slot_formula_when_page_aligned():
    """N requests sharing a page-aligned prefix Lp, each with suffix Ls, occupy
    Lp + N*Ls slots instead of N*(Lp+Ls) ("Accelerating GLM-5.3-Flash on H200",
    section 2, "KV-only decode RadixCache")."""
    Lp, Ls, N, P = 1024, 128, 4, 64
    w = wl.Workload("t", N, 1, 4, 16, 8, Lp + Ls, Lp, P, 8, seed=0)
    assert wl.slot_count(w) == Lp + N * Ls
    assert wl.slot_count(wl.shrink(w, share_pages=False)) == N * (Lp + Ls)
    inp = wl.make_inputs(w)
    assert inp.kv.shape[0] == Lp + N * Ls


def test_decode_workload_slots_with_page_alignment():
    """65,470 shared tokens are 1022 whole pages of 64 plus a 62-token tail that
    each request copies into its own pages: 65,408 + 128 * 128 = 81,792 slots
    (the ideal Lp + N*Ls would be 73,918; unshared 8,388,608)."""
    w = wl.DECODE_64K
    assert wl.slot_count(w) == 81_792
    assert w.shared_prefix + w.num_req * (w.ctx - w.shared_prefix) == 73_918
    assert wl.slot_count(wl.shrink(w, share_pages=False)) == 128 * 65_536


def test_block_table_shares_prefix_pages_and_permutes_private_ones():
    w = wl.Workload("t", 3, 2, 4, 16, 8, 100, 37, 8, 8, seed=3)
    inp = wl.make_inputs(w)
    bt = inp.block_table
    assert torch.equal(bt[0, :4], torch.arange(4, dtype=torch.int32))
    assert torch.equal(bt[1, :4], bt[0, :4]) and torch.equal(bt[2, :4], bt[0, :4])
    private = bt[:, 4:13].flatten()
    assert sorted(private.tolist()) == list(range(4, 4 + 27))
    assert inp.q_pos.tolist() == [98, 99] * 3 and inp.q_req.tolist() == [0, 0, 1, 1, 2, 2]


def test_tiny_workload_scores_have_exact_ties():
    inp = wl.make_inputs(wl.TINY)
    for i in range(wl.TINY.num_q):
        vis = int(inp.q_pos[i]) + 1
        row = inp.scores[i, :vis]
        assert vis - torch.unique(row).numel() >= int(0.05 * vis) // 2


def test_profiling_case_is_the_verify_block_on_fewer_requests():
    """bench.py resolves workload names through workloads.lookup: the five
    measured workloads, then the smaller profiling cases of the same kernels."""
    v, v19 = wl.lookup("verify_64k_8tok"), wl.lookup("verify_64k_8tok_19req")
    assert v is wl.VERIFY_64K
    assert (v19.num_req, v19.num_q) == (19, 152)
    for f in ("q_per_req", "heads", "d_latent", "d_rope", "ctx", "shared_prefix", "page_size", "k", "seed"):
        assert getattr(v19, f) == getattr(v, f), f
    assert set(wl.WORKLOADS).isdisjoint(wl.PROFILE_CASES)
    try:
        wl.lookup("no_such_workload")
    except KeyError:
        pass
    else:
        raise AssertionError("an unknown name must raise")
