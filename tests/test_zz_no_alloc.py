"""The attention entry point that allocates nothing.

Callers that may not allocate device memory while they run a step -- serving
loops that reserve all device memory at start-up and forbid later
allocations, or plug-in hosts that give the library no allocator -- call
dsa_sparse_mla_fwd_noalloc, whose scratch is a fixed array inside the
library.  These tests call it through the C ABI and compare it with the
regular dsa_sparse_mla_fwd (caller-provided workspace) on two calls in a
row, the second reusing the scratch the first left behind.  Both entry
points run the same kernels on the same inputs, so their results must agree
bit for bit; one call is also checked against the fp64 oracle.  The file
sits on its own so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import dsa_sparse_mla_topk_gb300 as dsa
from dsa_sparse_mla_topk_gb300 import workloads as wl

MAX_ABS, REL_L2, LSE_ABS = 1e-2, 5e-3, 1e-3


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, inp, idx, status, splits, out=None, lse=None, o_part=None, lse_part=None):
    w = inp.w
    return lib.dsa_sparse_mla_fwd_noalloc(
        _p(inp.q), _p(inp.kv), _p(inp.kv_scale), inp.kv.shape[0] // w.page_size, _p(inp.block_table),
        inp.block_table.shape[0], inp.block_table.shape[1], _p(inp.q_req), _p(idx), w.num_q, w.heads, w.d_latent,
        w.d_rope, w.page_size, idx.shape[1], w.scale, splits, _p(out), _p(lse), _p(o_part), _p(lse_part),
        _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [wl.Workload("noalloc_a", 3, 3, 64, 512, 64, 3000, 0, 64, 2048, seed=41, ctx_per_req=(3000, 2101, 700)),
         wl.Workload("noalloc_b", 8, 2, 64, 512, 64, 9000, 8000, 64, 2048, seed=42)]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_entry_point_matches_workspace_entry_point_on_two_calls(w):
    from dsa_sparse_mla_topk_gb300 import build
    build.build()
    lib = dsa.load_library()
    inp = wl.make_inputs(w, device="cuda")
    idx = dsa.topk_select(inp.scores, inp.q_pos, w.k)
    kw = dict(d_latent=w.d_latent, d_rope=w.d_rope, page_size=w.page_size, softmax_scale=w.scale)
    ref_out, ref_lse = dsa.sparse_mla_fwd(inp.q, inp.kv, inp.kv_scale, inp.block_table, inp.q_req, idx, **kw)
    ref_op, ref_lp = dsa.sparse_mla_fwd(inp.q, inp.kv, inp.kv_scale, inp.block_table, inp.q_req, idx, num_splits=2,
                                        **kw)
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):  # the second call finds the first call's scratch contents
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(lib, inp, idx, status, 1, out=out, lse=lse) == 0
        op = torch.full_like(ref_op, float("nan"))
        lp = torch.full_like(ref_lp, float("nan"))
        assert _noalloc(lib, inp, idx, status, 2, o_part=op, lse_part=lp) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), f"call {call}: unsplit result differs"
        assert torch.equal(op, ref_op) and torch.equal(lp, ref_lp), f"call {call}: split partials differ"
    # and against the fp64 oracle, through the Combine of the split call
    c_out, c_lse = dsa.combine(op, lp)
    torch.cuda.synchronize()
    host = lambda t: t.detach().cpu().numpy()
    ref_idx = oracle.topk(host(inp.scores), host(inp.q_pos), w.k)
    assert np.array_equal(host(idx), ref_idx)
    o_ref, l_ref = oracle.sparse_mla(host(inp.q.view(torch.int16)), host(inp.kv), host(inp.kv_scale),
                                     host(inp.block_table), host(inp.q_req), ref_idx, **kw)
    for got_o, got_l in ((out, lse), (c_out, c_lse)):
        a = host(got_o.float()).astype(np.float64)
        assert float(np.abs(a - o_ref).max()) <= MAX_ABS
        assert float(np.linalg.norm(a - o_ref) / np.linalg.norm(o_ref)) <= REL_L2
        assert float(np.abs(host(got_l) - l_ref).max()) <= LSE_ABS


@pytest.mark.gpu
def test_noalloc_entry_point_rejects_calls_beyond_its_scratch():
    """Size and shape checks return before anything is launched.  Every
    pointer is NULL: should the checks ever be reordered, the regular entry
    point's own NULL checks still stop the call before a launch."""
    from dsa_sparse_mla_topk_gb300 import build
    build.build()
    lib = dsa.load_library()
    # 4096 query tokens at top-k 2048 need more scratch than the fixed array holds
    st = lib.dsa_sparse_mla_fwd_noalloc(None, None, None, 4, None, 1, 4, None, None, 4096, 64, 512, 64, 64, 2048,
                                        0.04, 1, None, None, None, None, None, None)
    assert st == 3  # DSA_ERR_WORKSPACE_TOO_SMALL
    st = lib.dsa_sparse_mla_fwd_noalloc(None, None, None, 4, None, 1, 4, None, None, 1, 16, 64, 16, 16, 64, 0.1, 1,
                                        None, None, None, None, None, None)
    assert st == 2  # only the tensor-core shape
