"""The attention entry point that allocates nothing.

Callers that may not allocate device memory while they run a step -- serving
loops that reserve all device memory at start-up and forbid later
allocations, or plug-in hosts that give the library no allocator -- call
dsa_sparse_mla_fwd_noalloc, whose scratch is a fixed array inside the
library.  This test calls it through the C ABI and compares it with the
regular dsa_sparse_mla_fwd (caller-provided workspace) on two calls in a
row, the second reusing the scratch the first left behind.  It sits in its
own file so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import dsa_sparse_mla_topk_gb300 as dsa
from dsa_sparse_mla_topk_gb300 import workloads as wl

MAX_ABS, REL_L2, LSE_ABS = 1e-2, 5e-3, 1e-3


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, inp, idx, out, lse, status):
    w = inp.w
    return lib.dsa_sparse_mla_fwd_noalloc(
        _p(inp.q), _p(inp.kv), _p(inp.kv_scale), inp.kv.shape[0] // w.page_size, _p(inp.block_table),
        inp.block_table.shape[0], inp.block_table.shape[1], _p(inp.q_req), _p(idx), w.num_q, w.heads, w.d_latent,
        w.d_rope, w.page_size, idx.shape[1], w.scale, 1, _p(out), _p(lse), None, None, _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
def test_noalloc_entry_point_matches_workspace_entry_point_on_two_calls():
    from dsa_sparse_mla_topk_gb300 import build
    build.build()
    lib = dsa.load_library()
    cases = [wl.Workload("noalloc_a", 3, 3, 64, 512, 64, 3000, 0, 64, 2048, seed=41, ctx_per_req=(3000, 2101, 700)),
             wl.Workload("noalloc_b", 8, 2, 64, 512, 64, 9000, 8000, 64, 2048, seed=42)]
    for w in cases:
        inp = wl.make_inputs(w, device="cuda")
        idx = dsa.topk_select(inp.scores, inp.q_pos, w.k)
        ref_out, ref_lse = dsa.sparse_mla_fwd(inp.q, inp.kv, inp.kv_scale, inp.block_table, inp.q_req, idx,
                                              d_latent=w.d_latent, d_rope=w.d_rope, page_size=w.page_size,
                                              softmax_scale=w.scale)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, inp, idx, out, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        a = out.float().cpu().numpy().astype(np.float64)
        b = ref_out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all()
        assert float(np.abs(a - b).max()) <= MAX_ABS
        assert float(np.linalg.norm(a - b) / np.linalg.norm(b)) <= REL_L2
        assert float((lse - ref_lse).abs().max().item()) <= LSE_ABS


@pytest.mark.gpu
def test_noalloc_entry_point_rejects_calls_beyond_its_scratch():
    lib = dsa.load_library()
    fake = ctypes.c_void_p(0x10000)
    # 4096 query tokens at top-k 2048 need 64 MiB of scratch: rejected before any launch
    st = lib.dsa_sparse_mla_fwd_noalloc(fake, fake, fake, 4, fake, 1, 4, fake, fake, 4096, 64, 512, 64, 64, 2048,
                                        0.04, 1, fake, fake, None, None, None, None)
    assert st == 3  # DSA_ERR_WORKSPACE_TOO_SMALL
    st = lib.dsa_sparse_mla_fwd_noalloc(fake, fake, fake, 4, fake, 1, 4, fake, fake, 1, 16, 64, 16, 16, 64, 0.1, 1,
                                        fake, fake, None, None, None, None)
    assert st == 2  # only the tensor-core shape
