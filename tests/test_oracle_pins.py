"""Pins of the fp64 oracle against things other than itself.

Each test ties one part of the oracle to a library routine on a special
case, a closed form, brute force, an invariant the method must satisfy, or a
hand-written fixture.  A plausible slip in the oracle (a dropped scale, a
wrong page or row index, the wrong operand half for V, a wrong tie rule, a
wrong merge weight) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_topk_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- number formats --------------------------------------------------------

def test_e4m3_all_256_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.signbit(got[0x80]) and not np.signbit(got[0])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(512, generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_to_double(b) for b in bits])
    assert np.array_equal(got, x.to(torch.float64).numpy())


# ---- top-k ----------------------------------------------------------------

def _lexsort_topk(scores, q_pos, k):
    """Library special case: numpy's lexsort by (-score, position)."""
    out = np.full((scores.shape[0], k), -1, dtype=np.int32)
    for i, p in enumerate(q_pos):
        vis = p + 1
        s = scores[i, :vis].astype(np.float64)
        order = np.lexsort((np.arange(vis), -s))[: min(k, vis)]
        sel = np.sort(order)
        out[i, : len(sel)] = sel
    return out


@pytest.mark.parametrize("k", [1, 3, 8, 17, 64])
def test_topk_brute_force_with_many_ties(k):
    rng = np.random.default_rng(k)
    n, ld = 24, 97
    # small integer scores -> heavy ties, incl. signed zeros
    scores = rng.integers(-4, 5, size=(n, ld)).astype(np.float32)
    scores[rng.random((n, ld)) < 0.1] = -0.0
    q_pos = rng.integers(0, ld, size=n).astype(np.int32)
    got = oracle.topk(scores, q_pos, k)
    assert np.array_equal(got, _lexsort_topk(scores, q_pos, k))


def test_topk_random_floats_match_sort():
    rng = np.random.default_rng(1)
    scores = rng.standard_normal((8, 5000)).astype(np.float32)
    q_pos = np.array([4999, 4000, 2047, 2048, 100, 0, 3333, 4998], dtype=np.int32)
    got = oracle.topk(scores, q_pos, 2048)
    assert np.array_equal(got, _lexsort_topk(scores, q_pos, 2048))


def _golden_topk_cases():
    cases = []
    with open(os.path.join(GOLDEN, "topk_ties.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, qp, k, sc, exp = [t.strip() for t in line.split("|")]
            cases.append((name, int(qp), int(k), [float(v) for v in sc.split(",")], [int(v) for v in exp.split(",")]))
    return cases


@pytest.mark.parametrize("case", _golden_topk_cases(), ids=lambda c: c[0])
def test_topk_golden(case):
    name, qp, k, sc, exp = case
    got = oracle.topk(np.array([sc], dtype=np.float32), np.array([qp], dtype=np.int32), k)
    assert got[0].tolist() == exp


def test_topk_k_at_least_visible_is_all_positions():
    rng = np.random.default_rng(3)
    scores = rng.standard_normal((3, 50)).astype(np.float32)
    got = oracle.topk(scores, np.array([9, 49, 0], dtype=np.int32), 64)
    assert got[0].tolist() == list(range(10)) + [-1] * 54
    assert got[1].tolist() == list(range(50)) + [-1] * 14
    assert got[2].tolist() == [0] + [-1] * 63


# ---- attention ---------------------------------------------------------------

def _tiny(**kw):
    base = dict(num_req=3, q_per_req=2, heads=4, d_latent=16, d_rope=8, ctx=40, shared_prefix=20, page_size=8,
                k=64, seed=11, softmax_scale=0.3)
    base.update(kw)
    return wl.Workload("pin", **base)


def _run_oracle(inp, idx, splits=1, **kw):
    w = inp.w
    return oracle.sparse_mla(inp.q.view(torch.int16).numpy(), inp.kv.numpy(), inp.kv_scale.numpy(),
                             inp.block_table.numpy(), inp.q_req.numpy(), idx, d_latent=w.d_latent,
                             d_rope=w.d_rope, page_size=w.page_size, softmax_scale=w.scale, num_splits=splits, **kw)


def _logical_k(inp, r):
    """Dequantised rows of request r in position order, decoded by torch."""
    b, s = inp.logical[r]
    return b.view(torch.float8_e4m3fn).to(torch.float64) * s.to(torch.float64)[:, None]


def test_dense_case_matches_torch_sdpa():
    """k >= visible: sparse attention is dense causal attention (torch SDPA, fp64)."""
    w = _tiny()
    inp = wl.make_inputs(w, keep_logical=True)
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), w.k)
    out, lse = _run_oracle(inp, idx)
    for i in range(w.num_q):
        r, p = int(inp.q_req[i]), int(inp.q_pos[i])
        K = _logical_k(inp, r)[: p + 1]
        V = K[:, : w.d_latent]
        q = inp.q[i].to(torch.float64)  # [H, dqk]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :], K[None, None].expand(1, w.heads, -1, -1), V[None, None].expand(1, w.heads, -1, -1),
            scale=w.scale)[0, :, 0, :]
        ref_lse = torch.logsumexp((q @ K.T) * w.scale, dim=-1)
        np.testing.assert_allclose(out[i], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[i], ref_lse.numpy(), rtol=0, atol=1e-12)


def test_k_equals_one_returns_the_value_row():
    """One selected row: softmax weight 1, O is that row's latent part exactly."""
    w = _tiny(k=1)
    inp = wl.make_inputs(w, keep_logical=True)
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), 1)
    out, lse = _run_oracle(inp, idx)
    for i in range(w.num_q):
        r = int(inp.q_req[i])
        x = _logical_k(inp, r)[int(idx[i, 0])]
        for h in range(w.heads):
            assert np.array_equal(out[i, h], x[: w.d_latent].numpy())
        z = (inp.q[i].to(torch.float64) @ x) * w.scale
        np.testing.assert_allclose(lse[i], z.numpy(), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_values():
    """All logits equal: O = mean of the selected V rows, lse = ln n."""
    w = _tiny()
    inp = wl.make_inputs(w, keep_logical=True)
    inp.q.zero_()
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), 16)
    out, lse = _run_oracle(inp, idx)
    for i in range(w.num_q):
        r = int(inp.q_req[i])
        sel = idx[i][idx[i] >= 0]
        mean = _logical_k(inp, r)[sel][:, : w.d_latent].mean(0).numpy()
        for h in range(w.heads):
            np.testing.assert_allclose(out[i, h], mean, rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[i], math.log(len(sel)), rtol=0, atol=1e-14)


def test_empty_selection_gives_zero_and_minus_inf():
    w = _tiny()
    inp = wl.make_inputs(w)
    idx = np.full((w.num_q, 8), -1, dtype=np.int32)
    out, lse = _run_oracle(inp, idx)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_permuting_selected_indices_changes_nothing():
    w = _tiny()
    inp = wl.make_inputs(w)
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), 12)
    rng = np.random.default_rng(5)
    perm = np.stack([rng.permutation(idx.shape[1]) for _ in range(idx.shape[0])])
    idx2 = np.take_along_axis(idx, perm, axis=1)
    a, la = _run_oracle(inp, idx)
    b, lb = _run_oracle(inp, idx2)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-12)


def test_shared_prefix_pages_equal_copied_pages():
    """The same logical rows through shared pages or per-request copies give
    bit-identical results (page indirection only relocates rows)."""
    w = _tiny(shared_prefix=27)
    a = wl.make_inputs(w, keep_logical=True)
    b = wl.make_inputs(wl.shrink(w, share_pages=False), keep_logical=True)
    assert a.layout.n_shared_pages == 3 and b.layout.n_shared_pages == 0
    assert a.kv.shape[0] < b.kv.shape[0]
    for r in range(w.num_req):
        assert torch.equal(a.logical[r][0], b.logical[r][0])
    idx = oracle.topk(a.scores.numpy(), a.q_pos.numpy(), 24)
    oa, la = _run_oracle(a, idx)
    ob, lb = _run_oracle(b, idx)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


@pytest.mark.parametrize("splits", [2, 3, 7, 16])
def test_split_count_invariance_and_combine(splits):
    w = _tiny(ctx=90, shared_prefix=0, k=50)
    inp = wl.make_inputs(w)
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), w.k)
    o1, l1 = _run_oracle(inp, idx)
    oS, lS, op, lp = _run_oracle(inp, idx, splits=splits, return_partials=True)
    np.testing.assert_allclose(oS, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lS, l1, rtol=0, atol=1e-12)
    oc, lc = oracle.combine(op, lp)
    np.testing.assert_allclose(oc, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lc, l1, rtol=0, atol=1e-12)
    # with fewer rows than splits some chunks are empty: their partial is
    # (0, -inf) and the merge ignores it
    few = idx[:, :5]
    o5, l5 = _run_oracle(inp, few)
    o5S, l5S, op5, lp5 = _run_oracle(inp, few, splits=splits, return_partials=True)
    assert np.isneginf(lp5).any() == (splits > 5)
    assert np.all(op5[np.isneginf(lp5)] == 0)
    np.testing.assert_allclose(o5S, o5, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l5S, l5, rtol=0, atol=1e-12)


def test_page_indirection_is_used():
    """Moving a page's rows to another page id and updating the block table
    leaves the result unchanged; not updating it changes the result."""
    w = _tiny(shared_prefix=0)
    inp = wl.make_inputs(w)
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), 30)
    base, _ = _run_oracle(inp, idx)
    P = w.page_size
    bt = inp.block_table.numpy().copy()
    kv = inp.kv.numpy().copy()
    sc = inp.kv_scale.numpy().copy()
    pa, pb = int(bt[0, 1]), int(bt[1, 2])
    for arr in (kv, sc):
        tmp = arr[pa * P:(pa + 1) * P].copy()
        arr[pa * P:(pa + 1) * P] = arr[pb * P:(pb + 1) * P]
        arr[pb * P:(pb + 1) * P] = tmp
    kw = dict(d_latent=w.d_latent, d_rope=w.d_rope, page_size=P, softmax_scale=w.scale)
    q = inp.q.view(torch.int16).numpy()
    stale, _ = oracle.sparse_mla(q, kv, sc, bt, inp.q_req.numpy(), idx, **kw)
    bt[0, 1], bt[1, 2] = pb, pa
    fixed, _ = oracle.sparse_mla(q, kv, sc, bt, inp.q_req.numpy(), idx, **kw)
    assert np.array_equal(fixed, base)
    assert not np.allclose(stale, base)


def test_bad_index_and_page_are_reported():
    w = _tiny(shared_prefix=0)
    inp = wl.make_inputs(w)
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), 8)
    idx[0, 0] = -5
    with pytest.raises(ValueError):
        _run_oracle(inp, idx)
    bt = inp.block_table.numpy().copy()
    bt[:, 0] = 10 ** 6
    idx = oracle.topk(inp.scores.numpy(), inp.q_pos.numpy(), 40)
    with pytest.raises(ValueError):
        oracle.sparse_mla(inp.q.view(torch.int16).numpy(), inp.kv.numpy(), inp.kv_scale.numpy(), bt,
                          inp.q_req.numpy(), idx, d_latent=w.d_latent, d_rope=w.d_rope, page_size=w.page_size,
                          softmax_scale=w.scale)


# ---- KV cache write path: FP8 E4M3 encoding and paged scatter ----

def _e4m3_grid():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    ok = np.isfinite(vals)
    return codes[ok], vals[ok]


def test_e4m3_encode_matches_torch_on_grid_ties_and_random_values():
    """The encoder against torch's float8_e4m3fn cast (round to nearest even):
    every grid value, every midpoint between neighbours (ties), points just off
    the midpoints, and random values across the whole range."""
    _, vals = _e4m3_grid()
    pos = np.unique(vals[vals >= 0]).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(5)
    rand = np.concatenate([rng.uniform(-448, 448, 4000), rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000),
                           np.exp2(rng.uniform(-12, 8.8, 4000)) * rng.choice([-1, 1], 4000)])
    xs = np.concatenate([pos, -pos, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1000), rand])
    xs = xs[np.abs(xs) <= 448].astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in xs], dtype=np.uint8)
    # +0.0 and -0.0 both encode to a zero of their own sign in both
    assert np.array_equal(got, want)


def test_e4m3_encode_saturates_and_keeps_sign():
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(-448.0) == 0xFE
    assert oracle.e4m3_encode(464.0) == 0x7E and oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-3.4e38) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00 and oracle.e4m3_encode(-(2.0 ** -10)) == 0x80
    assert oracle.e4m3_encode(1.0) == 0x38 and oracle.e4m3_encode(-1.0) == 0xB8


def _rows_bf16(n, d, seed, spread=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, d), generator=g)
    if spread:  # per-row magnitudes from 2^-20 to 2^20
        x = x * torch.exp2(torch.randint(-20, 21, (n, 1), generator=g).float())
    return x.to(torch.bfloat16)


def test_kv_write_matches_an_independent_torch_quantiser():
    """Per-token quantisation (scale = max|x|/448, bytes = RNE(x/scale) on the
    E4M3 grid) against the input generator's torch implementation, on rows of
    very different magnitudes; identity block table."""
    n, d, P = 96, 576, 32
    x = _rows_bf16(n, d, 11, spread=True)
    want_b, want_s = wl.quantize_rows(x.float())
    kv = np.zeros((n, d), dtype=np.uint8)
    sc = np.zeros(n, dtype=np.float32)
    bt = np.arange(n // P, dtype=np.int32)[None, :]
    st = oracle.kv_write(x.view(torch.int16).numpy(), np.zeros(n, np.int32), np.arange(n, dtype=np.int32), bt, kv,
                         sc, page_size=P)
    assert st == oracle.OK
    assert np.array_equal(sc, want_s.numpy())
    assert np.array_equal(kv, want_b.numpy())


def test_kv_write_dequantises_within_half_a_step():
    """Dequantised values lie within half an E4M3 step (relative 2^-4, or the
    subnormal step) of the bf16 inputs, and the row maximum is exact."""
    n, d, P = 16, 80, 16
    x = _rows_bf16(n, d, 12)
    kv = np.zeros((n, d), dtype=np.uint8)
    sc = np.zeros(n, dtype=np.float32)
    oracle.kv_write(x.view(torch.int16).numpy(), np.zeros(n, np.int32), np.arange(n, dtype=np.int32),
                    np.arange(1, dtype=np.int32)[None, :], kv, sc, page_size=P)
    deq = np.array([[oracle.e4m3_to_double(b) for b in row] for row in kv]) * sc[:, None].astype(np.float64)
    xv = x.double().numpy()
    step = np.maximum(np.abs(xv) * 2.0 ** -4, sc[:, None] * 2.0 ** -10)
    assert np.all(np.abs(deq - xv) <= step * (1 + 1e-6))
    amax_rows = np.argmax(np.abs(xv), axis=1)
    assert np.allclose(np.abs(deq[np.arange(n), amax_rows]), np.abs(xv[np.arange(n), amax_rows]), rtol=1e-6)


def test_kv_write_scatters_through_the_block_table():
    """Rows land at block_table[req][pos // P] * P + pos % P and nowhere else;
    a zero row stores scale 0 and zero bytes; bad requests, positions and pages
    are flagged and skipped."""
    P, d = 8, 32
    bt = np.array([[5, 2, 7], [1, 6, 0]], dtype=np.int32)  # 8 pages
    req = np.array([0, 0, 1, 1, 1, 0, 2, 1], dtype=np.int32)
    pos = np.array([0, 13, 23, 9, 5, 30, 1, -1], dtype=np.int32)
    x = _rows_bf16(len(req), d, 13)
    x[4] = 0
    kv = np.full((8 * P, d), 0xAA, dtype=np.uint8)
    sc = np.full(8 * P, -1.0, dtype=np.float32)
    st = oracle.kv_write(x.view(torch.int16).numpy(), req, pos, bt, kv, sc, page_size=P)
    assert st == oracle.BAD_INDEX | oracle.BAD_PAGE  # pos 30 past the table and -1; request 2
    written = {}
    for i in range(5):
        slot = int(bt[req[i], pos[i] // P]) * P + int(pos[i]) % P
        written[slot] = i
        want_b, want_s = wl.quantize_rows(x[i:i + 1].float())
        if i == 4:
            assert sc[slot] == 0.0 and not kv[slot].any()
        else:
            assert sc[slot] == want_s.item() and np.array_equal(kv[slot], want_b.numpy()[0])
    untouched = np.array([s for s in range(8 * P) if s not in written])
    assert np.all(sc[untouched] == -1.0) and np.all(kv[untouched] == 0xAA)
    bad_page = np.array([[9]], dtype=np.int32)
    st = oracle.kv_write(x[:1].view(torch.int16).numpy(), np.zeros(1, np.int32), np.zeros(1, np.int32), bad_page,
                         kv, sc, page_size=P)
    assert st == oracle.BAD_PAGE


def test_topk_of_slice_topks_is_the_row_topk():
    """The sliced top-k for long rows keeps each fixed-size slice's own top k
    (score, position) in position order, concatenates the blocks in slice
    order, and takes the top k of that union; union order is position order,
    so the lower-index tie rule there is the lower-position rule.  Checked
    with the oracle alone: slices shorter than k, empty slices, and exact
    ties across slice boundaries must give the row's own top k."""
    rng = np.random.default_rng(17)
    slice_len, k = 96, 40
    ld = 5 * slice_len + 17
    scores = rng.standard_normal((6, ld)).astype(np.float32)
    scores[1] = rng.integers(0, 3, ld).astype(np.float32)          # heavy ties everywhere
    scores[2, 90:110] = 7.0                                        # a tie run across a slice edge
    scores[3, slice_len * 3:] += 5.0                               # the top k all in late slices
    q_pos = np.array([ld - 1, ld - 1, ld - 1, ld - 1, slice_len + 3, 2 * slice_len - 1], dtype=np.int32)
    want = oracle.topk(scores, q_pos, k)
    nsl = (ld + slice_len - 1) // slice_len
    for r in range(scores.shape[0]):
        vis = int(q_pos[r]) + 1
        blk_score, blk_pos = [], []
        for sl in range(nsl):
            lo = sl * slice_len
            n = max(0, min(vis - lo, slice_len))
            if n == 0:
                continue
            part = scores[r:r + 1, lo:lo + n]
            sel = oracle.topk(part, np.array([n - 1], dtype=np.int32), k)[0]
            sel = sel[sel >= 0]
            blk_score.append(part[0, sel])
            blk_pos.append(lo + sel)
        union_s = np.concatenate(blk_score)[None, :]
        union_p = np.concatenate(blk_pos)
        assert (np.diff(union_p) > 0).all()                        # union order is position order
        pick = oracle.topk(union_s, np.array([union_s.shape[1] - 1], dtype=np.int32), k)[0]
        got = np.where(pick >= 0, union_p[np.maximum(pick, 0)], -1)
        assert np.array_equal(got, want[r]), r
