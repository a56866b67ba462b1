"""GPU parity of the KV cache write path (dsa_kv_write) against the oracle.

The FP8 codes and the per-token scales are integers and exact fp32 values
decided in fp32 on both sides, so the comparison is bit for bit.  The last
test writes a whole pool through the C ABI and runs the attention path over
it against the oracle on the oracle-written pool.
"""
import numpy as np
import pytest
import torch

import oracle
import dsa_sparse_mla_topk_gb300 as dsa
from dsa_sparse_mla_topk_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dsa_sparse_mla_topk_gb300 import build
    build.build()
    dsa.load_library()


def _rows(n, d, seed):
    """bf16 rows: N(0,1) with per-row magnitudes 2^-20..2^20, plus special rows."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, d), generator=g) * torch.exp2(torch.randint(-20, 21, (n, 1), generator=g).float())
    x[0] = 0.0                                   # all zero: scale 0, zero bytes
    x[1] = -0.0                                  # negative zeros
    x[2, :] = 1e-3
    x[2, 0] = 1e3                                # one large value: the rest fall to subnormal codes
    x[3] = torch.linspace(-1.0, 1.0, d)          # dense grid, many ties after scaling
    return x.to(torch.bfloat16)


def _layout(n_pages, page, num_req, seed):
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_pages, generator=g).to(torch.int32)
    per = n_pages // num_req
    return perm[: per * num_req].view(num_req, per).contiguous()


@pytest.mark.parametrize("d,page", [(576, 64), (80, 16)])
def test_kv_write_bit_exact_against_oracle(d, page):
    num_req, n_pages = 4, 32
    bt = _layout(n_pages, page, num_req, seed=d)
    per = bt.shape[1] * page
    g = torch.Generator().manual_seed(7)
    n = 300
    req = torch.randint(0, num_req, (n,), generator=g, dtype=torch.int32)
    # distinct (req, pos) pairs so that no two rows aim at the same slot
    pairs = torch.randperm(num_req * per, generator=g)[:n]
    req, pos = (pairs // per).to(torch.int32), (pairs % per).to(torch.int32)
    x = _rows(n, d, seed=d + 1)
    slots = n_pages * page
    kv = torch.full((slots, d), 0xAA, dtype=torch.uint8, device="cuda")
    sc = torch.full((slots,), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.kv_write(x.cuda(), req.cuda(), pos.cuda(), bt.cuda(), kv, sc, page_size=page, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kv_ref = np.full((slots, d), 0xAA, dtype=np.uint8)
    sc_ref = np.full(slots, -1.0, dtype=np.float32)
    assert oracle.kv_write(x.view(torch.int16).numpy(), req.numpy(), pos.numpy(), bt.numpy(), kv_ref, sc_ref,
                           page_size=page) == oracle.OK
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(kv.cpu().numpy(), kv_ref)


def test_kv_write_flags_and_skips_bad_rows():
    d, page = 576, 64
    bt = torch.tensor([[3, 1], [0, 9]], dtype=torch.int32)  # page 9 does not exist (4 pages)
    req = torch.tensor([0, 0, 1, 2, 1, 0, -1], dtype=torch.int32)
    pos = torch.tensor([5, 130, 70, 0, 3, -2, 0], dtype=torch.int32)
    x = _rows(len(req), d, seed=3)
    kv = torch.full((4 * page, d), 0xAA, dtype=torch.uint8, device="cuda")
    sc = torch.full((4 * page,), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.kv_write(x.cuda(), req.cuda(), pos.cuda(), bt.cuda(), kv, sc, page_size=page, dev_status=status)
    torch.cuda.synchronize()
    kv_ref = np.full((4 * page, d), 0xAA, dtype=np.uint8)
    sc_ref = np.full(4 * page, -1.0, dtype=np.float32)
    st_ref = oracle.kv_write(x.view(torch.int16).numpy(), req.numpy(), pos.numpy(), bt.numpy(), kv_ref, sc_ref,
                             page_size=page)
    assert int(status.item()) == st_ref == dsa.DEV_BAD_INDEX | dsa.DEV_BAD_PAGE
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(kv.cpu().numpy(), kv_ref)


def test_written_pool_feeds_the_attention_path():
    """Write every KV row of a small multi-request workload through
    dsa_kv_write, then run top-k + attention over the GPU-written pool and
    compare with the oracle over the oracle-written pool."""
    w = wl.Workload("kvw_roundtrip", 3, 2, 64, 512, 64, 1200, 0, 64, 256, seed=23)
    inp = wl.make_inputs(w, device="cuda")
    bt = inp.block_table
    num_req, per = bt.shape[0], bt.shape[1] * w.page_size
    g = torch.Generator().manual_seed(29)
    x = (torch.randn((num_req * per, w.dqk), generator=g) * 0.5).to(torch.bfloat16)
    req = torch.arange(num_req, dtype=torch.int32).repeat_interleave(per)
    pos = torch.arange(per, dtype=torch.int32).repeat(num_req)
    kv = torch.zeros_like(inp.kv)
    sc = torch.zeros_like(inp.kv_scale)
    dsa.kv_write(x.cuda(), req.cuda(), pos.cuda(), bt, kv, sc, page_size=w.page_size)
    kv_ref = np.zeros(tuple(inp.kv.shape), dtype=np.uint8)
    sc_ref = np.zeros(tuple(inp.kv_scale.shape), dtype=np.float32)
    oracle.kv_write(x.view(torch.int16).numpy(), req.numpy(), pos.numpy(), bt.cpu().numpy(), kv_ref, sc_ref,
                    page_size=w.page_size)
    torch.cuda.synchronize()
    assert np.array_equal(kv.cpu().numpy(), kv_ref)
    out, lse, idx = dsa.sparse_mla_topk(inp.q, kv, sc, bt, inp.q_req, inp.q_pos, inp.scores, w.k,
                                        d_latent=w.d_latent, d_rope=w.d_rope, page_size=w.page_size,
                                        softmax_scale=w.scale)
    torch.cuda.synchronize()
    ref_idx = oracle.topk(inp.scores.cpu().numpy(), inp.q_pos.cpu().numpy(), w.k)
    ref_out, ref_lse = oracle.sparse_mla(inp.q.view(torch.int16).cpu().numpy(), kv_ref, sc_ref, bt.cpu().numpy(),
                                         inp.q_req.cpu().numpy(), ref_idx, d_latent=w.d_latent, d_rope=w.d_rope,
                                         page_size=w.page_size, softmax_scale=w.scale)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    got = out.float().cpu().numpy().astype(np.float64)
    assert float(np.abs(got - ref_out).max()) <= 1e-2
    assert float(np.linalg.norm(got - ref_out) / np.linalg.norm(ref_out)) <= 5e-3
    assert float(np.abs(lse.cpu().numpy() - ref_lse).max()) <= 1e-3


def test_kv_write_every_bf16_value_under_many_row_maxima():
    """Every finite bf16 value x is quantised under row maxima a >= |x| from
    every binade (three mantissas each, and three subnormal maxima): the
    codes and scales must equal the oracle's, whose divisions are IEEE fp32.
    This covers the kernel's reciprocal-and-correction quotient and its
    division fallback for tiny maxima, at the boundaries where either could
    round differently."""
    d, page = 576, 64
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    maxima = [(e << 7) | m for e in range(1, 255) for m in (0x00, 0x45, 0x7F)] + [0x0001, 0x0040, 0x007F]
    rows = []
    for ab in maxima:
        a = np.float32((np.uint32(ab) << 16).view(np.float32))
        xs = bits[finite & (np.abs(vals) <= a)].astype(np.uint16)
        per = d - 1
        for s in range(0, len(xs), per):
            row = np.full(d, ab, dtype=np.uint16)  # the row's maximum first, and as padding
            chunk = xs[s:s + per]
            row[1:1 + len(chunk)] = chunk
            rows.append(row)
    x_bits = np.stack(rows)
    n = x_bits.shape[0]
    pages = (n + page - 1) // page
    bt = torch.arange(pages, dtype=torch.int32)[None, :]
    req = torch.zeros(n, dtype=torch.int32)
    pos = torch.arange(n, dtype=torch.int32)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16)
    kv = torch.zeros((pages * page, d), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((pages * page,), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.kv_write(x.cuda(), req.cuda(), pos.cuda(), bt.cuda(), kv, sc, page_size=page, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kv_ref = np.zeros((pages * page, d), dtype=np.uint8)
    sc_ref = np.zeros(pages * page, dtype=np.float32)
    assert oracle.kv_write(x_bits.view(np.int16), req.numpy(), pos.numpy(), bt.numpy(), kv_ref, sc_ref,
                           page_size=page) == oracle.OK
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(kv.cpu().numpy(), kv_ref)
