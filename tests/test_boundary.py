"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, validates arguments before touching the device, and its host-side
planning helpers follow the tiling arithmetic of the pages."""
import ctypes
import os
import re

import pytest

import dsa_sparse_mla_topk_gb300 as dsa
from dsa_sparse_mla_topk_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa.load_library()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(dsa.EXPORTED_SYMBOLS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert dsa.status_string(0) == "ok"
    for s in range(1, 5):
        assert dsa.status_string(s) not in ("ok", "unknown status")
    assert dsa.status_string(99) == "unknown status"
    assert lib.dsa_version() >= 100


def test_tile_count_worked_example(lib):
    """"Accelerating GLM-5.3-Flash on H200", Figure 4: an index width of 2112
    takes 66 tiles of 32 or 17 tiles of 128; the 128-wide tiles cover 2176
    virtual columns of which the last 64 are padding."""
    assert dsa.kv_tile_count(2112, 32) == 66
    assert dsa.kv_tile_count(2112, 128) == 17
    assert dsa.kv_tile_count(2112, 128) * 128 == 2176
    assert dsa.kv_tile_count(2112, 128) * 128 - 2112 == 64
    assert dsa.kv_tile_count(0, 64) == 0
    assert dsa.kv_tile_count(5, 0) == -1


def test_split_rule(lib):
    """Splits only when query tokens alone leave SMs idle and splitting
    shortens the launch; never more splits than KV tiles."""
    tile = dsa.kv_tile_size(64, 512, 64)
    assert tile == 64 and dsa.kv_tile_size(16, 64, 16) == 32 and dsa.kv_tile_size(32, 512, 64) == -1
    ntiles = dsa.kv_tile_count(2048, tile)
    assert dsa.pick_num_splits(32768, 64, 512, 64, 2048, num_sms=152) == 1
    assert dsa.pick_num_splits(1024, 64, 512, 64, 2048, num_sms=152) == 1
    # 128 decode tokens on 152 SMs: one wave without splitting; splitting
    # would only add waves, partial writes and a combine
    assert dsa.pick_num_splits(128, 64, 512, 64, 2048, num_sms=152) == 1
    # 16 tokens of 1M context: split until the SMs are busy
    s_1m = dsa.pick_num_splits(16, 64, 512, 64, 2048, num_sms=152)
    assert 4 <= s_1m <= ntiles and 16 * s_1m <= 152
    assert dsa.pick_num_splits(1, 64, 512, 64, 100, num_sms=152) == 1  # a single tile cannot split
    for nq in (1, 2, 5, 16, 40, 100):
        s = dsa.pick_num_splits(nq, 64, 512, 64, 2048, num_sms=152)
        assert 1 <= s <= ntiles


# ---- argument validation: every case returns before any CUDA call ----
# The cases below hand the C ABI fake device addresses, which only the
# library's argument checks ever look at.  They run where no CUDA device is
# present, so that even a regression in the order of the checks could not
# launch a kernel on such an address.

def _has_cuda_device() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


no_device_only = pytest.mark.skipif(_has_cuda_device(),
                                    reason="fake device addresses are only used where no CUDA device is present")

VP = ctypes.c_void_p
FAKE = VP(0x10000)  # 16-byte aligned, never dereferenced on these paths
MISALIGNED = VP(0x10004)


def _fwd(lib, **over):
    a = dict(q=FAKE, kv=FAKE, kv_scale=FAKE, num_pages=4, bt=FAKE, num_req=1, bt_stride=4, q_req=FAKE, idx=FAKE,
             num_q=1, H=64, dl=512, dr=64, P=64, k=2048, scale=0.04, S=1, out=FAKE, lse=FAKE, op=None, lp=None,
             ws=FAKE, wsb=1 << 20, st=None, stream=None)
    a.update(over)
    return lib.dsa_sparse_mla_fwd(a["q"], a["kv"], a["kv_scale"], a["num_pages"], a["bt"], a["num_req"],
                                  a["bt_stride"], a["q_req"], a["idx"], a["num_q"], a["H"], a["dl"], a["dr"], a["P"],
                                  a["k"], a["scale"], a["S"], a["out"], a["lse"], a["op"], a["lp"], a["ws"],
                                  a["wsb"], a["st"], a["stream"])


@no_device_only
@pytest.mark.parametrize("over,expect", [
    (dict(H=32), 2), (dict(dl=256), 2), (dict(dr=32), 2),
    (dict(k=0), 1), (dict(P=0), 1), (dict(num_q=-1), 1), (dict(S=0), 1), (dict(S=65), 1),
    (dict(q=None), 1), (dict(kv=None), 1), (dict(idx=None), 1), (dict(out=None), 1),
    (dict(q=MISALIGNED), 1), (dict(kv=MISALIGNED), 1), (dict(out=MISALIGNED), 1), (dict(scale=float("inf")), 1),
    (dict(S=4, op=None, lp=FAKE), 1), (dict(S=4, op=MISALIGNED, lp=FAKE), 1), (dict(num_pages=0), 1),
    (dict(wsb=100), 3), (dict(ws=None), 1), (dict(ws=VP(0x10004)), 1), (dict(num_pages=1 << 26), 2),
    (dict(num_q=0), 0),
])
def test_fwd_argument_checks(lib, over, expect):
    assert _fwd(lib, **over) == expect


@no_device_only
@pytest.mark.parametrize("args,expect", [
    ((FAKE, 100, FAKE, 4, 0, FAKE, None, 0, None, None), 1),
    ((FAKE, 0, FAKE, 4, 8, FAKE, None, 0, None, None), 1),
    ((None, 100, FAKE, 4, 8, FAKE, None, 0, None, None), 1),
    ((FAKE, 100, None, 4, 8, FAKE, None, 0, None, None), 1),
    ((FAKE, 100, FAKE, 4, 8, None, None, 0, None, None), 1),
    ((FAKE, 100, FAKE, -1, 8, FAKE, None, 0, None, None), 1),
    ((FAKE, 100, FAKE, 0, 8, FAKE, None, 0, None, None), 0),
    # rows longer than 65,536 positions: a partial workspace is an error, a
    # sized one without a pointer too (both checked before any launch)
    ((FAKE, 1 << 20, FAKE, 16, 2048, FAKE, FAKE, 100, None, None), 3),
    ((FAKE, 1 << 20, FAKE, 16, 2048, FAKE, None, 16 * 16 * 2048 * 8, None, None), 1),
])
def test_topk_argument_checks(lib, args, expect):
    assert lib.dsa_topk_select(*args) == expect


@no_device_only
@pytest.mark.parametrize("args,expect", [
    ((FAKE, FAKE, 0, 4, 64, 512, FAKE, FAKE, None), 1),
    ((FAKE, FAKE, 65, 4, 64, 512, FAKE, FAKE, None), 1),
    ((FAKE, FAKE, 2, 4, 65, 512, FAKE, FAKE, None), 1),
    ((FAKE, FAKE, 2, 4, 64, 510, FAKE, FAKE, None), 1),
    ((None, FAKE, 2, 4, 64, 512, FAKE, FAKE, None), 1),
    ((MISALIGNED, FAKE, 2, 4, 64, 512, FAKE, FAKE, None), 1),
    ((FAKE, FAKE, 2, 0, 64, 512, FAKE, FAKE, None), 0),
])
def test_combine_argument_checks(lib, args, expect):
    assert lib.dsa_combine(*args) == expect


def _fused(lib, **over):
    a = dict(scores=FAKE, ld=4096, qpos=FAKE, k=2048, idx=FAKE, q=FAKE, kv=FAKE, kv_scale=FAKE, num_pages=4, bt=FAKE,
             num_req=1, bt_stride=4, q_req=FAKE, num_q=1, H=64, dl=512, dr=64, P=64, scale=0.04, out=FAKE, lse=FAKE,
             ws=FAKE, wsb=1 << 20, st=None, stream=None)
    a.update(over)
    return lib.dsa_sparse_mla_topk_fwd(a["scores"], a["ld"], a["qpos"], a["k"], a["idx"], a["q"], a["kv"],
                                       a["kv_scale"], a["num_pages"], a["bt"], a["num_req"], a["bt_stride"],
                                       a["q_req"], a["num_q"], a["H"], a["dl"], a["dr"], a["P"], a["scale"], a["out"],
                                       a["lse"], a["ws"], a["wsb"], a["st"], a["stream"])


@no_device_only
@pytest.mark.parametrize("over,expect", [
    (dict(H=16, dl=64, dr=16), 2), (dict(ld=65537), 2), (dict(k=100000), 2), (dict(ld=0), 1), (dict(k=0), 1),
    (dict(scores=None), 1), (dict(qpos=None), 1), (dict(idx=None), 1), (dict(out=None), 1), (dict(q=MISALIGNED), 1),
    (dict(wsb=100), 3), (dict(num_q=0), 0),
])
def test_fused_argument_checks(lib, over, expect):
    assert _fused(lib, **over) == expect


def _two(lib, **over):
    a = dict(scores=FAKE, ld=4096, qpos=FAKE, k=2048, idx=FAKE, q=FAKE, kv=FAKE, kv_scale=FAKE, num_pages=4, bt=FAKE,
             num_req=1, bt_stride=4, q_req=FAKE, num_q=1, H=64, dl=512, dr=64, P=64, scale=0.04, S=1, out=FAKE,
             lse=FAKE, op=None, lp=None, ws=FAKE, wsb=1 << 20, st=None, stream=None)
    a.update(over)
    return lib.dsa_topk_sparse_mla_fwd(a["scores"], a["ld"], a["qpos"], a["k"], a["idx"], a["q"], a["kv"],
                                       a["kv_scale"], a["num_pages"], a["bt"], a["num_req"], a["bt_stride"],
                                       a["q_req"], a["num_q"], a["H"], a["dl"], a["dr"], a["P"], a["scale"], a["S"],
                                       a["out"], a["lse"], a["op"], a["lp"], a["ws"], a["wsb"], a["st"], a["stream"])


@no_device_only
@pytest.mark.parametrize("over,expect", [
    (dict(H=16, dl=64, dr=16), 2), (dict(ld=65537), 2), (dict(ld=0), 1), (dict(k=0), 1),
    (dict(scores=None), 1), (dict(qpos=None), 1), (dict(idx=None), 1), (dict(out=None), 1), (dict(q=MISALIGNED), 1),
    (dict(bt=None), 1), (dict(q_req=None), 1), (dict(S=0), 1), (dict(S=65), 1), (dict(S=4, op=None, lp=FAKE), 1),
    (dict(wsb=100), 3), (dict(ws=None), 1), (dict(scale=float("nan")), 1), (dict(num_q=0), 0),
])
def test_two_kernel_argument_checks(lib, over, expect):
    assert _two(lib, **over) == expect


def test_fused_max_k(lib):
    assert lib.dsa_sparse_mla_topk_max_k() >= 2048


def test_topk_workspace_size(lib):
    # (score, position) blocks of k per 65,536-position slice of every row
    assert dsa.topk_workspace_size(16, 1 << 20, 2048) == 16 * 16 * 2048 * 8
    assert dsa.topk_workspace_size(3, 70001, 100) == 3 * 2 * 100 * 8
    assert dsa.topk_workspace_size(128, 65536, 2048) == 0        # one slice: no merge needed
    assert dsa.topk_workspace_size(4, 70001, 33000) == 0         # the union would exceed a row
    assert dsa.topk_workspace_size(0, 1 << 20, 2048) == 0


def test_workspace_size(lib):
    assert dsa.sparse_mla_workspace_size(128, 64, 512, 64, 2048) == 128 * 2048 * 8
    assert dsa.sparse_mla_workspace_size(2, 16, 64, 16, 64) == 0
    assert dsa.sparse_mla_workspace_size(0, 64, 512, 64, 2048) == 0


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        dsa.topk_select(torch.zeros(2, 8), torch.zeros(2, dtype=torch.int32), 4)
    with pytest.raises(TypeError):
        dsa.topk_select(torch.zeros(2, 8, dtype=torch.float64), torch.zeros(2, dtype=torch.int32), 4)


def _kvw(lib, **over):
    a = dict(rows=FAKE, n=4, d=576, req=FAKE, pos=FAKE, bt=FAKE, num_req=1, bt_stride=4, P=64, num_pages=4, kv=FAKE,
             sc=FAKE, st=None, stream=None)
    a.update(over)
    return lib.dsa_kv_write(a["rows"], a["n"], a["d"], a["req"], a["pos"], a["bt"], a["num_req"], a["bt_stride"],
                            a["P"], a["num_pages"], a["kv"], a["sc"], a["st"], a["stream"])


@no_device_only
@pytest.mark.parametrize("over,expect", [
    (dict(n=-1), 1), (dict(d=8), 1), (dict(d=584), 1), (dict(d=4096), 1), (dict(P=0), 1), (dict(num_pages=0), 1),
    (dict(num_req=0), 1), (dict(bt_stride=0), 1), (dict(rows=None), 1), (dict(kv=None), 1), (dict(sc=None), 1),
    (dict(req=None), 1), (dict(pos=None), 1), (dict(bt=None), 1), (dict(rows=MISALIGNED), 1),
    (dict(kv=MISALIGNED), 1), (dict(num_pages=1 << 30, P=64), 2), (dict(n=0, rows=None), 0),
])
def test_kv_write_argument_checks(lib, over, expect):
    """Every case returns before any CUDA call (fake device pointers)."""
    assert _kvw(lib, **over) == expect


def test_pick_num_splits_rule(lib):
    """The split rule on a 152-SM GB300 (no device needed): no split once the
    query tokens fill the SMs; the 16-token 1M-context workload splits 8 ways;
    never more splits than 64-row tiles; unsupported shapes get 1."""
    sms = 152
    assert dsa.pick_num_splits(128, 64, 512, 64, 2048, sms) == 1          # decode
    assert dsa.pick_num_splits(1024, 64, 512, 64, 2048, sms) == 1         # verify
    assert dsa.pick_num_splits(32768, 64, 512, 64, 2048, sms) == 1        # prefill
    assert dsa.pick_num_splits(16, 64, 512, 64, 2048, sms) == 8           # 1M context
    for nq in (1, 2, 5, 17, 75, 151, 152, 400):
        s = dsa.pick_num_splits(nq, 64, 512, 64, 2048, sms)
        assert 1 <= s <= 32                                               # 2048 / 64 tiles
        if nq >= sms:
            assert s == 1
    assert dsa.pick_num_splits(4, 64, 512, 64, 100, sms) <= 2             # 100 rows: 2 tiles
    assert dsa.pick_num_splits(4, 32, 512, 64, 2048, sms) == 1            # unsupported heads
    assert dsa.pick_num_splits(0, 64, 512, 64, 2048, sms) == 1
