"""GB300 (sm_103a) DSA sparse-MLA library: Python binding of the C ABI.

The three calls of the path -- ``topk_select``, ``sparse_mla_fwd`` and
``combine`` -- marshal torch tensors (device memory, the current CUDA stream)
into the C ABI declared in ``include/dsa.h`` and run entirely in the
library's CUDA kernels.  There is no CPU or PyTorch fallback: if the library
is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["DsaError", "load_library", "topk_select", "sparse_mla_fwd", "combine", "sparse_mla_topk",
           "topk_sparse_mla_fwd", "two_kernel_path_supported", "sparse_mla_topk_fused", "fused_path_supported",
           "kv_write",
           "PrefixCache",
           "kv_tile_count", "kv_tile_size", "pick_num_splits", "status_string", "EXPORTED_SYMBOLS",
           "DEV_BAD_QPOS", "DEV_BAD_INDEX", "DEV_BAD_PAGE", "DEV_TIMEOUT"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DEV_BAD_QPOS, DEV_BAD_INDEX, DEV_BAD_PAGE, DEV_TIMEOUT = 1, 2, 4, 8

# Every symbol include/dsa.h declares.
EXPORTED_SYMBOLS = ("dsa_status_string", "dsa_version", "dsa_topk_select", "dsa_topk_workspace_size",
                    "dsa_sparse_mla_fwd", "dsa_sparse_mla_workspace_size", "dsa_sparse_mla_fwd_noalloc",
                    "dsa_sparse_mla_topk_fwd", "dsa_sparse_mla_topk_max_k", "dsa_topk_sparse_mla_fwd",
                    "dsa_combine", "dsa_kv_write", "dsa_prefix_cache_create", "dsa_prefix_cache_destroy",
                    "dsa_prefix_cache_acquire", "dsa_prefix_cache_release", "dsa_prefix_cache_stats",
                    "dsa_kv_tile_count", "dsa_kv_tile_size", "dsa_pick_num_splits")

_lock = threading.Lock()
_lib = None


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")
        self.status = status


def load_library(path: str | None = None):
    """Load libdsa.so (built by ``__graft_entry__.build()`` or
    ``python -m dsa_sparse_mla_topk_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first "
                               "(python -m dsa_sparse_mla_topk_gb300.build)")
        lib = ctypes.CDLL(p)
        i32, i64, vp, f32, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
        lib.dsa_status_string.argtypes = [i32]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_version.argtypes = []
        lib.dsa_version.restype = i32
        lib.dsa_topk_select.argtypes = [vp, i64, vp, i32, i32, vp, vp, sz, vp, vp]
        lib.dsa_topk_select.restype = i32
        lib.dsa_topk_workspace_size.argtypes = [i32, i64, i32]
        lib.dsa_topk_workspace_size.restype = sz
        lib.dsa_sparse_mla_fwd.argtypes = [vp, vp, vp, i64, vp, i32, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                           f32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
        lib.dsa_sparse_mla_fwd_noalloc.argtypes = [vp, vp, vp, i64, vp, i32, i32, vp, vp, i32, i32, i32, i32, i32,
                                                   i32, f32, i32, vp, vp, vp, vp, vp, vp]
        lib.dsa_sparse_mla_fwd_noalloc.restype = i32
        lib.dsa_sparse_mla_topk_fwd.argtypes = [vp, i64, vp, i32, vp, vp, vp, vp, i64, vp, i32, i32, vp, i32, i32, i32,
                                                i32, i32, f32, vp, vp, vp, sz, vp, vp]
        lib.dsa_sparse_mla_topk_fwd.restype = i32
        lib.dsa_topk_sparse_mla_fwd.argtypes = [vp, i64, vp, i32, vp, vp, vp, vp, i64, vp, i32, i32, vp, i32, i32,
                                                i32, i32, i32, f32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
        lib.dsa_topk_sparse_mla_fwd.restype = i32
        lib.dsa_sparse_mla_topk_max_k.argtypes = []
        lib.dsa_sparse_mla_topk_max_k.restype = i32
        lib.dsa_sparse_mla_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.dsa_sparse_mla_workspace_size.restype = sz
        lib.dsa_sparse_mla_fwd.restype = i32
        lib.dsa_combine.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
        lib.dsa_combine.restype = i32
        lib.dsa_kv_write.argtypes = [vp, i32, i32, vp, vp, vp, i32, i32, i32, i64, vp, vp, vp, vp]
        lib.dsa_kv_write.restype = i32
        lib.dsa_prefix_cache_create.argtypes = [i32, i32]
        lib.dsa_prefix_cache_create.restype = vp
        lib.dsa_prefix_cache_destroy.argtypes = [vp]
        lib.dsa_prefix_cache_destroy.restype = None
        lib.dsa_prefix_cache_acquire.argtypes = [vp, vp, i64, vp, i32, vp, vp]
        lib.dsa_prefix_cache_acquire.restype = i32
        lib.dsa_prefix_cache_release.argtypes = [vp, vp, i32]
        lib.dsa_prefix_cache_release.restype = i32
        lib.dsa_prefix_cache_stats.argtypes = [vp, vp, vp, vp]
        lib.dsa_prefix_cache_stats.restype = i32
        lib.dsa_kv_tile_count.argtypes = [i32, i32]
        lib.dsa_kv_tile_count.restype = i32
        lib.dsa_kv_tile_size.argtypes = [i32, i32, i32]
        lib.dsa_kv_tile_size.restype = i32
        lib.dsa_pick_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.dsa_pick_num_splits.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().dsa_status_string(int(status)).decode()


def kv_tile_count(width: int, tile: int) -> int:
    return load_library().dsa_kv_tile_count(int(width), int(tile))


def kv_tile_size(heads: int, d_latent: int, d_rope: int) -> int:
    return load_library().dsa_kv_tile_size(heads, d_latent, d_rope)


def pick_num_splits(num_q: int, heads: int, d_latent: int, d_rope: int, k: int, num_sms: int = 0) -> int:
    return load_library().dsa_pick_num_splits(num_q, heads, d_latent, d_rope, k, num_sms)


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, ndim: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _call(fn: str, *args):
    st = getattr(load_library(), fn)(*args)
    if st != 0:
        raise DsaError(fn, st)


def topk_select(scores: torch.Tensor, q_pos: torch.Tensor, k: int, idx: torch.Tensor | None = None,
                dev_status: torch.Tensor | None = None, stream=None,
                workspace: torch.Tensor | None = None) -> torch.Tensor:
    """int32 [num_q, k] causal top-k positions (ascending, -1 padded).
    ``workspace`` (uint8, at least ``topk_workspace_size`` bytes) is allocated
    when the sliced path for rows longer than 65,536 positions applies and
    none is given; an empty tensor selects the in-place path instead."""
    _check(scores, "scores", torch.float32, 2)
    _check(q_pos, "q_pos", torch.int32, 1)
    num_q, ld = scores.shape
    if idx is None:
        idx = torch.empty((num_q, k), dtype=torch.int32, device=scores.device)
    _check(idx, "idx", torch.int32, 2)
    ws_bytes = topk_workspace_size(num_q, ld, k)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=scores.device)
    _call("dsa_topk_select", _p(scores), ld, _p(q_pos), num_q, k, _p(idx), _p(workspace),
          0 if workspace is None else workspace.numel(), _p(dev_status), _stream(stream))
    return idx


def sparse_mla_workspace_size(num_q: int, heads: int, d_latent: int, d_rope: int, k: int) -> int:
    return load_library().dsa_sparse_mla_workspace_size(num_q, heads, d_latent, d_rope, k)


def sparse_mla_fwd(q, kv, kv_scale, block_table, q_req, idx, *, d_latent: int, d_rope: int, page_size: int,
                   softmax_scale: float, num_splits: int = 1, out=None, lse=None, o_part=None, lse_part=None,
                   workspace=None, dev_status=None, stream=None):
    """Partial step.  num_splits == 1: returns (out bf16, lse fp32).
    num_splits > 1: returns (o_part fp32 [S, ...], lse_part fp32 [S, ...])."""
    _check(q, "q", torch.bfloat16, 3)
    _check(kv, "kv", torch.uint8, 2)
    _check(kv_scale, "kv_scale", torch.float32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    _check(q_req, "q_req", torch.int32, 1)
    _check(idx, "idx", torch.int32, 2)
    num_q, H, dqk = q.shape
    if dqk != d_latent + d_rope or kv.shape[1] != dqk or kv.shape[0] % page_size:
        raise ValueError("q / kv row sizes do not match d_latent + d_rope, or kv is not whole pages")
    dev = q.device
    if num_splits == 1:
        if out is None:
            out = torch.empty((num_q, H, d_latent), dtype=torch.bfloat16, device=dev)
        if lse is None:
            lse = torch.empty((num_q, H), dtype=torch.float32, device=dev)
    else:
        if o_part is None:
            o_part = torch.empty((num_splits, num_q, H, d_latent), dtype=torch.float32, device=dev)
        if lse_part is None:
            lse_part = torch.empty((num_splits, num_q, H), dtype=torch.float32, device=dev)
    ws_bytes = sparse_mla_workspace_size(num_q, H, d_latent, d_rope, idx.shape[1])
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _call("dsa_sparse_mla_fwd", _p(q), _p(kv), _p(kv_scale), kv.shape[0] // page_size, _p(block_table),
          block_table.shape[0], block_table.shape[1], _p(q_req), _p(idx), num_q, H, d_latent, d_rope, page_size,
          idx.shape[1], float(softmax_scale), num_splits, _p(out) if num_splits == 1 else None,
          _p(lse) if num_splits == 1 else None, _p(o_part) if num_splits > 1 else None,
          _p(lse_part) if num_splits > 1 else None, _p(workspace) if ws_bytes else None, ws_bytes,
          _p(dev_status), _stream(stream))
    return (out, lse) if num_splits == 1 else (o_part, lse_part)


def sparse_mla_fwd_noalloc(q, kv, kv_scale, block_table, q_req, idx, out, lse, *, d_latent: int, d_rope: int,
                           page_size: int, softmax_scale: float, dev_status=None, stream=None):
    """Partial step without a workspace (no device allocation inside the
    library call): scratch comes from a fixed array in the library; the
    caller provides out / lse.  See include/dsa.h for its limits."""
    for t, name, dt in ((q, "q", torch.bfloat16), (kv, "kv", torch.uint8), (kv_scale, "kv_scale", torch.float32),
                        (block_table, "block_table", torch.int32), (q_req, "q_req", torch.int32),
                        (idx, "idx", torch.int32), (out, "out", torch.bfloat16), (lse, "lse", torch.float32)):
        _check(t, name, dt)
    num_q, H, _ = q.shape
    _call("dsa_sparse_mla_fwd_noalloc", _p(q), _p(kv), _p(kv_scale), kv.shape[0] // page_size, _p(block_table),
          block_table.shape[0], block_table.shape[1], _p(q_req), _p(idx), num_q, H, d_latent, d_rope, page_size,
          idx.shape[1], float(softmax_scale), 1, _p(out), _p(lse), None, None, _p(dev_status), _stream(stream))
    return out, lse


def combine(o_part: torch.Tensor, lse_part: torch.Tensor, out=None, lse=None, stream=None):
    """Combine step: (out bf16 [num_q, H, dv], lse fp32 [num_q, H])."""
    _check(o_part, "o_part", torch.float32, 4)
    _check(lse_part, "lse_part", torch.float32, 3)
    S, num_q, H, dv = o_part.shape
    if out is None:
        out = torch.empty((num_q, H, dv), dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty((num_q, H), dtype=torch.float32, device=o_part.device)
    _call("dsa_combine", _p(o_part), _p(lse_part), S, num_q, H, dv, _p(out), _p(lse), _stream(stream))
    return out, lse


def topk_workspace_size(num_q: int, ld: int, k: int) -> int:
    """Workspace bytes dsa_topk_select can use (0 when no workspace applies)."""
    return int(load_library().dsa_topk_workspace_size(num_q, ld, k))


def kv_write(rows: torch.Tensor, req: torch.Tensor, pos: torch.Tensor, block_table: torch.Tensor,
             kv: torch.Tensor, kv_scale: torch.Tensor, *, page_size: int, dev_status=None, stream=None):
    """Quantise bf16 rows [n, d_qk] to FP8 E4M3 with one fp32 scale per token
    and store them, in place, into the paged cache ``kv`` (uint8 [slots, d_qk])
    and ``kv_scale`` (fp32 [slots]) at each row's (request, position) slot."""
    _check(rows, "rows", torch.bfloat16, 2)
    _check(req, "req", torch.int32, 1)
    _check(pos, "pos", torch.int32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    _check(kv, "kv", torch.uint8, 2)
    _check(kv_scale, "kv_scale", torch.float32, 1)
    n, d = rows.shape
    if req.shape != (n,) or pos.shape != (n,) or kv.shape[1] != d or kv.shape[0] != kv_scale.shape[0]:
        raise ValueError("inconsistent shapes")
    if kv.shape[0] % page_size:
        raise ValueError("kv rows must be a whole number of pages")
    _call("dsa_kv_write", _p(rows), n, d, _p(req), _p(pos), _p(block_table), block_table.shape[0],
          block_table.shape[1], page_size, kv.shape[0] // page_size, _p(kv), _p(kv_scale), _p(dev_status),
          _stream(stream))
    return kv, kv_scale


class PrefixCache:
    """KV-only prefix-sharing page allocator (host side): requests sharing
    whole-page prefixes get the same page ids; see dsa_prefix_cache_* in
    include/dsa.h."""

    def __init__(self, page_size: int, num_pages: int):
        self._lib = load_library()
        self.page_size, self.num_pages = page_size, num_pages
        self._h = self._lib.dsa_prefix_cache_create(page_size, num_pages)
        if not self._h:
            raise DsaError("dsa_prefix_cache_create", 1)

    def acquire(self, tokens):
        """int32 page ids of a request's tokens, and how many of the leading
        ones were already cached (their KV rows need not be written)."""
        import numpy as np
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n_pages = (len(t) + self.page_size - 1) // self.page_size
        bt = np.empty(max(1, n_pages), dtype=np.int32)
        np_out, ns_out = ctypes.c_int32(0), ctypes.c_int32(0)
        st = self._lib.dsa_prefix_cache_acquire(self._h, t.ctypes.data_as(ctypes.c_void_p), len(t),
                                                bt.ctypes.data_as(ctypes.c_void_p), n_pages, ctypes.byref(np_out),
                                                ctypes.byref(ns_out))
        if st != 0:
            raise DsaError("dsa_prefix_cache_acquire", st)
        return bt[:np_out.value].copy(), ns_out.value

    def release(self, block_table):
        import numpy as np
        bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
        st = self._lib.dsa_prefix_cache_release(self._h, bt.ctypes.data_as(ctypes.c_void_p), len(bt))
        if st != 0:
            raise DsaError("dsa_prefix_cache_release", st)

    def stats(self):
        """(pages referenced by live requests, pages cached, pages free)."""
        a, b, c = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        self._lib.dsa_prefix_cache_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
        return a.value, b.value, c.value

    def close(self):
        if self._h:
            self._lib.dsa_prefix_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sparse_mla_topk_fused(q, kv, kv_scale, block_table, q_req, q_pos, scores, k: int, *, d_latent: int,
                          d_rope: int, page_size: int, softmax_scale: float, idx=None, out=None, lse=None,
                          workspace=None, dev_status=None, stream=None):
    """Top-k and the Partial step (one KV split) in one kernel call
    (dsa_sparse_mla_topk_fwd); same results as topk_select followed by
    sparse_mla_fwd.  Returns (out, lse, idx)."""
    for t, name, dt in ((q, "q", torch.bfloat16), (kv, "kv", torch.uint8), (kv_scale, "kv_scale", torch.float32),
                        (block_table, "block_table", torch.int32), (q_req, "q_req", torch.int32),
                        (q_pos, "q_pos", torch.int32), (scores, "scores", torch.float32)):
        _check(t, name, dt)
    num_q, H, dqk = q.shape
    if dqk != d_latent + d_rope or kv.shape[1] != dqk or kv.shape[0] % page_size:
        raise ValueError("q / kv row sizes do not match d_latent + d_rope, or kv is not whole pages")
    dev = q.device
    if idx is None:
        idx = torch.empty((num_q, k), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((num_q, H, d_latent), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((num_q, H), dtype=torch.float32, device=dev)
    ws_bytes = sparse_mla_workspace_size(num_q, H, d_latent, d_rope, k)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _call("dsa_sparse_mla_topk_fwd", _p(scores), scores.shape[1], _p(q_pos), k, _p(idx), _p(q), _p(kv),
          _p(kv_scale), kv.shape[0] // page_size, _p(block_table), block_table.shape[0], block_table.shape[1],
          _p(q_req), num_q, H, d_latent, d_rope, page_size, float(softmax_scale), _p(out), _p(lse),
          _p(workspace) if ws_bytes else None, ws_bytes, _p(dev_status), _stream(stream))
    return out, lse, idx


def two_kernel_path_supported(heads: int, d_latent: int, d_rope: int, ld: int) -> bool:
    """Whether topk_sparse_mla_fwd takes this shape: the tensor-core head
    shape and rows of at most 65,536 positions (any k, any KV split)."""
    return (heads, d_latent, d_rope) == (64, 512, 64) and ld <= 65536


def topk_sparse_mla_fwd(q, kv, kv_scale, block_table, q_req, q_pos, scores, k: int, *, d_latent: int, d_rope: int,
                        page_size: int, softmax_scale: float, num_splits: int = 1, idx=None, out=None, lse=None,
                        o_part=None, lse_part=None, workspace=None, dev_status=None, stream=None):
    """topk_select followed by sparse_mla_fwd as two kernels, the top-k also
    looking up each selected position's page and scale
    (dsa_topk_sparse_mla_fwd); bit for bit the results of the two calls.
    Returns (out, lse, idx), or (o_part, lse_part, idx) when num_splits > 1."""
    for t, name, dt in ((q, "q", torch.bfloat16), (kv, "kv", torch.uint8), (kv_scale, "kv_scale", torch.float32),
                        (block_table, "block_table", torch.int32), (q_req, "q_req", torch.int32),
                        (q_pos, "q_pos", torch.int32), (scores, "scores", torch.float32)):
        _check(t, name, dt)
    num_q, H, dqk = q.shape
    if dqk != d_latent + d_rope or kv.shape[1] != dqk or kv.shape[0] % page_size:
        raise ValueError("q / kv row sizes do not match d_latent + d_rope, or kv is not whole pages")
    dev = q.device
    if idx is None:
        idx = torch.empty((num_q, k), dtype=torch.int32, device=dev)
    if num_splits == 1:
        if out is None:
            out = torch.empty((num_q, H, d_latent), dtype=torch.bfloat16, device=dev)
        if lse is None:
            lse = torch.empty((num_q, H), dtype=torch.float32, device=dev)
    else:
        if o_part is None:
            o_part = torch.empty((num_splits, num_q, H, d_latent), dtype=torch.float32, device=dev)
        if lse_part is None:
            lse_part = torch.empty((num_splits, num_q, H), dtype=torch.float32, device=dev)
    ws_bytes = sparse_mla_workspace_size(num_q, H, d_latent, d_rope, k)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _call("dsa_topk_sparse_mla_fwd", _p(scores), scores.shape[1], _p(q_pos), k, _p(idx), _p(q), _p(kv),
          _p(kv_scale), kv.shape[0] // page_size, _p(block_table), block_table.shape[0], block_table.shape[1],
          _p(q_req), num_q, H, d_latent, d_rope, page_size, float(softmax_scale), num_splits,
          _p(out) if num_splits == 1 else None, _p(lse) if num_splits == 1 else None,
          _p(o_part) if num_splits > 1 else None, _p(lse_part) if num_splits > 1 else None,
          _p(workspace) if ws_bytes else None, ws_bytes, _p(dev_status), _stream(stream))
    return (out, lse, idx) if num_splits == 1 else (o_part, lse_part, idx)


def fused_path_supported(num_q: int, heads: int, d_latent: int, d_rope: int, ld: int, k: int,
                         num_splits: int) -> bool:
    """Whether the single-kernel path (dsa_sparse_mla_topk_fwd: the row's top-k,
    the page lookup and the Partial in one CTA per query token) can run this
    shape: the tensor-core head shape, one KV split, rows of at most 65,536
    positions and k within the kernel's limit.

    sparse_mla_topk does not pick it by itself: measured on GB300, the separate
    calls are faster at every decode batch tried (8 to 128 requests of a 64K
    context, and the 8-token verify and prefill shapes): the single kernel's
    selection and tile loop run a little slower, and it cannot split the KV
    range, which the small batches need."""
    del num_q
    if (heads, d_latent, d_rope) != (64, 512, 64) or num_splits != 1 or ld > 65536:
        return False
    return k <= load_library().dsa_sparse_mla_topk_max_k()


def sparse_mla_topk(q, kv, kv_scale, block_table, q_req, q_pos, scores, k: int, *, d_latent: int, d_rope: int,
                    page_size: int, softmax_scale: float, num_splits: int | None = None, buffers: dict | None = None,
                    dev_status=None, stream=None, fused: bool | None = None):
    """One pass of the whole path: top-k -> Partial -> Combine (when split).
    ``buffers`` (optional) holds preallocated idx / out / lse / o_part /
    lse_part / workspace tensors.  ``fused``: True runs top-k and the Partial
    step in one kernel (dsa_sparse_mla_topk_fwd, where fused_path_supported);
    False or None, the faster path: where two_kernel_path_supported, the top-k
    with the page lookup and then the attention kernel
    (dsa_topk_sparse_mla_fwd), else topk_select and sparse_mla_fwd.  The
    results are the same every way.  Returns (out, lse, idx)."""
    b = buffers or {}
    num_q, H, _ = q.shape
    if num_splits is None:
        num_splits = pick_num_splits(num_q, H, d_latent, d_rope, k)
    if fused:
        if num_splits != 1:
            raise ValueError("the fused path has one KV split")
        return sparse_mla_topk_fused(q, kv, kv_scale, block_table, q_req, q_pos, scores, k, d_latent=d_latent,
                                     d_rope=d_rope, page_size=page_size, softmax_scale=softmax_scale,
                                     idx=b.get("idx"), out=b.get("out"), lse=b.get("lse"),
                                     workspace=b.get("workspace"), dev_status=dev_status, stream=stream)
    if two_kernel_path_supported(H, d_latent, d_rope, scores.shape[1]):
        r = topk_sparse_mla_fwd(q, kv, kv_scale, block_table, q_req, q_pos, scores, k, d_latent=d_latent,
                                d_rope=d_rope, page_size=page_size, softmax_scale=softmax_scale,
                                num_splits=num_splits, idx=b.get("idx"), out=b.get("out"), lse=b.get("lse"),
                                o_part=b.get("o_part"), lse_part=b.get("lse_part"), workspace=b.get("workspace"),
                                dev_status=dev_status, stream=stream)
        if num_splits == 1:
            return r
        out, lse = combine(r[0], r[1], out=b.get("out"), lse=b.get("lse"), stream=stream)
        return out, lse, r[2]
    idx = topk_select(scores, q_pos, k, idx=b.get("idx"), dev_status=dev_status, stream=stream,
                      workspace=b.get("topk_workspace"))
    if num_splits == 1:
        out, lse = sparse_mla_fwd(q, kv, kv_scale, block_table, q_req, idx, d_latent=d_latent, d_rope=d_rope,
                                  page_size=page_size, softmax_scale=softmax_scale, num_splits=1, out=b.get("out"),
                                  lse=b.get("lse"), workspace=b.get("workspace"), dev_status=dev_status,
                                  stream=stream)
        return out, lse, idx
    op, lp = sparse_mla_fwd(q, kv, kv_scale, block_table, q_req, idx, d_latent=d_latent, d_rope=d_rope,
                            page_size=page_size, softmax_scale=softmax_scale, num_splits=num_splits,
                            o_part=b.get("o_part"), lse_part=b.get("lse_part"), workspace=b.get("workspace"),
                            dev_status=dev_status, stream=stream)
    out, lse = combine(op, lp, out=b.get("out"), lse=b.get("lse"), stream=stream)
    return out, lse, idx
