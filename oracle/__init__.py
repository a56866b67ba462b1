"""fp64 CPU oracle for DSA sparse MLA with top-k selection (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never touches it and the
two share no code: this side is plain C (``dsa_oracle.c``) compiled with gcc,
wrapped here with ctypes over numpy arrays.  Each function states the
definition it follows; see ``dsa_oracle.c`` for the page citations.

Parity pins: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, BAD_QPOS, BAD_INDEX, BAD_PAGE, NOMEM = 0, 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: it runs on x86 and Arm)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c_i32, c_i64, c_p, c_d = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = c_d
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = c_d
            lib.oracle_topk.argtypes = [c_p, c_i64, c_p, c_i32, c_i32, c_p, ctypes.c_int]
            lib.oracle_topk.restype = ctypes.c_int
            lib.oracle_sparse_mla.argtypes = [c_p, c_p, c_p, c_i64, c_p, c_i64, c_p, c_p, c_i64, c_i32, c_i32,
                                              c_i32, c_i32, c_i32, c_d, c_i32, c_p, c_p, c_p, c_p, ctypes.c_int]
            lib.oracle_sparse_mla.restype = ctypes.c_int
            lib.oracle_combine.argtypes = [c_p, c_p, c_i32, c_i64, c_i32, c_i32, c_p, c_p]
            lib.oracle_combine.restype = ctypes.c_int
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_kv_write.argtypes = [c_p, c_i64, c_i32, c_p, c_p, c_p, c_i32, c_i32, c_i32, c_i64, c_p, c_p]
            lib.oracle_kv_write.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def e4m3_to_double(code: int) -> float:
    """Value of one FP8 E4M3 byte (exact)."""
    return _load().oracle_e4m3_to_double(int(code))


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def topk(scores: np.ndarray, q_pos: np.ndarray, k: int, nthreads: int = 0) -> np.ndarray:
    """int32 [num_q, k]: the min(k, q_pos+1) visible positions with the
    largest scores, ties to the lower position, ascending, -1 padded."""
    s = _c(scores, np.float32)
    qp = _c(q_pos, np.int32)
    assert s.ndim == 2 and qp.shape == (s.shape[0],)
    idx = np.empty((s.shape[0], k), dtype=np.int32)
    st = _load().oracle_topk(_ptr(s), s.shape[1], _ptr(qp), s.shape[0], k, _ptr(idx), nthreads)
    if st != OK:
        raise ValueError(f"oracle_topk status {st}")
    return idx


def sparse_mla(q_bits, kv, kv_scale, block_table, q_req, idx, *, d_latent, d_rope, page_size, softmax_scale,
               num_splits: int = 1, return_partials: bool = False, nthreads: int = 0, check: bool = True):
    """fp64 (out[num_q, H, d_latent], lse[num_q, H]) of softmax attention over
    the selected rows.  ``q_bits`` holds the bf16 bit patterns (uint16 or
    int16) [num_q, H, d_latent+d_rope]; ``kv`` the e4m3 bytes [slots, dqk]."""
    q = _c(q_bits, np.uint16) if np.asarray(q_bits).dtype != np.int16 else _c(np.asarray(q_bits).view(np.uint16), np.uint16)
    kvb = _c(kv, np.uint8)
    sc = _c(kv_scale, np.float32)
    bt = _c(block_table, np.int32)
    qr = _c(q_req, np.int32)
    ix = _c(idx, np.int32)
    num_q, H, dqk = q.shape
    assert dqk == d_latent + d_rope and kvb.shape[1] == dqk and ix.shape[0] == num_q
    assert kvb.shape[0] % page_size == 0 and sc.shape == (kvb.shape[0],)
    num_pages = kvb.shape[0] // page_size
    out = np.empty((num_q, H, d_latent), dtype=np.float64)
    lse = np.empty((num_q, H), dtype=np.float64)
    op = lp = None
    if return_partials:
        op = np.empty((num_splits, num_q, H, d_latent), dtype=np.float64)
        lp = np.empty((num_splits, num_q, H), dtype=np.float64)
    st = _load().oracle_sparse_mla(_ptr(q), _ptr(kvb), _ptr(sc), num_pages, _ptr(bt), bt.shape[1], _ptr(qr), _ptr(ix),
                                   num_q, ix.shape[1], H, d_latent, d_rope, page_size, float(softmax_scale),
                                   num_splits, _ptr(out), _ptr(lse), None if op is None else _ptr(op),
                                   None if lp is None else _ptr(lp), nthreads)
    if check and st != OK:
        raise ValueError(f"oracle_sparse_mla status {st}")
    if return_partials:
        return out, lse, op, lp
    return out, lse


def combine(o_part, lse_part):
    """fp64 log-sum-exp merge of partials [S, num_q, H, dv] / [S, num_q, H]."""
    op = _c(o_part, np.float64)
    lp = _c(lse_part, np.float64)
    S, num_q, H, dv = op.shape
    out = np.empty((num_q, H, dv), dtype=np.float64)
    lse = np.empty((num_q, H), dtype=np.float64)
    _load().oracle_combine(_ptr(op), _ptr(lp), S, num_q, H, dv, _ptr(out), _ptr(lse))
    return out, lse


def e4m3_encode(x: float) -> int:
    """Nearest FP8 E4M3 code of a finite float32, ties to even, saturating at 448."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def kv_write(rows_bits, req, pos, block_table, kv, kv_scale, *, page_size):
    """Quantise bf16 rows ([n, d] bit patterns) to FP8 E4M3 with one fp32 scale
    per token (scale = max|x| / 448, bytes = e4m3(x / scale), fp32 divisions)
    and store them, in place, into ``kv`` (uint8 [slots, d]) and ``kv_scale``
    (fp32 [slots]) at slot = block_table[req][pos // P] * P + pos % P.
    Returns the status bits (BAD_INDEX, BAD_PAGE) of skipped rows."""
    x = np.asarray(rows_bits)
    x = _c(x.view(np.uint16) if x.dtype == np.int16 else x, np.uint16)
    rq = _c(req, np.int32)
    ps = _c(pos, np.int32)
    bt = _c(block_table, np.int32)
    assert kv.dtype == np.uint8 and kv.flags.c_contiguous and kv_scale.dtype == np.float32
    assert kv_scale.flags.c_contiguous and kv.shape == (kv_scale.shape[0], x.shape[1])
    assert kv.shape[0] % page_size == 0
    return _load().oracle_kv_write(_ptr(x), x.shape[0], x.shape[1], _ptr(rq), _ptr(ps), _ptr(bt), bt.shape[0],
                                   bt.shape[1], page_size, kv.shape[0] // page_size, _ptr(kv), _ptr(kv_scale))
