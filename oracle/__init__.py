"""CPU oracle for batched paged-KV context attention (fp64).

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg (and its ``--impl reference`` arm) may import this package.
The product path never does; it shares no code with it.

``oracle.c`` holds the arithmetic; this module compiles it with gcc and
marshals torch CPU tensors into it.  Which passage of the pages each step
follows is written at the top of oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OR_BF16 = 1
OR_FP8_E4M3 = 2
LAYOUTS = {"HND": 0, "NHD": 1}


class _Pool(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
    ]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to oracle.c (gcc, -O2, OpenMP)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_gather.restype = ctypes.c_int
        lib.oracle_worklist.restype = ctypes.c_int
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_append_kv.restype = ctypes.c_int64
        lib.oracle_gather_ragged.restype = ctypes.c_int
        lib.oracle_ragged_lengths.restype = None
        _lib = lib
    return _lib


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _pool(t: torch.Tensor) -> _Pool:
    assert t.dim() == 4 and t.device.type == "cpu"
    if t.dtype == torch.bfloat16:
        dt = OR_BF16
    elif t.dtype == torch.float8_e4m3fn:
        dt = OR_FP8_E4M3
    else:
        raise TypeError(t.dtype)
    p = _Pool()
    p.data = t.data_ptr()
    p.dtype = dt
    for i in range(4):
        p.shape[i] = t.shape[i]
        p.stride[i] = t.stride(i)
    return p


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code to the binary32 value x (ties to the even code, +-448 saturation)."""
    return _load().oracle_e4m3_encode(x)


def append_kv(k_new: torch.Tensor, v_new: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
              cache_loc: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0, layout: str = "HND") -> int:
    """Write token n's K/V rows ([T, Hkv, D] bf16) into slot cache_loc[n] of the CPU pools, in place.

    Returns the number of tokens whose slot lies outside the pool (not written).
    """
    lib = _load()
    assert k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16 and k_new.dim() == 3
    assert k_new.shape == v_new.shape and k_new.stride() == v_new.stride() and k_new.stride(2) == 1
    loc = cache_loc.to(torch.int32).contiguous()
    assert loc.numel() == k_new.shape[0]
    kp, vp = _pool(k_pool), _pool(v_pool)
    return int(lib.oracle_append_kv(
        _ptr(k_new), _ptr(v_new), ctypes.c_int64(k_new.shape[0]), ctypes.c_int64(k_new.stride(0)),
        ctypes.c_int64(k_new.stride(1)), _ptr(loc), ctypes.byref(kp), ctypes.byref(vp),
        ctypes.c_int(LAYOUTS[layout]), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
    ))


def attention(inp, rows=None, threads: int | None = None):
    """Rows of the output in float64.

    ``rows``: None for every (token, head) row, else an int64 array of
    token * H + head.  Returns (out [n_rows, D] float64, status [n_rows]
    int32, threads used).
    """
    lib = _load()
    q = inp.q
    assert q.dtype == torch.bfloat16 and q.stride(2) == 1
    T, H, D = q.shape
    if rows is None:
        n_rows = T * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.size
    out = np.zeros((n_rows, D), dtype=np.float64)
    status = np.zeros((n_rows,), dtype=np.int32)
    kp, vp = _pool(inp.k_pool), _pool(inp.v_pool)
    bt = inp.block_tables.contiguous()
    sl = inp.seq_lens.contiguous()
    cq = inp.cum_q.contiguous()
    sinks = None if inp.sinks is None else inp.sinks.to(torch.float32).contiguous()
    used = lib.oracle_attention(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_int64(q.stride(0)), ctypes.c_int64(q.stride(1)),
        ctypes.c_int(T), ctypes.c_int(H), ctypes.c_int(D),
        ctypes.byref(kp), ctypes.byref(vp), ctypes.c_int(LAYOUTS[inp.layout]),
        _ptr(bt), ctypes.c_int64(bt.stride(0)), _ptr(sl), _ptr(cq), ctypes.c_int(sl.numel()),
        ctypes.c_double(inp.bmm1_scale), ctypes.c_double(inp.bmm2_scale),
        ctypes.c_int(inp.window_left),
        None if sinks is None else _ptr(sinks),
        None if rows_arr is None else rows_arr.ctypes.data_as(ctypes.c_void_p),
        ctypes.c_int64(n_rows),
        out.ctypes.data_as(ctypes.c_void_p), status.ctypes.data_as(ctypes.c_void_p),
        ctypes.c_int(0 if threads is None else int(threads)),
    )
    return out, status, used


def gather(inp, which: str = "k"):
    """Contiguous [sum(seq_lens), Hkv, D] copy of the K (or V) tokens, same dtype.

    Returns (tensor, ok).  ok is False when a referenced page id is outside
    the pool (those elements are zero).
    """
    lib = _load()
    pool = inp.k_pool if which == "k" else inp.v_pool
    Hkv = inp.num_kv_heads
    D = inp.head_dim
    total = int(inp.seq_lens.sum())
    out = torch.zeros((total, Hkv, D), dtype=pool.dtype)
    p = _pool(pool)
    bt = inp.block_tables.contiguous()
    rc = lib.oracle_gather(
        ctypes.byref(p), ctypes.c_int(LAYOUTS[inp.layout]), _ptr(bt), ctypes.c_int64(bt.stride(0)),
        _ptr(inp.seq_lens.contiguous()), _ptr(inp.cum_kv.contiguous()), ctypes.c_int(inp.batch),
        ctypes.c_void_p(out.data_ptr()),
    )
    return out, rc == 0


def worklist(inp, rows_per_tile: int, n_qtiles: int, kv_tile: int, cost_cap: int, cap: int | None = None):
    """The stable longest-first work list; int32 array [n, 4] of (b, kv head, item, cost)."""
    lib = _load()
    B = inp.batch
    if cap is None:
        per = rows_per_tile * n_qtiles
        cap = max(1, B * inp.num_kv_heads * ((max(inp.max_q_len, 1) + per - 1) // per))
    out = np.zeros((cap, 4), dtype=np.int32)
    n = lib.oracle_worklist(
        _ptr(inp.cum_q.contiguous()), _ptr(inp.seq_lens.contiguous()), ctypes.c_int(B),
        ctypes.c_int(inp.num_kv_heads), ctypes.c_int(rows_per_tile), ctypes.c_int(n_qtiles),
        ctypes.c_int(kv_tile), ctypes.c_int(inp.window_left), ctypes.c_int(inp.max_q_len),
        ctypes.c_int(inp.max_kv_len), ctypes.c_int(inp.page_size), ctypes.c_int(inp.block_tables.shape[1]),
        ctypes.c_int(inp.q.shape[0]), ctypes.c_int(cost_cap),
        out.ctypes.data_as(ctypes.c_void_p), ctypes.c_int(cap),
    )
    if n < 0:
        raise ValueError("work list larger than cap")
    return out[:n].copy()


def ragged_lengths(indptr: torch.Tensor, last_page_len: torch.Tensor, page_size: int) -> torch.Tensor:
    """Kv length of each request of a ragged page table (-1: malformed)."""
    lib = _load()
    ip = indptr.to(torch.int32).contiguous()
    lp = last_page_len.to(torch.int32).contiguous()
    B = ip.numel() - 1
    out = torch.zeros((max(B, 0),), dtype=torch.int32)
    lib.oracle_ragged_lengths(_ptr(ip), _ptr(lp), ctypes.c_int(B), ctypes.c_int(page_size), _ptr(out))
    return out


def gather_ragged(inp, indices, indptr, last_page_len, which: str = "k"):
    """Contiguous [sum(kv lengths), Hkv, D] copy of the K (or V) tokens through a
    ragged page table, at row offsets inp.cum_kv.  Returns (tensor, ok)."""
    lib = _load()
    pool = inp.k_pool if which == "k" else inp.v_pool
    kv = ragged_lengths(indptr, last_page_len, inp.page_size)
    ends = inp.cum_kv[:-1].to(torch.int64) + kv.clamp_min(0).to(torch.int64)
    total = max(int(inp.cum_kv[-1]), int(ends.max()) if ends.numel() else 0)  # every row the gather may write
    out = torch.zeros((total, inp.num_kv_heads, inp.head_dim), dtype=pool.dtype)
    p = _pool(pool)
    idx = indices.to(torch.int32).contiguous()
    ip = indptr.to(torch.int32).contiguous()
    lp = last_page_len.to(torch.int32).contiguous()
    rc = lib.oracle_gather_ragged(ctypes.byref(p), ctypes.c_int(LAYOUTS[inp.layout]), _ptr(idx), _ptr(ip), _ptr(lp),
                                  _ptr(inp.cum_kv.contiguous()), ctypes.c_int(ip.numel() - 1),
                                  ctypes.c_void_p(out.data_ptr()))
    return out, rc == 0


def attention_ragged(inp, indices, indptr, last_page_len, rows=None, threads: int | None = None):
    """attention() for a batch whose pages come from a ragged page table: each
    request's slice of the flat page ids becomes its block-table row and its kv
    length follows the ragged rule; inp supplies q, the pools, cum_q, scales,
    window and sinks."""
    import copy

    kv = ragged_lengths(indptr, last_page_len, inp.page_size)
    B = kv.numel()
    ip = indptr.tolist()
    width = max([ip[b + 1] - ip[b] for b in range(B)] + [1])
    table = torch.full((B, width), -1, dtype=torch.int32)
    for b in range(B):
        n = ip[b + 1] - ip[b]
        if n > 0:
            table[b, :n] = indices[ip[b]:ip[b + 1]].to(torch.int32)
    r = copy.copy(inp)
    r.block_tables = table
    r.seq_lens = kv
    return attention(r, rows=rows, threads=threads)
