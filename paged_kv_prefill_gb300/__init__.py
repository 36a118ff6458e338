"""Python binding of libb2pa.so: batched paged-KV context attention on GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/b2pa.h; this module turns torch
tensors into b2pa_tensor descriptors and calls it.  There is no fallback:
if the library is missing, load() raises.

The call mirrors flashinfer.prefill.trtllm_batch_context_with_kv_cache
(FlashInfer API reference, parameter list): ``query``, ``kv_cache`` (a
(K, V) tuple or one [N, 2, ...] tensor), ``block_tables``, ``seq_lens``,
``max_q_len``, ``max_kv_len``, ``bmm1_scale``, ``bmm2_scale``,
``cum_seq_lens_q``, ``cum_seq_lens_kv``, ``window_left``, ``out``,
``kv_layout`` and ``sinks``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libb2pa.so")

B2PA_BF16, B2PA_FP8_E4M3, B2PA_FP32, B2PA_INT32 = 1, 2, 3, 4
LAYOUTS = {"HND": 0, "NHD": 1}
PATH_AUTO, PATH_TCGEN05, PATH_GENERIC = 0, 1, 2
STATUS = {0: "B2PA_OK", -1: "B2PA_ERR_INVALID_ARG", -2: "B2PA_ERR_UNSUPPORTED", -3: "B2PA_ERR_CUDA",
          -4: "B2PA_ERR_DEVICE"}
DEV_BAD_REQUEST, DEV_BAD_PAGE, DEV_TIMEOUT, DEV_BAD_CUM_KV, DEV_OVERFLOW = 1, 2, 4, 8, 16
DEV_BAD_SLOT, DEV_BAD_SCALE = 32, 64

_DTYPES = {
    torch.bfloat16: B2PA_BF16,
    torch.float8_e4m3fn: B2PA_FP8_E4M3,
    torch.float32: B2PA_FP32,
    torch.int32: B2PA_INT32,
}

EXPORTED = [
    "b2pa_context_attention",
    "b2pa_context_attention_tensor_scales",
    "b2pa_batch_decode",
    "b2pa_context_attention_ragged",
    "b2pa_debug_gather_ragged",
    "b2pa_context_attention_noalloc",
    "b2pa_debug_worklist",
    "b2pa_debug_gather",
    "b2pa_append_kv",
    "b2pa_get_device_status",
    "b2pa_set_kernel_path",
    "b2pa_query_path",
    "b2pa_set_debug_checks",
    "b2pa_set_wait_limit_ns",
    "b2pa_debug_inject_stall",
    "b2pa_set_timing_events",
    "b2pa_status_string",
    "b2pa_last_error_message",
    "b2pa_release",
]


class B2paTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 5),
        ("stride", ctypes.c_int64 * 5),
    ]


class B2paError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load libb2pa.so (built by paged_kv_prefill_gb300.build); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with paged_kv_prefill_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(B2paTensor)
    lib.b2pa_context_attention.argtypes = [P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_int32, P, ctypes.c_int32, P, ctypes.c_void_p]
    lib.b2pa_context_attention.restype = ctypes.c_int
    lib.b2pa_context_attention_tensor_scales.argtypes = [P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int32, P, P,
                                                         ctypes.c_int32, P, ctypes.c_int32, P, ctypes.c_void_p]
    lib.b2pa_context_attention_tensor_scales.restype = ctypes.c_int
    lib.b2pa_batch_decode.argtypes = [P, P, P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int32, P, ctypes.c_int32, P, ctypes.c_void_p]
    lib.b2pa_batch_decode.restype = ctypes.c_int
    lib.b2pa_context_attention_ragged.argtypes = [P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int32,
                                                  ctypes.c_float, ctypes.c_float, ctypes.c_int32, P, ctypes.c_int32,
                                                  P, ctypes.c_void_p]
    lib.b2pa_context_attention_ragged.restype = ctypes.c_int
    lib.b2pa_debug_gather_ragged.argtypes = [P, P, P, P, P, P, ctypes.c_int32, P, P, ctypes.c_void_p]
    lib.b2pa_debug_gather_ragged.restype = ctypes.c_int
    lib.b2pa_context_attention_noalloc.argtypes = [P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_float, ctypes.c_float, ctypes.c_int32, P,
                                                   ctypes.c_int32, P, ctypes.c_void_p, ctypes.c_void_p]
    lib.b2pa_context_attention_noalloc.restype = ctypes.c_int
    lib.b2pa_debug_worklist.argtypes = [P, P, P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p]
    lib.b2pa_debug_worklist.restype = ctypes.c_int
    lib.b2pa_debug_gather.argtypes = [P, P, P, P, P, ctypes.c_int32, P, P, ctypes.c_void_p]
    lib.b2pa_debug_gather.restype = ctypes.c_int
    lib.b2pa_append_kv.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_int32, ctypes.c_void_p]
    lib.b2pa_get_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.b2pa_get_device_status.restype = ctypes.c_int
    lib.b2pa_set_kernel_path.argtypes = [ctypes.c_int32]
    lib.b2pa_set_kernel_path.restype = ctypes.c_int
    lib.b2pa_query_path.argtypes = [P, P, P, P, ctypes.c_int32]
    lib.b2pa_query_path.restype = ctypes.c_int
    lib.b2pa_set_timing_events.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.b2pa_set_timing_events.restype = ctypes.c_int
    lib.b2pa_set_debug_checks.argtypes = [ctypes.c_int32]
    lib.b2pa_set_debug_checks.restype = ctypes.c_int
    lib.b2pa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.b2pa_set_wait_limit_ns.restype = ctypes.c_int
    lib.b2pa_debug_inject_stall.argtypes = [ctypes.c_int32]
    lib.b2pa_debug_inject_stall.restype = ctypes.c_int
    lib.b2pa_status_string.argtypes = [ctypes.c_int32]
    lib.b2pa_status_string.restype = ctypes.c_char_p
    lib.b2pa_last_error_message.argtypes = []
    lib.b2pa_last_error_message.restype = ctypes.c_char_p
    lib.b2pa_release.argtypes = []
    lib.b2pa_release.restype = None
    _lib = lib
    return lib


def desc(t: Optional[torch.Tensor]) -> Optional[B2paTensor]:
    """b2pa_tensor describing a torch tensor (strides in elements)."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 5:
        raise ValueError("rank > 5")
    d = B2paTensor()
    d.data = t.data_ptr()
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str):
    if status != 0:
        msg = load().b2pa_last_error_message().decode()
        raise B2paError(status, where, msg)


def split_kv_cache(kv_cache, kv_layout: str) -> Tuple[torch.Tensor, torch.Tensor]:
    """(K, V) pools from a tuple or from one [N, 2, ...] tensor (its two strided views)."""
    if isinstance(kv_cache, (tuple, list)):
        k, v = kv_cache
        return k, v
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2:
        raise ValueError("a single kv_cache tensor must be [num_pages, 2, ...]; the shared K=V form is not supported")
    return kv_cache[:, 0], kv_cache[:, 1]


def context_attention(
    query: torch.Tensor,
    kv_cache: Union[torch.Tensor, Sequence[torch.Tensor]],
    block_tables: torch.Tensor,
    seq_lens: torch.Tensor,
    max_q_len: int,
    max_kv_len: int,
    bmm1_scale: Union[float, torch.Tensor],
    bmm2_scale: Union[float, torch.Tensor],
    cum_seq_lens_q: torch.Tensor,
    cum_seq_lens_kv: Optional[torch.Tensor] = None,
    window_left: int = -1,
    out: Optional[torch.Tensor] = None,
    kv_layout: str = "HND",
    sinks: Optional[torch.Tensor] = None,
    stream=None,
) -> torch.Tensor:
    """Batched context attention over a paged KV cache (see include/b2pa.h).

    bmm1_scale / bmm2_scale are floats, or one-element fp32 device tensors (then
    both must be tensors and b2pa_context_attention_tensor_scales is called)."""
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    if out is None:
        out = torch.empty_like(query)
    if isinstance(sinks, (list, tuple)):
        if len(sinks) != 1:
            raise ValueError("sinks: one fp32 [num_heads] tensor")
        sinks = sinks[0]
    dq, dk, dv, dbt, dsl, dcq = (desc(x) for x in (query, k, v, block_tables, seq_lens, cum_seq_lens_q))
    dck, dsk, do = desc(cum_seq_lens_kv), desc(sinks), desc(out)
    if isinstance(bmm1_scale, torch.Tensor) or isinstance(bmm2_scale, torch.Tensor):
        if not (isinstance(bmm1_scale, torch.Tensor) and isinstance(bmm2_scale, torch.Tensor)):
            raise TypeError("bmm1_scale and bmm2_scale must both be floats or both be tensors")
        d1, d2 = desc(bmm1_scale), desc(bmm2_scale)
        st = lib.b2pa_context_attention_tensor_scales(
            ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(dbt), ctypes.byref(dsl),
            ctypes.byref(dcq), _ref(dck), int(max_q_len), int(max_kv_len), ctypes.byref(d1), ctypes.byref(d2),
            int(window_left), _ref(dsk), LAYOUTS[kv_layout], ctypes.byref(do), ctypes.c_void_p(_stream_handle(stream)),
        )
        _check(st, "b2pa_context_attention_tensor_scales")
        return out
    st = lib.b2pa_context_attention(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(dbt), ctypes.byref(dsl),
        ctypes.byref(dcq), _ref(dck), int(max_q_len), int(max_kv_len), float(bmm1_scale), float(bmm2_scale),
        int(window_left), _ref(dsk), LAYOUTS[kv_layout], ctypes.byref(do), ctypes.c_void_p(_stream_handle(stream)),
    )
    _check(st, "b2pa_context_attention")
    return out


def batch_decode(
    query: torch.Tensor,
    kv_cache: Union[torch.Tensor, Sequence[torch.Tensor]],
    block_tables: torch.Tensor,
    seq_lens: torch.Tensor,
    max_seq_len: int,
    bmm1_scale: float,
    bmm2_scale: float,
    window_left: int = -1,
    out: Optional[torch.Tensor] = None,
    kv_layout: str = "HND",
    sinks: Optional[torch.Tensor] = None,
    q_len_per_req: int = 1,
    stream=None,
) -> torch.Tensor:
    """Decode attention over a paged KV cache: request b owns query rows
    b * q_len_per_req .. + q_len_per_req - 1, the last q_len_per_req positions
    of its seq_lens[b] keys (mirrors trtllm_batch_decode_with_kv_cache as the
    TokenSpeed trtllm backend calls it; see include/b2pa.h)."""
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    if out is None:
        out = torch.empty_like(query)
    if isinstance(sinks, (list, tuple)):
        if len(sinks) != 1:
            raise ValueError("sinks: one fp32 [num_heads] tensor")
        sinks = sinks[0]
    dq, dk, dv, dbt, dsl = (desc(x) for x in (query, k, v, block_tables, seq_lens))
    dsk, do = desc(sinks), desc(out)
    st = lib.b2pa_batch_decode(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(dbt), ctypes.byref(dsl),
        int(q_len_per_req), int(max_seq_len), float(bmm1_scale), float(bmm2_scale), int(window_left), _ref(dsk),
        LAYOUTS[kv_layout], ctypes.byref(do), ctypes.c_void_p(_stream_handle(stream)),
    )
    _check(st, "b2pa_batch_decode")
    return out


def context_attention_ragged(
    query: torch.Tensor,
    kv_cache: Union[torch.Tensor, Sequence[torch.Tensor]],
    paged_kv_indices: torch.Tensor,
    paged_kv_indptr: torch.Tensor,
    paged_kv_last_page_len: torch.Tensor,
    max_q_len: int,
    max_kv_len: int,
    bmm1_scale: float,
    bmm2_scale: float,
    cum_seq_lens_q: torch.Tensor,
    window_left: int = -1,
    out: Optional[torch.Tensor] = None,
    kv_layout: str = "HND",
    sinks: Optional[torch.Tensor] = None,
    stream=None,
) -> torch.Tensor:
    """context_attention with FlashInfer's ragged page table (flat page ids, their
    per-request offsets and the valid tokens of each last page) in place of
    block_tables and seq_lens (see include/b2pa.h)."""
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    if out is None:
        out = torch.empty_like(query)
    if isinstance(sinks, (list, tuple)):
        if len(sinks) != 1:
            raise ValueError("sinks: one fp32 [num_heads] tensor")
        sinks = sinks[0]
    d = [desc(x) for x in (query, k, v, paged_kv_indices, paged_kv_indptr, paged_kv_last_page_len, cum_seq_lens_q)]
    dsk, do = desc(sinks), desc(out)
    st = lib.b2pa_context_attention_ragged(
        *(ctypes.byref(x) for x in d), int(max_q_len), int(max_kv_len), float(bmm1_scale), float(bmm2_scale),
        int(window_left), _ref(dsk), LAYOUTS[kv_layout], ctypes.byref(do), ctypes.c_void_p(_stream_handle(stream)),
    )
    _check(st, "b2pa_context_attention_ragged")
    return out


def context_attention_noalloc(
    query: torch.Tensor,
    kv_cache: Union[torch.Tensor, Sequence[torch.Tensor]],
    block_tables: torch.Tensor,
    seq_lens: torch.Tensor,
    max_q_len: int,
    max_kv_len: int,
    bmm1_scale: float,
    bmm2_scale: float,
    cum_seq_lens_q: torch.Tensor,
    out: torch.Tensor,
    cum_seq_lens_kv: Optional[torch.Tensor] = None,
    window_left: int = -1,
    kv_layout: str = "HND",
    sinks: Optional[torch.Tensor] = None,
    status: Optional[torch.Tensor] = None,
    stream=None,
) -> torch.Tensor:
    """context_attention through b2pa_context_attention_noalloc: the library
    allocates no GPU memory (its scratch is a fixed array of 65536 work items;
    see include/b2pa.h).  `out` must be given; `status`, if given, is a device
    int32/uint32 tensor of one element that receives the call's device error bits."""
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    if isinstance(sinks, (list, tuple)):
        if len(sinks) != 1:
            raise ValueError("sinks: one fp32 [num_heads] tensor")
        sinks = sinks[0]
    if status is not None:
        # the library writes 4 bytes there with a device-to-device copy
        if (not status.is_cuda or status.device != query.device or status.dtype not in (torch.int32, torch.uint32)
                or status.numel() < 1 or not status.is_contiguous()):
            raise ValueError("status must be a contiguous int32/uint32 CUDA tensor of at least one element on "
                             "the query's device")
    dq, dk, dv, dbt, dsl, dcq = (desc(x) for x in (query, k, v, block_tables, seq_lens, cum_seq_lens_q))
    dck, dsk, do = desc(cum_seq_lens_kv), desc(sinks), desc(out)
    st = lib.b2pa_context_attention_noalloc(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(dbt), ctypes.byref(dsl),
        ctypes.byref(dcq), _ref(dck), int(max_q_len), int(max_kv_len), float(bmm1_scale), float(bmm2_scale),
        int(window_left), _ref(dsk), LAYOUTS[kv_layout], ctypes.byref(do),
        ctypes.c_void_p(status.data_ptr() if status is not None else 0), ctypes.c_void_p(_stream_handle(stream)),
    )
    _check(st, "b2pa_context_attention_noalloc")
    return out


def debug_worklist(query, k_pool, block_tables, seq_lens, cum_seq_lens_q, max_q_len, max_kv_len,
                   window_left=-1, kv_layout="HND", stream=None):
    """Run the scheduler alone; returns (items int32 [n, 4] on the host, geometry dict)."""
    import numpy as np

    lib = load()
    H = query.shape[1]
    Hkv = k_pool.shape[1] if kv_layout == "HND" else k_pool.shape[2]
    per = 128 // (H // Hkv)  # tokens of one query tile: an item holds at least one
    cap = max(1, seq_lens.numel() * Hkv * ((max(max_q_len, 1) + per - 1) // per))
    items = np.zeros((cap, 4), dtype=np.int32)
    n = ctypes.c_int32(0)
    geo = (ctypes.c_int32 * 4)()
    d = [desc(x) for x in (query, k_pool, block_tables, seq_lens, cum_seq_lens_q)]
    st = lib.b2pa_debug_worklist(*(ctypes.byref(x) for x in d), int(max_q_len), int(max_kv_len), int(window_left),
                                 LAYOUTS[kv_layout], items.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(n),
                                 ctypes.byref(geo), ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "b2pa_debug_worklist")
    geometry = {"rows_per_tile": geo[0], "n_qtiles": geo[1], "kv_tile": geo[2], "cost_cap": geo[3]}
    return items[: min(n.value, cap)].copy(), geometry


def debug_gather(kv_cache, block_tables, seq_lens, cum_seq_lens_kv, total_rows: int, kv_layout="HND", stream=None):
    """Contiguous [total_rows, Hkv, D] K and V gathered through the kernel's page loads."""
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    Hkv = k.shape[1] if kv_layout == "HND" else k.shape[2]
    D = k.shape[3]
    k_out = torch.zeros((total_rows, Hkv, D), dtype=k.dtype, device=k.device)
    v_out = torch.zeros_like(k_out)
    d = [desc(x) for x in (k, v, block_tables, seq_lens, cum_seq_lens_kv)]
    dko, dvo = desc(k_out), desc(v_out)
    st = lib.b2pa_debug_gather(*(ctypes.byref(x) for x in d), LAYOUTS[kv_layout], ctypes.byref(dko),
                               ctypes.byref(dvo), ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "b2pa_debug_gather")
    return k_out, v_out


def debug_gather_ragged(kv_cache, paged_kv_indices, paged_kv_indptr, paged_kv_last_page_len, cum_seq_lens_kv,
                        total_rows: int, kv_layout="HND", stream=None):
    """debug_gather for the ragged page table."""
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    Hkv = k.shape[1] if kv_layout == "HND" else k.shape[2]
    D = k.shape[3]
    k_out = torch.zeros((total_rows, Hkv, D), dtype=k.dtype, device=k.device)
    v_out = torch.zeros_like(k_out)
    d = [desc(x) for x in (k, v, paged_kv_indices, paged_kv_indptr, paged_kv_last_page_len, cum_seq_lens_kv)]
    dko, dvo = desc(k_out), desc(v_out)
    st = lib.b2pa_debug_gather_ragged(*(ctypes.byref(x) for x in d), LAYOUTS[kv_layout], ctypes.byref(dko),
                                      ctypes.byref(dvo), ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "b2pa_debug_gather_ragged")
    return k_out, v_out


def append_kv(k_new: torch.Tensor, v_new: torch.Tensor, kv_cache, cache_loc: torch.Tensor, k_scale: float = 1.0,
              v_scale: float = 1.0, kv_layout: str = "HND", stream=None):
    """Write token n's K/V rows (bf16 [T, Hkv, D]) into slot cache_loc[n] (int32) of the pools, in place.

    An e4m3 pool stores x / scale rounded to the nearest e4m3 value (saturating at +-448); a bf16
    pool stores the values unchanged.  Slots outside the pool are skipped and flagged in
    device_status().
    """
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    d = [desc(x) for x in (k_new, v_new, k, v, cache_loc)]
    st = lib.b2pa_append_kv(*(ctypes.byref(x) for x in d), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
                            LAYOUTS[kv_layout], ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "b2pa_append_kv")


def device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device error bits of its workspace."""
    lib = load()
    bits = ctypes.c_uint32(0)
    st = lib.b2pa_get_device_status(ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(bits))
    if st not in (0, -4):
        _check(st, "b2pa_get_device_status")
    return bits.value


def set_kernel_path(path: Union[int, str]):
    m = {"auto": PATH_AUTO, "tcgen05": PATH_TCGEN05, "generic": PATH_GENERIC}
    _check(load().b2pa_set_kernel_path(m[path] if isinstance(path, str) else int(path)), "b2pa_set_kernel_path")


def query_path(query, kv_cache, out=None, kv_layout="HND") -> str:
    lib = load()
    k, v = split_kv_cache(kv_cache, kv_layout)
    if out is None:
        out = query
    st = lib.b2pa_query_path(ctypes.byref(desc(query)), ctypes.byref(desc(k)), ctypes.byref(desc(v)),
                             ctypes.byref(desc(out)), LAYOUTS[kv_layout])
    if st < 0:
        _check(st, "b2pa_query_path")
    return {PATH_TCGEN05: "tcgen05", PATH_GENERIC: "generic"}[st]


def set_wait_limit_ns(limit_ns: int):
    """Longest pipeline wait inside the attention kernel (ns); 0 restores the 2 s default."""
    _check(load().b2pa_set_wait_limit_ns(int(limit_ns)), "b2pa_set_wait_limit_ns")


def debug_inject_stall(on: bool):
    """Failure-detection tests: later attention kernels make one wait nothing completes (see include/b2pa.h)."""
    _check(load().b2pa_debug_inject_stall(1 if on else 0), "b2pa_debug_inject_stall")


def set_debug_checks(on: bool):
    load().b2pa_set_debug_checks(1 if on else 0)


def set_timing_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]):
    """Record start/stop around each later attention-kernel launch (tensor-core path); None, None turns it off."""
    lib = load()
    if start is None or stop is None:
        lib.b2pa_set_timing_events(None, None)
    else:
        lib.b2pa_set_timing_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))


def release():
    load().b2pa_release()
