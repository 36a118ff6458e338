"""The C-ABI library without a GPU: it builds, loads, exports every entry
point include/b2pa.h declares, and rejects malformed arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_prefill_gb300 import build

    build.build()
    import paged_kv_prefill_gb300 as pkg

    return pkg.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "b2pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(b2pa_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    import paged_kv_prefill_gb300 as pkg

    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(pkg.EXPORTED) == names


def test_status_strings(lib):
    assert lib.b2pa_status_string(0) == b"B2PA_OK"
    assert lib.b2pa_status_string(-1) == b"B2PA_ERR_INVALID_ARG"
    assert lib.b2pa_status_string(-4) == b"B2PA_ERR_DEVICE"


def test_kernel_path_option(lib):
    assert lib.b2pa_set_kernel_path(2) == 0
    assert lib.b2pa_set_kernel_path(0) == 0
    assert lib.b2pa_set_kernel_path(9) == -1
    assert b"unknown kernel path" in lib.b2pa_last_error_message()


def _fake(shape, dtype, base=1 << 20):
    """A descriptor with a fake (never dereferenced) pointer and contiguous strides."""
    import paged_kv_prefill_gb300 as pkg

    d = pkg.B2paTensor()
    d.data = base
    d.dtype = dtype
    d.ndim = len(shape)
    st = 1
    strides = []
    for s in reversed(shape):
        strides.append(st)
        st *= s
    strides.reverse()
    for i, s in enumerate(shape):
        d.shape[i] = s
        d.stride[i] = strides[i]
    return d


def _call(lib, q, k, v, bt, sl, cq, bmm1=0.1, layout=0, out=None, sinks=None):
    r = ctypes.byref
    out = out or q
    return lib.b2pa_context_attention(r(q), r(k), r(v), r(bt), r(sl), r(cq), None, 8, 8, bmm1, 1.0, -1,
                                      None if sinks is None else r(sinks), layout, r(out), None)


def test_host_validation_without_gpu(lib):
    BF, F8, F32, I32 = 1, 2, 3, 4
    q = _fake([8, 4, 128], BF)
    k = _fake([10, 2, 32, 128], BF)
    v = _fake([10, 2, 32, 128], BF)
    bt = _fake([2, 4], I32)
    sl = _fake([2], I32)
    cq = _fake([3], I32)
    # H % Hkv != 0
    assert _call(lib, _fake([8, 3, 128], BF), k, v, bt, sl, cq, out=_fake([8, 3, 128], BF)) == -1
    # head_dim mismatch
    assert _call(lib, _fake([8, 4, 64], BF), k, v, bt, sl, cq, out=_fake([8, 4, 64], BF)) == -1
    # K/V dtype mismatch
    assert _call(lib, q, k, _fake([10, 2, 32, 128], F8), bt, sl, cq) == -1
    # cum_q length
    assert _call(lib, q, k, v, bt, sl, _fake([2], I32)) == -1
    # block table rows
    assert _call(lib, q, k, v, _fake([3, 4], I32), sl, cq) == -1
    # bmm1_scale must be > 0 and finite
    assert _call(lib, q, k, v, bt, sl, cq, bmm1=0.0) == -1
    assert _call(lib, q, k, v, bt, sl, cq, bmm1=float("nan")) == -1
    # layout
    assert _call(lib, q, k, v, bt, sl, cq, layout=5) == -1
    # sinks length
    assert _call(lib, q, k, v, bt, sl, cq, sinks=_fake([3], F32)) == -1
    # non-unit head_dim stride
    bad = _fake([8, 4, 128], BF)
    bad.stride[2] = 2
    assert _call(lib, bad, k, v, bt, sl, cq) == -1
    # head_dim above 256
    assert _call(lib, _fake([8, 4, 512], BF), _fake([10, 2, 32, 512], BF), _fake([10, 2, 32, 512], BF), bt, sl, cq,
                 out=_fake([8, 4, 512], BF)) == -2
    assert len(lib.b2pa_last_error_message()) > 0


def test_tensor_scale_validation_without_gpu(lib):
    """The device-tensor scales are checked on the host for what the host can
    see: one fp32 element, 4-byte aligned, not null."""
    BF, F32, I32 = 1, 3, 4
    q = _fake([8, 4, 128], BF)
    k = _fake([10, 2, 32, 128], BF)
    bt, sl, cq = _fake([2, 4], I32), _fake([2], I32), _fake([3], I32)
    r = ctypes.byref

    def call(s1, s2):
        return lib.b2pa_context_attention_tensor_scales(r(q), r(k), r(k), r(bt), r(sl), r(cq), None, 8, 8,
                                                        None if s1 is None else r(s1), None if s2 is None else r(s2),
                                                        -1, None, 0, r(q), None)

    good = _fake([1], F32)
    assert call(None, good) == -1
    assert call(good, _fake([2], F32)) == -1                 # two elements
    assert call(_fake([1], BF), good) == -1                  # not fp32
    assert call(good, _fake([1], F32, base=(1 << 20) + 2)) == -1  # misaligned
    assert b"bmm2_scale" in lib.b2pa_last_error_message()


def test_binding_describes_torch_tensors():
    import paged_kv_prefill_gb300 as pkg

    t = torch.zeros((3, 4, 8), dtype=torch.bfloat16).permute(1, 0, 2)
    d = pkg.desc(t)
    assert d.ndim == 3 and d.dtype == 1
    assert list(d.shape)[:3] == [4, 3, 8] and list(d.stride)[:3] == [8, 32, 1]
    kv = torch.zeros((5, 2, 2, 16, 64), dtype=torch.float8_e4m3fn)
    k, v = pkg.split_kv_cache(kv, "HND")
    assert k.shape == (5, 2, 16, 64) and k.stride(0) == 2 * 2 * 16 * 64
    assert v.data_ptr() - k.data_ptr() == 2 * 16 * 64


def _append(lib, kn, vn, k, v, loc, ks=1.0, vs=1.0, layout=0):
    r = ctypes.byref
    return lib.b2pa_append_kv(r(kn), r(vn), r(k), r(v), r(loc), ks, vs, layout, None)


def test_append_host_validation_without_gpu(lib):
    BF, F8, F32, I32 = 1, 2, 3, 4
    kn, vn = _fake([6, 2, 128], BF), _fake([6, 2, 128], BF)
    k, v = _fake([10, 2, 32, 128], BF), _fake([10, 2, 32, 128], BF)
    loc = _fake([6], I32)
    # kv heads or head_dim differ from the pools
    assert _append(lib, _fake([6, 3, 128], BF), _fake([6, 3, 128], BF), k, v, loc) == -1
    assert _append(lib, _fake([6, 2, 64], BF), _fake([6, 2, 64], BF), k, v, loc) == -1
    # new rows must be bf16, and K and V alike
    assert _append(lib, _fake([6, 2, 128], F32), _fake([6, 2, 128], F32), k, v, loc) == -1
    assert _append(lib, kn, _fake([7, 2, 128], BF), k, v, loc) == -1
    # cache_loc: int32, one per token
    assert _append(lib, kn, vn, k, v, _fake([5], I32)) == -1
    assert _append(lib, kn, vn, k, v, _fake([6], F32)) == -1
    # an e4m3 pool needs finite scales > 0
    k8, v8 = _fake([10, 2, 32, 128], F8), _fake([10, 2, 32, 128], F8)
    assert _append(lib, kn, vn, k8, v8, loc, ks=0.0) == -1
    assert _append(lib, kn, vn, k8, v8, loc, vs=float("inf")) == -1
    # token stride not a multiple of 8 elements
    bk, bv = _fake([6, 2, 128], BF), _fake([6, 2, 128], BF)
    bk.stride[0] = bv.stride[0] = 260
    assert _append(lib, bk, bv, k, v, loc) == -1
    # head_dim not a multiple of 8
    assert _append(lib, _fake([6, 2, 12], BF), _fake([6, 2, 12], BF), _fake([10, 2, 32, 12], BF),
                   _fake([10, 2, 32, 12], BF), loc) == -2
    # no tokens: nothing to do, and no CUDA call; empty tensors may carry null data pointers
    assert _append(lib, _fake([0, 2, 128], BF), _fake([0, 2, 128], BF), k, v, _fake([0], I32)) == 0
    assert _append(lib, _fake([0, 2, 128], BF, base=0), _fake([0, 2, 128], BF, base=0), k, v,
                   _fake([0], I32, base=0)) == 0
    # but not when there are tokens
    assert _append(lib, _fake([6, 2, 128], BF, base=0), vn, k, v, loc) == -1
