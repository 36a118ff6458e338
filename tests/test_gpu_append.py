"""The K/V write into the paged pools (b2pa_append_kv) on the GPU, against
the oracle bit for bit: the bf16 copy and the e4m3 quantising write, both
layouts, strided token rows, saturating scales, slots outside the pool, and
the new tokens of the ragged FP8 workload at their block-table positions."""
import pytest
import torch

import oracle
import workload
from bench import new_token_slots

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pools(layout, fp8, N, P, H, D, g):
    shape = (N, H, P, D) if layout == "HND" else (N, P, H, D)
    if fp8:
        k = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
        v = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
    else:
        k = torch.randn(shape, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, generator=g).to(torch.bfloat16)
    return k, v


def _new_rows(T, H, D, g, strided):
    """Token rows [T, H, D] bf16 on the host and on the device (strided: K and V views of one [T, 2, H, D])."""
    if strided:
        kv = (torch.randn((T, 2, H, D), generator=g) * 4).to(torch.bfloat16)
        kvd = kv.to(DEV)
        return kv[:, 0], kv[:, 1], kvd[:, 0], kvd[:, 1]
    k = (torch.randn((T, H, D), generator=g) * 4).to(torch.bfloat16)
    v = (torch.randn((T, H, D), generator=g) * 3).to(torch.bfloat16)
    return k, v, k.to(DEV), v.to(DEV)


def _same_bits(dev_t, host_t):
    return torch.equal(dev_t.cpu().view(torch.uint8), host_t.view(torch.uint8))


CASES = [
    # layout, fp8, T, N, P, H, D, scales, strided
    ("HND", False, 777, 64, 32, 8, 128, (1.0, 1.0), False),
    ("NHD", False, 300, 40, 64, 4, 64, (1.0, 1.0), True),
    ("HND", True, 500, 48, 32, 8, 128, (0.02, 0.015), True),
    ("NHD", True, 400, 64, 16, 4, 64, (0.012, 0.004), False),  # quotients up to ~1000: saturation
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{'e4m3' if c[1] else 'bf16'}-D{c[6]}-P{c[4]}" for c in CASES])
def test_append_bit_exact(cuda_lib, case):
    b2pa = cuda_lib
    layout, fp8, T, N, P, H, D, scales, strided = case
    g = torch.Generator().manual_seed(101 + CASES.index(case))
    kp, vp = _pools(layout, fp8, N, P, H, D, g)
    k_new, v_new, dk_new, dv_new = _new_rows(T, H, D, g, strided)
    loc = torch.randperm(N * P, generator=g)[:T].to(torch.int32)
    dk, dv = kp.to(DEV), vp.to(DEV)
    want_k, want_v = kp.clone(), vp.clone()
    assert oracle.append_kv(k_new, v_new, want_k, want_v, loc, scales[0], scales[1], layout) == 0
    b2pa.append_kv(dk_new, dv_new, (dk, dv), loc.to(DEV), scales[0], scales[1], layout)
    assert b2pa.device_status() == 0
    assert _same_bits(dk, want_k) and _same_bits(dv, want_v)


def test_append_skips_and_flags_slots_outside_the_pool(cuda_lib):
    b2pa = cuda_lib
    g = torch.Generator().manual_seed(41)
    N, P, H, D, T = 16, 16, 2, 64, 50
    kp, vp = _pools("HND", True, N, P, H, D, g)
    k_new, v_new, dk_new, dv_new = _new_rows(T, H, D, g, False)
    loc = torch.randperm(N * P, generator=g)[:T].to(torch.int32)
    loc[5], loc[17], loc[49] = -1, N * P, 2 ** 31 - 1
    dk, dv = kp.to(DEV), vp.to(DEV)
    want_k, want_v = kp.clone(), vp.clone()
    assert oracle.append_kv(k_new, v_new, want_k, want_v, loc, 0.05, 0.05, "HND") == 3
    b2pa.append_kv(dk_new, dv_new, (dk, dv), loc.to(DEV), 0.05, 0.05, "HND")
    assert b2pa.device_status() == 32  # B2PA_DEV_BAD_SLOT
    assert _same_bits(dk, want_k) and _same_bits(dv, want_v)


def test_append_of_no_tokens_is_a_no_op(cuda_lib):
    b2pa = cuda_lib
    g = torch.Generator().manual_seed(43)
    kp, vp = _pools("HND", False, 4, 16, 2, 64, g)
    dk, dv = kp.to(DEV), vp.to(DEV)
    empty = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    b2pa.append_kv(empty, empty, (dk, dv), torch.empty((0,), dtype=torch.int32, device=DEV))
    assert b2pa.device_status() == 0
    assert _same_bits(dk, kp) and _same_bits(dv, vp)


def test_append_new_tokens_of_the_ragged_fp8_workload(cuda_lib):
    """Full size: every new token of the ragged FP8 workload written into its e4m3 pool."""
    b2pa = cuda_lib
    inp = workload.config(5)
    g = torch.Generator().manual_seed(45)
    T, H, D = inp.q.shape[0], inp.num_kv_heads, inp.head_dim
    k_new, v_new, dk_new, dv_new = _new_rows(T, H, D, g, False)
    loc = new_token_slots(inp)
    ks, vs = inp.meta["k_scale"], inp.meta["v_scale"]
    dk, dv = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
    want_k, want_v = inp.k_pool.clone(), inp.v_pool.clone()
    assert oracle.append_kv(k_new, v_new, want_k, want_v, loc, ks, vs, inp.layout) == 0
    b2pa.append_kv(dk_new, dv_new, (dk, dv), loc.to(DEV), ks, vs, inp.layout)
    assert b2pa.device_status() == 0
    assert _same_bits(dk, want_k) and _same_bits(dv, want_v)
