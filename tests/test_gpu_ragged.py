"""GPU parity of the ragged page table (FlashInfer's paged_kv_indices /
paged_kv_indptr / paged_kv_last_page_len) through the C ABI: the ragged debug
gather bit for bit against the oracle's ragged gather, and the attention
against the oracle fed the same ragged table, on both kernel paths."""
import numpy as np
import pytest
import torch

import oracle
import workload
from test_gpu_parity import DEV, TC_CASES, _errors, TOL_MAX, TOL_MEAN, TOL_MAX_FP8, TOL_ROW_REL

pytestmark = pytest.mark.gpu


def _ragged_dev(inp):
    idx, ip, last = workload.ragged_page_table(inp)
    return idx, ip, last, idx.to(DEV), ip.to(DEV), last.to(DEV)


def _compare_ragged(got, inp, idx, ip, last, rows=None):
    ref, st, _ = oracle.attention_ragged(inp, idx, ip, last, rows=rows)
    assert (st == 0).all()
    T, H, D = got.shape
    g = got.float().cpu().reshape(T * H, D).double()
    if rows is not None:
        g = g[torch.as_tensor(rows)]
    assert torch.isfinite(g).all()
    mx, mean, rel, row_rel = _errors(g, torch.from_numpy(ref))
    msg = f"max_abs={mx:.3e} mean_abs={mean:.3e} max_row_rel={row_rel:.3e}"
    if inp.meta.get("kv_dtype") == "fp8_e4m3":
        assert mx <= TOL_MAX_FP8, msg
    else:
        assert mx <= TOL_MAX and mean <= TOL_MEAN, msg
    assert row_rel <= TOL_ROW_REL, msg


def _run_ragged(b2pa, inp, path="auto", out=None):
    idx, ip, last, d_idx, d_ip, d_last = _ragged_dev(inp)
    b2pa.set_kernel_path(path)
    try:
        q = inp.q.to(DEV)
        k, v = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
        if out is None:
            out = torch.full_like(q, float("nan"))
        b2pa.context_attention_ragged(q, (k, v), d_idx, d_ip, d_last, inp.max_q_len, inp.max_kv_len, inp.bmm1_scale,
                                      inp.bmm2_scale, inp.cum_q.to(DEV), inp.window_left, out, inp.layout,
                                      None if inp.sinks is None else inp.sinks.to(DEV))
        bits = b2pa.device_status()
    finally:
        b2pa.set_kernel_path("auto")
    return out, bits, (idx, ip, last)


@pytest.mark.parametrize("layout,kvd,P,D", [("HND", "bf16", 32, 128), ("NHD", "bf16", 16, 64),
                                            ("HND", "fp8_e4m3", 32, 128), ("NHD", "bf16", 256, 128),
                                            ("HND", "bf16", 8, 64)])
def test_debug_gather_ragged_bit_exact(cuda_lib, layout, kvd, P, D):
    inp = workload.build([10, 1, 0, 300], [130, 77, 0, 600], 8, 4, D, P, layout, kv_dtype=kvd, seed=31,
                         table_pad="garbage")
    idx, ip, last, d_idx, d_ip, d_last = _ragged_dev(inp)
    total = int(inp.seq_lens.sum())
    k_out, v_out = cuda_lib.debug_gather_ragged((inp.k_pool.to(DEV), inp.v_pool.to(DEV)), d_idx, d_ip, d_last,
                                                inp.cum_kv.to(DEV), total, layout)
    assert cuda_lib.device_status() == 0
    k_ref, ok1 = oracle.gather_ragged(inp, idx, ip, last, "k")
    v_ref, ok2 = oracle.gather_ragged(inp, idx, ip, last, "v")
    assert ok1 and ok2
    assert torch.equal(k_out.cpu().view(torch.uint8), k_ref.view(torch.uint8))
    assert torch.equal(v_out.cpu().view(torch.uint8), v_ref.view(torch.uint8))


@pytest.mark.parametrize("path", ["tcgen05", "generic"])
@pytest.mark.parametrize("case", [0, 1, 3, 5, 9, 11])
def test_ragged_attention_parity(cuda_lib, case, path):
    ql, kl, H, Hkv, D, P, lay, W, sinks, kvd = TC_CASES[case]
    inp = workload.build(ql, kl, H, Hkv, D, P, lay, kv_dtype=kvd, window_left=W, with_sinks=sinks, seed=800 + case)
    out, bits, (idx, ip, last) = _run_ragged(cuda_lib, inp, path)
    assert bits == 0
    _compare_ragged(out, inp, idx, ip, last)


def test_ragged_equals_block_table_call(cuda_lib):
    """The same pages described both ways give the same bits (the kernels see
    the same keys in the same order)."""
    inp = workload.config(2)
    out_r, bits, _ = _run_ragged(cuda_lib, inp)
    assert bits == 0
    d = {n: getattr(inp, n).to(DEV) for n in ("q", "k_pool", "v_pool", "block_tables", "seq_lens", "cum_q")}
    out_b = torch.full_like(d["q"], float("nan"))
    cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_q_len,
                               inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"], None, -1, out_b,
                               inp.layout)
    assert cuda_lib.device_status() == 0
    assert torch.equal(out_r.view(torch.int16), out_b.view(torch.int16))


@pytest.mark.parametrize("path", ["tcgen05", "generic"])
def test_ragged_bad_last_page_len_flagged(cuda_lib, path):
    inp = workload.build([30, 20, 25], [60, 40, 25], 8, 2, 128, 32, "HND", seed=32)
    idx, ip, last = workload.ragged_page_table(inp)
    last[1] = 0  # a request with pages must have 1..P tokens in its last page
    T, H, D = inp.q.shape
    out = torch.full((T, H, D), 7.0, dtype=torch.bfloat16, device=DEV)
    cuda_lib.set_kernel_path(path)
    try:
        cuda_lib.context_attention_ragged(inp.q.to(DEV), (inp.k_pool.to(DEV), inp.v_pool.to(DEV)), idx.to(DEV),
                                          ip.to(DEV), last.to(DEV), inp.max_q_len, inp.max_kv_len, inp.bmm1_scale,
                                          inp.bmm2_scale, inp.cum_q.to(DEV), -1, out, "HND")
        bits = cuda_lib.device_status()
    finally:
        cuda_lib.set_kernel_path("auto")
    assert bits & cuda_lib.DEV_BAD_REQUEST
    assert (out[30:50] == 7).all()
    rows = np.array([t * H + h for t in list(range(0, 30)) + list(range(50, 75)) for h in range(H)])
    ref, st, _ = oracle.attention(inp, rows=rows)
    err = (out.float().cpu().reshape(T * H, D).double()[torch.as_tensor(rows)] - torch.from_numpy(ref)).abs()
    assert err.max().item() <= TOL_MAX
