"""GPU parity of the decode sibling, b2pa_batch_decode, through the C ABI.

A decode batch is the context operation with every request holding the same
number of query tokens (q_len_per_req, 1 for plain decoding and more for
speculative verification, as the TokenSpeed trtllm backend's forward_decode
passes it), so the fp64 oracle's row definition covers it unchanged: its
inputs are built with q_lens = [q_len_per_req] * batch.  Every row of every
case is compared, within the same bars as the context parity tests
(tests/test_gpu_parity.py), across ragged kv lengths up to 32768 that make
the tensor-core path cut requests into several kv chunks.
"""
import numpy as np
import pytest
import torch

import workload
from test_gpu_parity import DEV, _compare, _to_dev

pytestmark = pytest.mark.gpu


def _decode_inputs(batch, n, kv_max, seed, H=32, Hkv=8, D=128, P=32, layout="HND", kvd="bf16", window=-1,
                   sinks=False, kv_min=None):
    g = torch.Generator().manual_seed(seed)
    lo = n if kv_min is None else kv_min
    kv = torch.randint(lo, kv_max + 1, (batch,), generator=g).tolist()
    return workload.build([n] * batch, kv, H, Hkv, D, P, layout, kv_dtype=kvd, window_left=window, with_sinks=sinks,
                          seed=seed, table_pad="garbage")


def _decode(b2pa, inp, n, path="auto", out=None):
    b2pa.set_kernel_path(path)
    try:
        d = _to_dev(inp)
        if out is None:
            out = torch.full_like(d["q"], float("nan"))
        b2pa.batch_decode(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_kv_len,
                          inp.bmm1_scale, inp.bmm2_scale, inp.window_left, out, inp.layout, d["sinks"],
                          q_len_per_req=n)
        bits = b2pa.device_status()
    finally:
        b2pa.set_kernel_path("auto")
    return out, bits


DECODE_CASES = [
    # (batch, q_len_per_req, kv_max, H, Hkv, D, P, layout, kv dtype, window, sinks)
    (16, 1, 32768, 32, 8, 128, 32, "HND", "bf16", -1, False),     # long ragged rows: many kv chunks
    (16, 4, 32768, 32, 8, 128, 32, "HND", "bf16", -1, True),      # speculative verification, sinks
    (2, 1, 32768, 32, 8, 128, 32, "NHD", "bf16", -1, False),      # two requests: dozens of chunks each
    (64, 1, 4096, 32, 8, 128, 16, "HND", "bf16", -1, False),      # a larger batch, few or no chunks
    (16, 4, 32768, 32, 8, 128, 32, "HND", "fp8_e4m3", -1, False),  # e4m3 cache
    (8, 2, 20000, 64, 8, 64, 16, "HND", "bf16", 127, True),       # D = 64, sliding window + sinks
    (8, 3, 9000, 12, 4, 128, 64, "NHD", "bf16", -1, False),       # G = 3 (rows 126 of 128), q_len 3
    (4, 40, 9000, 32, 8, 128, 32, "HND", "fp8_e4m3", -1, True),   # e4m3, more rows than one tile: not split
]


@pytest.mark.parametrize("case", range(len(DECODE_CASES)))
def test_decode_parity(cuda_lib, case):
    B, n, kv_max, H, Hkv, D, P, lay, kvd, W, sinks = DECODE_CASES[case]
    inp = _decode_inputs(B, n, kv_max, seed=500 + case, H=H, Hkv=Hkv, D=D, P=P, layout=lay, kvd=kvd, window=W,
                         sinks=sinks)
    out, bits = _decode(cuda_lib, inp, n)
    assert bits == 0
    _compare(out, inp)


@pytest.mark.parametrize("case", [0, 1, 5])
def test_decode_generic_path(cuda_lib, case):
    B, n, kv_max, H, Hkv, D, P, lay, kvd, W, sinks = DECODE_CASES[case]
    inp = _decode_inputs(B, n, kv_max // 4, seed=600 + case, H=H, Hkv=Hkv, D=D, P=P, layout=lay, kvd=kvd, window=W,
                         sinks=sinks)
    out, bits = _decode(cuda_lib, inp, n, path="generic")
    assert bits == 0
    _compare(out, inp)


def test_decode_matches_context_call(cuda_lib):
    """The same batch through the context entry point (cum_q = b * q_len_per_req)
    and through decode: both meet the oracle's bars, and they agree closely
    (the decode path sums its kv chunks in another order)."""
    B, n = 8, 4
    inp = _decode_inputs(B, n, 16000, seed=700)
    dec, bits = _decode(cuda_lib, inp, n)
    assert bits == 0
    d = _to_dev(inp)
    ctx = torch.full_like(d["q"], float("nan"))
    cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], n,
                               inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"], d["cum_kv"], -1, ctx,
                               inp.layout)
    assert cuda_lib.device_status() == 0
    _compare(dec, inp)
    _compare(ctx, inp)
    assert (dec.float() - ctx.float()).abs().max().item() <= 2e-2


def test_decode_short_sequence_flagged(cuda_lib):
    """seq_lens[b] < q_len_per_req leaves query rows without a visible key: the
    request is rejected on the device and its rows are not written."""
    B, n = 4, 4
    inp = _decode_inputs(B, n, 300, seed=701, kv_min=10)
    d = _to_dev(inp)
    d["seq_lens"][2] = 3
    out = torch.full_like(d["q"], 7.0)
    cuda_lib.batch_decode(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_kv_len,
                          inp.bmm1_scale, inp.bmm2_scale, -1, out, inp.layout, None, q_len_per_req=n)
    assert cuda_lib.device_status() & cuda_lib.DEV_BAD_REQUEST
    assert (out[2 * n:3 * n] == 7).all()
    H = inp.num_heads
    rows = np.array([t * H + h for t in list(range(0, 2 * n)) + list(range(3 * n, 4 * n)) for h in range(H)])
    _compare(out, inp, rows=rows)


def test_decode_rejects_wrong_token_count(cuda_lib):
    inp = _decode_inputs(4, 2, 300, seed=702)
    d = _to_dev(inp)
    with pytest.raises(cuda_lib.B2paError, match="q_len_per_req"):
        cuda_lib.batch_decode(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_kv_len,
                              inp.bmm1_scale, inp.bmm2_scale, -1, None, inp.layout, None, q_len_per_req=3)


@pytest.mark.parametrize("n,kvd", [(1, "bf16"), (4, "bf16"), (1, "fp8_e4m3")])
def test_decode_named_workloads(cuda_lib, n, kvd):
    """The timed decode batches (32 requests, kv lengths uniform up to 32768),
    every row against the oracle."""
    inp = workload.decode_config(n, kv_dtype=kvd)
    out, bits = _decode(cuda_lib, inp, n)
    assert bits == 0
    _compare(out, inp)
