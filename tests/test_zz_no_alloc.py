"""The allocation-free entry point, b2pa_context_attention_noalloc.

Some callers cannot let a library allocate GPU memory: a serving engine
that reserves nearly all of HBM for its KV pool at start-up, or a framework
whose allocator must account for every byte.  For them the library offers
a variant of b2pa_context_attention whose scratch (error word, work counter
and work list) is a fixed array inside the library instead of a cudaMalloc'd
workspace.  These tests call it through the C ABI and check it against the
ordinary entry point: both run the same deterministic kernels, so the outputs
must be equal bit for bit.  One output is also checked against the fp64
oracle, within the parity bars.

The file is named so that pytest collects it last.
"""
import pytest
import torch

import oracle
import workload

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_MAX_FP8 = 2e-2, 2e-3, 3e-2
DEV = "cuda:0"


def _dev(inp):
    d = {n: getattr(inp, n).to(DEV) for n in ("q", "k_pool", "v_pool", "block_tables", "seq_lens", "cum_q", "cum_kv")}
    d["sinks"] = None if inp.sinks is None else inp.sinks.to(DEV)
    return d


def _args(inp, d):
    return (d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_q_len, inp.max_kv_len,
            inp.bmm1_scale, inp.bmm2_scale, d["cum_q"])


def _close_to_oracle(got, inp, fp8):
    ref, st, _ = oracle.attention(inp)
    assert (st == 0).all()
    T, H, D = got.shape
    err = (got.float().cpu().reshape(T * H, D).double() - torch.from_numpy(ref)).abs()
    mx, mean = err.max().item(), err.mean().item()
    if fp8:
        assert mx <= TOL_MAX_FP8, (mx, mean)
    else:
        assert mx <= TOL_MAX and mean <= TOL_MEAN, (mx, mean)


def test_noalloc_matches_context_attention_on_two_calls_in_a_row(cuda_lib):
    b2pa = cuda_lib
    b2pa.set_kernel_path("auto")
    # two different problems, so the second call runs on scratch the first one left behind
    first = workload.build([70, 130, 5], [300, 130, 5], 8, 2, 128, 32, "HND", with_sinks=True, seed=901,
                           table_pad="garbage")
    second = workload.build([96, 1, 40], [4000, 3000, 40], 32, 8, 128, 32, "HND", kv_dtype="fp8_e4m3", seed=902,
                            window_left=300, table_pad="garbage")
    cases = []
    for inp in (first, second):
        d = _dev(inp)
        want = torch.full_like(d["q"], float("nan"))
        b2pa.context_attention(*_args(inp, d), d["cum_kv"], inp.window_left, want, inp.layout, d["sinks"])
        assert b2pa.device_status() == 0
        cases.append((inp, d, want))
    torch.cuda.synchronize()

    status = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    outs = []
    for k, (inp, d, _) in enumerate(cases):  # back to back, no synchronisation in between
        got = torch.full_like(d["q"], float("nan"))
        b2pa.context_attention_noalloc(*_args(inp, d), got, d["cum_kv"], inp.window_left, inp.layout, d["sinks"],
                                       status=status[k:k + 1])
        outs.append(got)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]
    for (inp, _, want), got in zip(cases, outs):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    _close_to_oracle(outs[0], first, fp8=False)


def test_noalloc_rejects_bounds_beyond_its_scratch(cuda_lib):
    b2pa = cuda_lib
    inp = workload.build([64], [64], 32, 8, 128, 32, "HND", seed=903)
    d = _dev(inp)
    out = torch.empty_like(d["q"])
    # 1 request x 8 kv heads x ceil(max_q_len / 64) items > 65536
    with pytest.raises(b2pa.B2paError, match="at most 65536"):
        b2pa.context_attention_noalloc(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                       64 * 8193, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"], out,
                                       d["cum_kv"], -1, inp.layout)
