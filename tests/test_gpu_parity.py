"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Bars for bf16 outputs on N(0,1) inputs:
max-abs <= 2e-2 and mean-abs <= 2e-3; FP8 KV: max-abs <= 3e-2 against the
oracle fed the same e4m3 values and scales.  Integer work (gathered K/V and
the work list) must match bit for bit.

Those absolute bars alone are loose on long rows: with N(0,1) inputs the
softmax of a row with n visible keys is nearly flat and its output is an
average of order 1/sqrt(n) (about 0.03 on the Llama-3-8B-shaped prefill), so
a lost or doubled K/V tile could stay under 2e-2.  Two things make the
comparison bind there:

* every case also runs "sharp", with q scaled by 4 before its bf16 rounding,
  which peaks the softmax and lifts outputs to order 1.  Its q is no longer
  N(0,1), and an output near a single V value reaches |o| of 4 to 5, where
  half a bf16 ulp alone is 2^-6 = 0.0156; so the sharp runs take their
  elementwise bar from the same arithmetic instead of the fixed 2e-2:
  |e| <= 2^-8 (|o_ref| + bmm2 max|V|), twice the sum of the output rounding
  (2^-9 |o|) and the P rounding (2^-9 sum_j p_j |V_j| / l <= 2^-9 bmm2 max|V|);
* each row must also meet a relative bar, ||o - o_ref|| / ||o_ref|| <= 1e-2
  over its head_dim elements.  The arithmetic fixes the expected value: the
  bf16 output and the bf16 (f16 on the e4m3 path) P each round with a
  relative error of at most 2^-9, independent from element to element, so a
  row's relative L2 error is about 2^-9 (2e-3); 1e-2 leaves a factor of five,
  while a dropped tile of a row with t tiles gives about 1/t.

Every assertion message reports max-abs, mean-abs, the largest elementwise
relative error |e| / max(|o_ref|, 1e-3) and the largest row-relative error.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workload

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_MAX_FP8 = 2e-2, 2e-3, 3e-2
TOL_ROW_REL = 1e-2
Q_SCALES = [1.0, 4.0]
DEV = "cuda:0"


def _to_dev(inp):
    d = {}
    for name in ("q", "k_pool", "v_pool", "block_tables", "seq_lens", "cum_q", "cum_kv"):
        d[name] = getattr(inp, name).to(DEV)
    d["sinks"] = None if inp.sinks is None else inp.sinks.to(DEV)
    return d


def _run(b2pa, inp, path="auto", out=None, dev=None):
    b2pa.set_kernel_path(path)
    try:
        d = dev or _to_dev(inp)
        if out is None:
            out = torch.full_like(d["q"], float("nan"))
        b2pa.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_q_len,
                               inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"], d["cum_kv"],
                               inp.window_left, out, inp.layout, d["sinks"])
        bits = b2pa.device_status()
    finally:
        b2pa.set_kernel_path("auto")
    return out, bits


def _errors(g, ref):
    """max-abs, mean-abs, max elementwise relative, max row-relative L2 error of g vs ref ([rows, D] float64).

    The row-relative error divides by max(||o_ref||, 1e-3): a row whose exact
    output is smaller than that (no visible key, or a sink term e^700 times the
    rest of the denominator, which fp32 rounds to an output of 0) is held to an
    absolute 1e-5 instead."""
    err = (g - ref).abs()
    rel = (err / ref.abs().clamp_min(1e-3)).max().item()
    row_rel = (err.norm(dim=1) / ref.norm(dim=1).clamp_min(1e-3)).max().item()
    return err.max().item(), err.mean().item(), rel, row_rel


def _compare(got, inp, rows=None, fp8=None):
    """got: [T, H, D] device tensor.  rows: None = all, else int64 token*H+h."""
    fp8 = inp.meta.get("kv_dtype") == "fp8_e4m3" if fp8 is None else fp8
    ref, st, _ = oracle.attention(inp, rows=rows)
    assert (st == 0).all()
    T, H, D = got.shape
    g = got.float().cpu().reshape(T * H, D).double()
    if rows is not None:
        g = g[torch.as_tensor(rows)]
    assert torch.isfinite(g).all(), "non-finite output"
    ref = torch.from_numpy(ref)
    mx, mean, rel, row_rel = _errors(g, ref)
    msg = (f"{inp.name}: max_abs={mx:.3e} mean_abs={mean:.3e} max_rel={rel:.3e} max_row_rel={row_rel:.3e} "
           f"rows={g.shape[0]}")
    print(msg)
    if inp.meta.get("q_scale", 1.0) != 1.0:
        vmax = inp.v_pool.float().abs().nan_to_num(0.0).max().item() * abs(inp.bmm2_scale)
        bar = 2.0 ** -8 * (ref.abs() + vmax)
        worst = ((g - ref).abs() / bar).max().item()
        assert worst <= 1.0, f"{msg} elementwise error / derived bar = {worst:.3f}"
        assert mean <= TOL_MEAN, msg
    elif fp8:
        assert mx <= TOL_MAX_FP8, msg
    else:
        assert mx <= TOL_MAX and mean <= TOL_MEAN, msg
    assert row_rel <= TOL_ROW_REL, msg
    return mx, mean


# ----------------------------------------------------------------- tensor-core path, small cases

TC_CASES = [
    # (q_lens, kv_lens, H, Hkv, D, P, layout, window, sinks, kv_dtype)
    ([70, 130, 5], [300, 130, 5], 8, 2, 128, 32, "HND", -1, True, "bf16"),
    ([64, 1, 200], [64, 513, 700], 32, 8, 128, 16, "NHD", -1, False, "bf16"),
    ([257, 33], [257, 33], 4, 4, 128, 64, "HND", -1, False, "bf16"),          # MHA, G = 1
    ([150, 90], [900, 90], 64, 8, 128, 128, "NHD", -1, True, "bf16"),          # G = 8
    ([300], [1200], 16, 1, 128, 256, "HND", -1, False, "bf16"),               # G = 16, P > tile
    ([200, 77], [200, 300], 16, 2, 64, 16, "HND", 127, True, "bf16"),          # D = 64, window
    ([129, 3, 260], [129, 500, 260], 8, 2, 64, 8, "NHD", -1, False, "bf16"),
    ([100, 140], [1000, 140], 8, 2, 128, 32, "HND", 0, True, "bf16"),          # window 0
    ([333, 50], [700, 50], 8, 2, 128, 32, "HND", 200, False, "bf16"),
    ([96, 1, 40], [4000, 3000, 40], 32, 8, 128, 32, "HND", -1, False, "fp8_e4m3"),
    ([300, 7], [300, 600], 8, 2, 128, 64, "NHD", 77, True, "fp8_e4m3"),
    ([0, 40, 0, 10], [10, 100, 0, 10], 8, 2, 128, 32, "HND", -1, False, "bf16"),  # empty requests
    ([24, 24], [24, 24], 12, 4, 128, 32, "HND", -1, True, "bf16"),              # G = 3: rows 126 of 128
    # short windows at D = 64: the one-window-tile kernel
    ([1, 160, 64], [90, 160, 2000], 32, 2, 64, 8, "NHD", 100, False, "bf16"),  # G = 16, P = 8
    ([300, 45], [300, 1000], 16, 2, 64, 32, "HND", 0, True, "bf16"),           # window 0, P = 32
    ([130, 64], [500, 64], 8, 2, 64, 16, "HND", 100, True, "bf16"),            # G = 4
]


@pytest.mark.parametrize("q_scale", Q_SCALES)
@pytest.mark.parametrize("case", range(len(TC_CASES)))
def test_tcgen05_parity_small(cuda_lib, case, q_scale):
    ql, kl, H, Hkv, D, P, lay, W, sinks, kvd = TC_CASES[case]
    inp = workload.build(ql, kl, H, Hkv, D, P, lay, kv_dtype=kvd, window_left=W, with_sinks=sinks, seed=100 + case,
                         table_pad="garbage", q_scale=q_scale)
    assert cuda_lib.query_path(inp.q.to(DEV), (inp.k_pool.to(DEV), inp.v_pool.to(DEV)), kv_layout=lay) == "tcgen05"
    out, bits = _run(cuda_lib, inp, "tcgen05")
    assert bits == 0
    _compare(out, inp)


# the tensor-core path's limits: the largest kv-head group (one token per 128-row
# query tile) and a wide group at D = 64
LIMIT_CASES = [
    ([40, 3], [300, 3], 128, 1, 128, 32, "HND", -1, True, "bf16"),   # G = 128
    ([50, 20], [90, 200], 64, 2, 64, 16, "NHD", 60, False, "bf16"),  # G = 32, window
]


@pytest.mark.parametrize("case", range(len(LIMIT_CASES)))
def test_tcgen05_group_size_limits(cuda_lib, case):
    ql, kl, H, Hkv, D, P, lay, W, sinks, kvd = LIMIT_CASES[case]
    inp = workload.build(ql, kl, H, Hkv, D, P, lay, kv_dtype=kvd, window_left=W, with_sinks=sinks, seed=700 + case,
                         table_pad="garbage")
    out, bits = _run(cuda_lib, inp, "tcgen05")
    assert bits == 0
    _compare(out, inp)


def test_scheduler_batch_limit(cuda_lib):
    """4096 requests (the most the scheduler takes) on the tensor-core path, and
    one more: the tensor-core path then refuses it and the automatic choice
    computes it on the generic path."""
    g = torch.Generator().manual_seed(77)
    B = 4096
    ql = torch.randint(0, 3, (B,), generator=g).tolist()
    kl = [q + x for q, x in zip(ql, torch.randint(0, 40, (B,), generator=g).tolist())]
    inp = workload.build(ql, kl, 8, 2, 128, 16, "HND", seed=78)
    out, bits = _run(cuda_lib, inp, "tcgen05")
    assert bits == 0
    _compare(out, inp)
    inp2 = workload.build(ql + [2], kl + [5], 8, 2, 128, 16, "HND", seed=79)
    with pytest.raises(cuda_lib.B2paError, match="batch"):
        _run(cuda_lib, inp2, "tcgen05")
    out2, bits2 = _run(cuda_lib, inp2, "auto")
    assert bits2 == 0
    _compare(out2, inp2)


@pytest.mark.parametrize("q_scale", Q_SCALES)
@pytest.mark.parametrize("case", range(len(TC_CASES)))
def test_generic_parity_small(cuda_lib, case, q_scale):
    ql, kl, H, Hkv, D, P, lay, W, sinks, kvd = TC_CASES[case]
    inp = workload.build(ql, kl, H, Hkv, D, P, lay, kv_dtype=kvd, window_left=W, with_sinks=sinks, seed=100 + case,
                         q_scale=q_scale)
    out, bits = _run(cuda_lib, inp, "generic")
    assert bits == 0
    _compare(out, inp)


GENERIC_ONLY = [
    ([5, 3], [9, 3], 2, 1, 16, 4, "HND", -1, False, "bf16"),
    ([17, 9], [40, 9], 6, 3, 40, 5, "NHD", 6, True, "bf16"),
    ([33], [33], 4, 2, 256, 7, "HND", -1, True, "fp8_e4m3"),
    ([12, 1], [12, 30], 3, 1, 96, 3, "NHD", -1, False, "bf16"),
]


@pytest.mark.parametrize("case", range(len(GENERIC_ONLY)))
def test_generic_only_shapes(cuda_lib, case):
    ql, kl, H, Hkv, D, P, lay, W, sinks, kvd = GENERIC_ONLY[case]
    inp = workload.build(ql, kl, H, Hkv, D, P, lay, kv_dtype=kvd, window_left=W, with_sinks=sinks, seed=300 + case)
    assert cuda_lib.query_path(inp.q.to(DEV), (inp.k_pool.to(DEV), inp.v_pool.to(DEV)), kv_layout=lay) == "generic"
    out, bits = _run(cuda_lib, inp)
    assert bits == 0
    _compare(out, inp)


def test_tiny_config(cuda_lib):
    inp = workload.config(1)
    out, bits = _run(cuda_lib, inp)
    assert bits == 0
    _compare(out, inp)


# ----------------------------------------------------------------- the named workloads at full size

def _sample_rows(inp, n_random, seed):
    """Boundary rows of every request (first / last query, window edge) plus random rows."""
    H = inp.num_heads
    g = np.random.default_rng(seed)
    rows = set()
    for b in range(inp.batch):
        q0, q1 = int(inp.cum_q[b]), int(inp.cum_q[b + 1])
        if q1 == q0:
            continue
        toks = {q0, q1 - 1, min(q1 - 1, q0 + 1)}
        if inp.window_left >= 0:
            toks.add(min(q1 - 1, q0 + inp.window_left))
        for t in toks:
            for h in (0, H - 1, int(g.integers(H))):
                rows.add(t * H + h)
    T = inp.q.shape[0]
    rows.update(g.integers(0, T * H, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


# Every row of the bench workload and of the sliding-window layer is compared
# (the oracle does them in seconds on the host cores); the chunked-prefix, full
# D = 64 and ragged FP8 workloads on every request's boundary rows plus 4000
# random rows.
FULL_ROWS = {(2, None), (4, None)}


@pytest.mark.parametrize("q_scale", Q_SCALES)
@pytest.mark.parametrize("index,window", [(2, None), (3, None), (4, None), (4, -1), (5, None)])
def test_named_workloads(cuda_lib, index, window, q_scale):
    inp = workload.config(index, window_left=window, q_scale=q_scale)
    out, bits = _run(cuda_lib, inp)
    assert bits == 0
    rows = None if (index, window) in FULL_ROWS else _sample_rows(inp, 4000, seed=index)
    _compare(out, inp, rows=rows)
    # properties that hold at any size: finite everywhere, and every row of a
    # valid request was written (the NaN fill is gone)
    assert torch.isfinite(out).all()


# ----------------------------------------------------------------- FP8 KV and the scales

@pytest.mark.parametrize("kvd", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("q_scale", [1e5, 1e-6])
@pytest.mark.parametrize("path", ["tcgen05", "generic"])
def test_extreme_query_magnitudes(cuda_lib, kvd, q_scale, path):
    """Queries far outside N(0,1) lose nothing: on the e4m3 path each Q row is
    scaled by a power of two into f16's range before its conversion (and the
    scale taken out of its scores), so |q| ~ 1e5 (a one-hot softmax) and
    |q| ~ 1e-6 (a flat one) neither overflow nor fall into f16's subnormals."""
    inp = workload.build([70, 130, 5], [300, 130, 5], 8, 2, 128, 32, "HND", kv_dtype=kvd, with_sinks=True,
                         seed=61, q_scale=q_scale)
    out, bits = _run(cuda_lib, inp, path)
    assert bits == 0
    _compare(out, inp)


def _run_tensor_scales(b2pa, inp, path, s1, s2):
    b2pa.set_kernel_path(path)
    try:
        d = _to_dev(inp)
        out = torch.full_like(d["q"], float("nan"))
        b2pa.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_q_len,
                               inp.max_kv_len, torch.tensor([s1], dtype=torch.float32, device=DEV),
                               torch.tensor([s2], dtype=torch.float32, device=DEV), d["cum_q"], d["cum_kv"],
                               inp.window_left, out, inp.layout, d["sinks"])
        bits = b2pa.device_status()
    finally:
        b2pa.set_kernel_path("auto")
    return out, bits


@pytest.mark.parametrize("kvd", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("path", ["tcgen05", "generic"])
def test_tensor_scales_equal_float_scales(cuda_lib, kvd, path):
    """bmm1_scale / bmm2_scale as device fp32 tensors (FlashInfer API reference:
    float | Tensor) give the same bits as the same values passed as floats, and
    match the oracle."""
    inp = workload.build([70, 130, 5], [300, 130, 5], 8, 2, 128, 32, "HND", kv_dtype=kvd, with_sinks=True,
                         seed=62, window_left=200)
    want, bits = _run(cuda_lib, inp, path)
    assert bits == 0
    got, bits = _run_tensor_scales(cuda_lib, inp, path, inp.bmm1_scale, inp.bmm2_scale)
    assert bits == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    _compare(got, inp)


@pytest.mark.parametrize("bad", [(-1.0, 1.0), (0.0, 1.0), (float("nan"), 1.0), (0.1, float("inf"))])
@pytest.mark.parametrize("path", ["tcgen05", "generic"])
def test_bad_tensor_scale_flagged(cuda_lib, bad, path):
    """A device scale the host cannot check: nothing is written and the error
    word says why."""
    inp = workload.build([40, 7], [90, 7], 8, 2, 128, 32, "HND", seed=63)
    out, bits = _run_tensor_scales(cuda_lib, inp, path, *bad)
    assert bits & cuda_lib.DEV_BAD_SCALE
    assert torch.isnan(out.float()).all()


# ----------------------------------------------------------------- bit-exact integer work

@pytest.mark.parametrize("layout,kvd,P,D", [("HND", "bf16", 32, 128), ("NHD", "bf16", 16, 64),
                                            ("HND", "fp8_e4m3", 32, 128), ("NHD", "bf16", 256, 128),
                                            ("HND", "bf16", 8, 64)])
def test_debug_gather_bit_exact(cuda_lib, layout, kvd, P, D):
    inp = workload.build([10, 1, 300], [130, 77, 600], 8, 4, D, P, layout, kv_dtype=kvd, seed=7, table_pad="garbage")
    d = _to_dev(inp)
    total = int(inp.seq_lens.sum())
    k_out, v_out = cuda_lib.debug_gather((d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], d["cum_kv"],
                                         total, layout)
    assert cuda_lib.device_status() == 0
    k_ref, ok1 = oracle.gather(inp, "k")
    v_ref, ok2 = oracle.gather(inp, "v")
    assert ok1 and ok2
    assert torch.equal(k_out.cpu().view(torch.uint8), k_ref.view(torch.uint8))
    assert torch.equal(v_out.cpu().view(torch.uint8), v_ref.view(torch.uint8))


def test_debug_gather_strided_views(cuda_lib):
    # one [N, 2, P, Hkv, D] cache viewed as HND pools with NHD strides
    # (TokenSpeed _get_kv_cache_permuted), Hkv = 1 (canonicalize_stride's case)
    inp = workload.build([5, 40], [200, 40], 4, 1, 128, 32, "NHD", seed=8, combined_kv=True)
    hnd = workload.build([5, 40], [200, 40], 4, 1, 128, 32, "NHD", seed=8, combined_kv=True)
    hnd.layout = "HND"
    hnd.k_pool = inp.k_pool.permute(0, 2, 1, 3)
    hnd.v_pool = inp.v_pool.permute(0, 2, 1, 3)
    d = _to_dev(hnd)
    total = int(inp.seq_lens.sum())
    k_out, v_out = cuda_lib.debug_gather((d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], d["cum_kv"],
                                         total, "HND")
    k_ref, _ = oracle.gather(inp, "k")
    v_ref, _ = oracle.gather(inp, "v")
    assert torch.equal(k_out.cpu().view(torch.uint8), k_ref.view(torch.uint8))
    assert torch.equal(v_out.cpu().view(torch.uint8), v_ref.view(torch.uint8))
    out, bits = _run(cuda_lib, hnd, "tcgen05")
    assert bits == 0
    _compare(out, inp)


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_worklist_bit_exact(cuda_lib, index):
    inp = workload.config(index)
    d = _to_dev(inp)
    items, geo = cuda_lib.debug_worklist(d["q"], d["k_pool"], d["block_tables"], d["seq_lens"], d["cum_q"],
                                         inp.max_q_len, inp.max_kv_len, inp.window_left, inp.layout)
    ref = oracle.worklist(inp, geo["rows_per_tile"], geo["n_qtiles"], geo["kv_tile"], geo["cost_cap"])
    assert items.shape == ref.shape
    assert np.array_equal(items, ref)


@pytest.mark.parametrize("window", [-1, 0, 5, 300])
def test_worklist_bit_exact_ragged(cuda_lib, window):
    ql = [1, 0, 700, 64, 65, 3000, 31]
    kl = [1, 5, 900, 64, 1000, 3000, 4000]
    inp = workload.build(ql, kl, 16, 2, 128, 32, "HND", window_left=window, seed=9)
    d = _to_dev(inp)
    items, geo = cuda_lib.debug_worklist(d["q"], d["k_pool"], d["block_tables"], d["seq_lens"], d["cum_q"],
                                         inp.max_q_len, inp.max_kv_len, window, "HND")
    ref = oracle.worklist(inp, geo["rows_per_tile"], geo["n_qtiles"], geo["kv_tile"], geo["cost_cap"])
    assert np.array_equal(items, ref)


# ----------------------------------------------------------------- robustness

@pytest.mark.parametrize("path", ["tcgen05", "generic"])
def test_poisoned_pool_tails_and_padding(cuda_lib, path):
    inp = workload.build([70, 9, 130], [301, 9, 200], 8, 2, 128, 32, "HND", with_sinks=True, seed=11,
                         table_pad="garbage", pool_factor=2.0)
    # NaN into every slot no request reads at a position below its kv_len
    used = set()
    for b in range(inp.batch):
        for t in range(int(inp.seq_lens[b])):
            used.add((int(inp.block_tables[b, t // 32]), t % 32))
    for pg in range(inp.k_pool.shape[0]):
        for sl in range(32):
            if (pg, sl) not in used:
                inp.k_pool[pg, :, sl] = float("nan")
                inp.v_pool[pg, :, sl] = float("nan")
    out, bits = _run(cuda_lib, inp, path)
    assert bits == 0
    _compare(out, inp)


def test_poisoned_fp8_tails(cuda_lib):
    inp = workload.build([40, 100], [77, 300], 8, 2, 128, 32, "HND", kv_dtype="fp8_e4m3", seed=12)
    nan8 = torch.tensor([0x7F], dtype=torch.uint8).view(torch.float8_e4m3fn)
    used = set()
    for b in range(inp.batch):
        for t in range(int(inp.seq_lens[b])):
            used.add((int(inp.block_tables[b, t // 32]), t % 32))
    for pg in range(inp.k_pool.shape[0]):
        for sl in range(32):
            if (pg, sl) not in used:
                inp.k_pool[pg, :, sl] = nan8
                inp.v_pool[pg, :, sl] = nan8
    out, bits = _run(cuda_lib, inp, "tcgen05")
    assert bits == 0
    _compare(out, inp)


@pytest.mark.parametrize("path", ["tcgen05", "generic"])
def test_output_canaries_and_bad_request(cuda_lib, path):
    inp = workload.build([30, 20, 25], [60, 20, 25], 8, 2, 128, 32, "HND", seed=13)
    d = _to_dev(inp)
    # request 1 claims 20 queries but only 10 keys: rejected, its rows untouched
    d["seq_lens"][1] = 10
    T, H, D = inp.q.shape
    big = torch.full((T + 8, H, D), 7.0, dtype=torch.bfloat16, device=DEV)
    out = big[4:4 + T]
    cuda_lib.set_kernel_path(path)
    try:
        cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                   inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"], None,
                                   -1, out, "HND")
        bits = cuda_lib.device_status()
    finally:
        cuda_lib.set_kernel_path("auto")
    assert bits & cuda_lib.DEV_BAD_REQUEST
    assert (big[:4] == 7).all() and (big[4 + T:] == 7).all()
    assert (out[30:50] == 7).all()
    ok = inp.cum_q.tolist()
    rows = np.array([t * H + h for t in list(range(0, 30)) + list(range(50, 75)) for h in range(H)])
    _compare(out, inp, rows=rows)


def test_bad_page_id_flagged(cuda_lib):
    inp = workload.build([16], [100], 8, 2, 128, 32, "HND", seed=14)
    d = _to_dev(inp)
    d["block_tables"][0, 1] = inp.k_pool.shape[0] + 10
    cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], 16, 100,
                               inp.bmm1_scale, 1.0, d["cum_q"], None, -1, None, "HND")
    assert cuda_lib.device_status() & cuda_lib.DEV_BAD_PAGE


def test_bitwise_deterministic(cuda_lib):
    inp = workload.config(2)
    d = _to_dev(inp)
    a, _ = _run(cuda_lib, inp, dev=d)
    b, _ = _run(cuda_lib, inp, dev=d)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_cuda_graph_replay(cuda_lib):
    inp = workload.build([100, 260], [400, 260], 8, 2, 128, 32, "HND", seed=15, with_sinks=True)
    d = _to_dev(inp)
    s = torch.cuda.Stream()
    out = torch.zeros_like(d["q"])
    with torch.cuda.stream(s):
        args = (d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_q_len, inp.max_kv_len,
                inp.bmm1_scale, inp.bmm2_scale, d["cum_q"], d["cum_kv"], -1, out, "HND", d["sinks"])
        cuda_lib.context_attention(*args, stream=s)  # sizes this stream's workspace
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            cuda_lib.context_attention(*args, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    _compare(out, inp)


def test_invalid_arguments_rejected_on_host(cuda_lib):
    inp = workload.build([4], [8], 4, 2, 128, 32, "HND", seed=16)
    d = _to_dev(inp)
    with pytest.raises(cuda_lib.B2paError):
        cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], 4, 8,
                                   -1.0, 1.0, d["cum_q"], None, -1, None, "HND")
    with pytest.raises(cuda_lib.B2paError):
        q3 = d["q"][:, :3]
        cuda_lib.context_attention(q3, (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], 4, 8, 0.1,
                                   1.0, d["cum_q"], None, -1, None, "HND")


def test_two_streams_concurrently(cuda_lib):
    """Calls on two streams at once: each stream has its own workspace, so the
    work-distribution words and work lists of the two launches are separate;
    both results must match the oracle (and the single-stream result bit for
    bit), round after round."""
    a = workload.build([300, 1, 700, 64], [900, 40, 700, 2000], 32, 8, 128, 32, "HND", seed=71, with_sinks=True)
    b = workload.build([129, 1000], [129, 3000], 16, 2, 64, 16, "NHD", seed=72, window_left=200)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for inp in (a, b):
        d = _to_dev(inp)
        outs.append((inp, d, torch.full_like(d["q"], float("nan"))))
    torch.cuda.synchronize()
    for _ in range(20):
        for (inp, d, out), st in zip(outs, (s1, s2)):
            cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                       inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"],
                                       d["cum_kv"], inp.window_left, out, inp.layout, d["sinks"], stream=st)
    assert cuda_lib.device_status(s1) == 0 and cuda_lib.device_status(s2) == 0
    torch.cuda.synchronize()
    for inp, d, out in outs:
        _compare(out, inp)
        single, bits = _run(cuda_lib, inp)
        assert bits == 0
        assert torch.equal(single.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("which", ["ragged_lone_tiles", "cfg2", "cfg5"])
def test_stress_back_to_back_calls(cuda_lib, which):
    """Hundreds of calls in a row (the pattern a timed benchmark produces): no
    device error bit, and the last output still matches the oracle."""
    if which == "cfg2":
        inp = workload.config(2)
    elif which == "cfg5":
        inp = workload.config(5)
    else:
        ql = [1, 33, 64, 65, 97, 7, 128, 31, 200, 3]
        kl = [900, 33, 1000, 65, 2000, 7, 300, 1500, 200, 3000]
        inp = workload.build(ql, kl, 32, 8, 128, 32, "HND", seed=21, with_sinks=True)
    d = _to_dev(inp)
    out = torch.zeros_like(d["q"])
    for _ in range(300 if which != "cfg5" else 60):
        cuda_lib.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                   inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"],
                                   d["cum_kv"], inp.window_left, out, inp.layout, d["sinks"])
    assert cuda_lib.device_status() == 0
    rows = _sample_rows(inp, 300, seed=5)
    _compare(out, inp, rows=rows)


# ----------------------------------------------------------------- failure detection

@pytest.mark.parametrize("variant", ["bf16_d128", "bf16_d64_window", "bf16_d64_window_tile", "fp8", "decode_split"])
def test_wait_timeout_returns_error_and_recovers(cuda_lib, variant):
    """A pipeline wait that runs out: with the stall injected, each CTA's MMA
    warp waits on a barrier that nothing arrives on, the 2 ms wait limit runs
    out, and the CTA drains its copies and MMAs and exits; the call reports
    B2PA_DEV_TIMEOUT without a GPU fault.  The same context then computes the
    batch correctly with the stall off and the default limit."""
    if variant == "decode_split":
        inp = workload.build([1] * 4, [20000, 9000, 31000, 700], 32, 8, 128, 32, "HND", seed=43)
    elif variant == "bf16_d64_window_tile":
        inp = workload.build([200, 130], [900, 130], 16, 2, 64, 16, "HND", window_left=127, seed=42)
    else:
        D, W, kvd = {"bf16_d128": (128, -1, "bf16"), "bf16_d64_window": (64, 127, "bf16"),
                     "fp8": (128, -1, "fp8_e4m3")}[variant]
        inp = workload.build([200, 130], [900, 130], 8, 2, D, 32, "HND", kv_dtype=kvd, window_left=W, seed=41)

    def call():
        if variant == "decode_split":
            d = _to_dev(inp)
            out = torch.full_like(d["q"], float("nan"))
            cuda_lib.batch_decode(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                  inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, -1, out, "HND", None,
                                  q_len_per_req=1)
            return out, cuda_lib.device_status()
        return _run(cuda_lib, inp, "tcgen05")

    cuda_lib.set_wait_limit_ns(2_000_000)
    cuda_lib.debug_inject_stall(True)
    try:
        _, bits = call()
    finally:
        cuda_lib.debug_inject_stall(False)
        cuda_lib.set_wait_limit_ns(0)
    assert bits & cuda_lib.DEV_TIMEOUT
    out, bits = call()
    assert bits == 0
    _compare(out, inp)
