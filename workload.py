"""Seeded synthetic inputs for batched paged-KV context attention.

This module only draws inputs: request lengths, page placement, the page
table, q/K/V values, scales and sinks.  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it without sharing any of the method.

Shapes follow the API contract of
flashinfer.prefill.trtllm_batch_context_with_kv_cache (FlashInfer API
reference, parameter list): query [num_tokens, num_heads, head_dim]; a K and a
V page pool [num_pages, num_kv_heads, page_size, head_dim] (HND) or
[num_pages, page_size, num_kv_heads, head_dim] (NHD); int32 block_tables
[batch, max_pages]; int32 seq_lens [batch] holding kv lengths; int32
cum_seq_lens_q / cum_seq_lens_kv [batch + 1].

The length conventions come from the TokenSpeed trtllm backend
(runtime/layers/attention/backends/trtllm.py, _init_extend_metadata): the kv
length of a request is its cached prefix plus its new tokens, the query
length is the number of new tokens, and cum_seq_lens_kv is the zero-padded
cumulative sum of seq_lens.  Unused table columns hold the dummy page id 0,
as that backend's gather_page_table_with_padding(dummy_slot=0) and the
TensorRT-LLM teardown (6), section "prepare_flash_mla", describe.

All draws use a torch.Generator on the CPU, so the same seed gives the same
bytes on any machine.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

FP8_E4M3_MAX = 448.0


@dataclass
class Inputs:
    """One batch of host (CPU) tensors for a context-attention call."""

    q: torch.Tensor                 # [T, H, D] bf16
    k_pool: torch.Tensor            # HND [N, Hkv, P, D] / NHD [N, P, Hkv, D]; bf16 or float8_e4m3fn
    v_pool: torch.Tensor            # same shape and dtype as k_pool
    block_tables: torch.Tensor      # [B, max_pages] int32
    seq_lens: torch.Tensor          # [B] int32 (kv lengths)
    cum_q: torch.Tensor             # [B + 1] int32
    cum_kv: torch.Tensor            # [B + 1] int32
    max_q_len: int
    max_kv_len: int
    bmm1_scale: float
    bmm2_scale: float
    window_left: int = -1
    sinks: Optional[torch.Tensor] = None   # [H] float32 or None
    layout: str = "HND"
    name: str = "custom"
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_pool.shape[1] if self.layout == "HND" else self.k_pool.shape[2])

    @property
    def page_size(self) -> int:
        return int(self.k_pool.shape[2] if self.layout == "HND" else self.k_pool.shape[1])

    @property
    def q_lens(self) -> list[int]:
        c = self.cum_q.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    @property
    def kv_lens(self) -> list[int]:
        return self.seq_lens.tolist()


def _normal_bf16(shape, gen: torch.Generator, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def _pool_shape(layout: str, n_pages: int, hkv: int, page: int, d: int):
    if layout == "HND":
        return (n_pages, hkv, page, d)
    if layout == "NHD":
        return (n_pages, page, hkv, d)
    raise ValueError(f"layout must be HND or NHD, got {layout!r}")


def build(
    q_lens,
    kv_lens,
    num_heads: int,
    num_kv_heads: int,
    head_dim: int,
    page_size: int,
    layout: str = "HND",
    kv_dtype: str = "bf16",
    window_left: int = -1,
    with_sinks: bool = False,
    pool_factor: float = 2.0,
    extra_pages: int = 0,
    max_pages: Optional[int] = None,
    seed: int = 0,
    bmm1_scale: Optional[float] = None,
    bmm2_scale: float = 1.0,
    table_pad: str = "zero",
    q_scale: float = 1.0,
    name: str = "custom",
    sink_scale: float = 1.0,
    combined_kv: bool = False,
) -> Inputs:
    """Draw one batch with the given per-request query and kv lengths.

    q/K/V values are N(0,1) (q optionally times ``q_scale``) rounded to bf16.
    With ``kv_dtype="fp8_e4m3"`` K and V are drawn N(0,1) in fp32, each pool
    gets a per-tensor scale amax/448, and the scaled values are cast to e4m3
    (round to nearest even, torch's CPU cast).  The K scale is folded into
    bmm1_scale and the V scale into bmm2_scale, as the TokenSpeed backend's
    _compute_scales folds k_scale into bmm1_scale.

    Pages are placed at random: every page a request uses is a distinct page
    of a pool of ``ceil(pool_factor * pages_needed) + extra_pages`` pages,
    taken from a seeded permutation.  Page-table columns past a request's
    last used page hold 0 (``table_pad="zero"``) or garbage ids
    (``table_pad="garbage"``: -1 and values far past the pool).
    """
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    assert len(q_lens) == len(kv_lens)
    B = len(q_lens)
    assert num_heads % num_kv_heads == 0
    gen = torch.Generator().manual_seed(seed)

    T = sum(q_lens)
    H, Hkv, D, P = num_heads, num_kv_heads, head_dim, page_size
    pages_per_req = [(k + P - 1) // P for k in kv_lens]
    need = sum(pages_per_req)
    n_pages = max(1, int(math.ceil(pool_factor * need)) + extra_pages)
    if max_pages is None:
        max_pages = max(1, max(pages_per_req) if pages_per_req else 1)
    assert max_pages >= max(pages_per_req, default=0)

    perm = torch.randperm(n_pages, generator=gen)
    table = torch.zeros((B, max_pages), dtype=torch.int32)
    if table_pad == "garbage":
        junk = torch.randint(n_pages + 1000, n_pages + 100000, (B, max_pages), generator=gen, dtype=torch.int32)
        junk[:, ::2] = -1
        table.copy_(junk)
    elif table_pad != "zero":
        raise ValueError(table_pad)
    pos = 0
    for b in range(B):
        n = pages_per_req[b]
        table[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n

    q = _normal_bf16((T, H, D), gen, q_scale)
    shape = _pool_shape(layout, n_pages, Hkv, P, D)
    if combined_kv:
        # one [N, 2, ...] tensor; K and V are strided views of it
        if layout == "HND":
            full_shape = (n_pages, 2, Hkv, P, D)
        else:
            full_shape = (n_pages, 2, P, Hkv, D)
    if kv_dtype == "bf16":
        if combined_kv:
            kv = _normal_bf16(full_shape, gen)
            k_pool, v_pool = kv[:, 0], kv[:, 1]
        else:
            k_pool = _normal_bf16(shape, gen)
            v_pool = _normal_bf16(shape, gen)
        k_scale = v_scale = 1.0
    elif kv_dtype == "fp8_e4m3":
        if combined_kv:
            kf = torch.randn(full_shape, generator=gen, dtype=torch.float32)
            k32, v32 = kf[:, 0], kf[:, 1]
        else:
            k32 = torch.randn(shape, generator=gen, dtype=torch.float32)
            v32 = torch.randn(shape, generator=gen, dtype=torch.float32)
        k_scale = float(k32.abs().max()) / FP8_E4M3_MAX
        v_scale = float(v32.abs().max()) / FP8_E4M3_MAX
        if combined_kv:
            kv = torch.empty(full_shape, dtype=torch.float8_e4m3fn)
            kv[:, 0] = (k32 / k_scale).to(torch.float8_e4m3fn)
            kv[:, 1] = (v32 / v_scale).to(torch.float8_e4m3fn)
            k_pool, v_pool = kv[:, 0], kv[:, 1]
        else:
            k_pool = (k32 / k_scale).to(torch.float8_e4m3fn)
            v_pool = (v32 / v_scale).to(torch.float8_e4m3fn)
    else:
        raise ValueError(kv_dtype)

    if bmm1_scale is None:
        bmm1_scale = 1.0 / math.sqrt(D)
    bmm1 = float(bmm1_scale) * k_scale
    bmm2 = float(bmm2_scale) * v_scale

    sinks = None
    if with_sinks:
        sinks = torch.randn((H,), generator=gen, dtype=torch.float32) * sink_scale

    cum_q = [0]
    for x in q_lens:
        cum_q.append(cum_q[-1] + x)
    cum_kv = [0]
    for x in kv_lens:
        cum_kv.append(cum_kv[-1] + x)

    return Inputs(
        q=q,
        k_pool=k_pool,
        v_pool=v_pool,
        block_tables=table,
        seq_lens=torch.tensor(kv_lens, dtype=torch.int32),
        cum_q=torch.tensor(cum_q, dtype=torch.int32),
        cum_kv=torch.tensor(cum_kv, dtype=torch.int32),
        max_q_len=max(q_lens) if q_lens else 0,
        max_kv_len=max(kv_lens) if kv_lens else 0,
        bmm1_scale=bmm1,
        bmm2_scale=bmm2,
        window_left=window_left,
        sinks=sinks,
        layout=layout,
        name=name,
        seed=seed,
        meta={"k_scale": k_scale, "v_scale": v_scale, "kv_dtype": kv_dtype, "pool_pages": n_pages,
              "q_scale": q_scale},
    )


# ---------------------------------------------------------------------------
# The five named workloads.  Each draws its lengths from its own seeded
# generator (seed 1234 + index), then its values with build().
# ---------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny_b2_h2kv1_d16_p4",
    2: "llama3_8b_prefill_b8_l512-2048_h32kv8_d128_p32_hnd",
    3: "chunked_prefix_b16_kv1024-8192_q512_h64kv8_d128_p64_nhd",
    4: "swa127_sinks_b4_l4096_h64kv8_d64_p16_hnd",
    5: "ragged_fp8kv_b32_qlog1-4096_prefix0-28672_h32kv8_d128_p32_hnd",
}


def _uniform_int(gen, lo, hi, n):
    """n integers uniform on [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def config(index: int, window_left: Optional[int] = None, seed: Optional[int] = None, q_scale: float = 1.0) -> Inputs:
    """The named workloads 1..5.

    1: batch 2, q_lens [5,3], kv_lens [9,3], H 2 / Hkv 1, D 16, P 4, HND, pool
       of 8 pages, page table from a seeded permutation.
    2: batch 8, q = kv ~ U[512, 2048], H 32 / Hkv 8, D 128, P 32, HND, pool 2x.
    3: batch 16, kv ~ U[1024, 8192], q = 512, H 64 / Hkv 8, D 128, P 64, NHD.
    4: batch 4, q = kv = 4096, H 64 / Hkv 8, D 64, P 16, HND, window 127,
       fp32 sinks ~ N(0,1); ``window_left=-1`` gives its full-attention layer.
    5: batch 32, q log-uniform [1, 4096], prefix ~ U[0, 28672], H 32 / Hkv 8,
       D 128, P 32, HND, K/V e4m3 with per-tensor scales.

    ``q_scale`` multiplies q before its bf16 rounding (the "sharp" variant:
    q x 4 makes the softmax peaked, so that outputs of long rows are no longer
    averages near zero); every other draw is unchanged.
    """
    s = 1234 + index if seed is None else seed
    g = torch.Generator().manual_seed(s)
    name = CONFIG_NAMES[index] + ("" if q_scale == 1.0 else f"_qx{q_scale:g}")
    if index == 1:
        # 9 + 3 tokens need 3 + 1 pages of an 8-page pool.
        inp = build([5, 3], [9, 3], 2, 1, 16, 4, "HND", pool_factor=1.0, extra_pages=4,
                    max_pages=3, seed=s, name=name, q_scale=q_scale)
        return inp
    if index == 2:
        L = _uniform_int(g, 512, 2048, 8)
        return build(L, L, 32, 8, 128, 32, "HND", pool_factor=2.0, seed=s, name=name, q_scale=q_scale)
    if index == 3:
        K = _uniform_int(g, 1024, 8192, 16)
        return build([512] * 16, K, 64, 8, 128, 64, "NHD", pool_factor=2.0, seed=s, name=name, q_scale=q_scale)
    if index == 4:
        W = 127 if window_left is None else window_left
        nm = name if W == 127 else name.replace("swa127", f"swa{W}" if W >= 0 else "full")
        return build([4096] * 4, [4096] * 4, 64, 8, 64, 16, "HND", window_left=W, with_sinks=True,
                     pool_factor=2.0, seed=s, name=nm, q_scale=q_scale)
    if index == 5:
        u = torch.rand((32,), generator=g, dtype=torch.float64) * math.log(4096.0)
        ql = [min(4096, max(1, int(round(math.exp(x))))) for x in u.tolist()]
        pre = _uniform_int(g, 0, 28672, 32)
        kv = [a + b for a, b in zip(ql, pre)]
        return build(ql, kv, 32, 8, 128, 32, "HND", kv_dtype="fp8_e4m3", pool_factor=2.0,
                     seed=s, name=name, q_scale=q_scale)
    raise ValueError(index)


# ---------------------------------------------------------------------------
# Decode batches (the decode sibling): every request holds q_len_per_req query
# tokens, the last of its kv sequence (TokenSpeed trtllm backend,
# forward_decode; q_len_per_req > 1 is speculative verification).  Shaped like
# the ragged FP8 workload's long rows: 32 requests, kv lengths uniform in
# [q_len_per_req, 32768], H 32 / Hkv 8, D 128, P 32, HND, bf16.
# ---------------------------------------------------------------------------

def decode_config(q_len_per_req: int = 1, seed: Optional[int] = None, kv_dtype: str = "bf16") -> Inputs:
    s = 1300 + q_len_per_req if seed is None else seed
    g = torch.Generator().manual_seed(s)
    kv = _uniform_int(g, q_len_per_req, 32768, 32)
    name = f"decode_b32_q{q_len_per_req}_kv-32768_h32kv8_d128_p32_hnd" + ("" if kv_dtype == "bf16" else "_fp8kv")
    return build([q_len_per_req] * 32, kv, 32, 8, 128, 32, "HND", kv_dtype=kv_dtype, pool_factor=2.0, seed=s,
                 name=name)


def ragged_page_table(inp: Inputs):
    """The same batch's pages as FlashInfer's ragged page table: the flat page ids
    of every request (its first ceil(kv_len / P) block-table columns, in order),
    their per-request offsets [B + 1], and the tokens in each request's last
    page (P for a full page; 0 for a request without pages, where it is not
    read).  Returns int32 tensors (indices, indptr, last_page_len)."""
    P = inp.page_size
    ids, indptr, last = [], [0], []
    for b, L in enumerate(inp.kv_lens):
        n = (L + P - 1) // P
        ids.extend(inp.block_tables[b, :n].tolist())
        indptr.append(indptr[-1] + n)
        last.append(L - (n - 1) * P if n > 0 else 0)
    return (torch.tensor(ids, dtype=torch.int32), torch.tensor(indptr, dtype=torch.int32),
            torch.tensor(last, dtype=torch.int32))
