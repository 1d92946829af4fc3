"""Shared plumbing of the GPU parity tests: run the library and the oracle on
the same seeded inputs and compare them.  Inputs come from the package's
seeded generators; expected values come only from ``oracle``."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W

# Tolerances for attention outputs (bf16 cache, fp32 accumulation): elementwise
# absolute error, and per (b, h) row the max error relative to the row's max |ref|.
ABS_TOL = 2e-2
REL_TOL = 1e-2
LSE_ABS_TOL = 2e-2


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor (through its bit patterns)."""
    return O.bf16_bits_to_f64(W.bf16_to_bits(t))


def dims_of(w: W.Workload) -> mla.Dims:
    return mla.dims(w.heads, w.page_size, int8=w.int8, fp8=w.fp8)


def gpu_cache(inp: dict, w: W.Workload, rope_theta: float | None = None):
    """Device cache for the library: the drawn bf16 pool, or for INT8 / FP8
    workloads the pool built from the drawn source rows by the library's own
    append."""
    if not w.quantised:
        return inp["cache"].cuda(), None
    theta = w.rope_theta if rope_theta is None else rope_theta
    npg, P = inp["num_pages"], w.page_size
    cache = torch.zeros((npg, P, W.LATENT_DIM + W.ROPE_DIM), dtype=torch.int8 if w.int8 else torch.uint8,
                        device="cuda")
    sz = torch.zeros((npg, P, 2) if w.int8 else (npg, P), dtype=torch.float32, device="cuda")
    mla.cache_append(dims_of(w), cache, sz, inp["block_table"].cuda(), inp["src_seq_ids"].cuda(),
                     inp["src_positions"].cuda(), inp["src_c_kv"].cuda(), inp["src_k_pe"].cuda(), theta)
    return cache, sz


def oracle_cache(inp: dict, w: W.Workload, seqs, rope_theta: float | None = None):
    """The oracle's view of the cache, restricted to the pages of `seqs`:
    (cache numpy, scale_zero numpy or None, remapped block table)."""
    table = inp["block_table"].cpu().numpy()
    lens = inp["seq_lens"].cpu().numpy().astype(np.int64)
    P = w.page_size
    pages = sorted({int(p) for b in seqs for p in table[b, : (lens[b] + P - 1) // P]})
    remap = {p: i for i, p in enumerate(pages)}
    sub = np.full_like(table, -1)
    for b in seqs:
        n = (lens[b] + P - 1) // P
        sub[b, :n] = [remap[int(p)] for p in table[b, :n]]
    npg = max(len(pages), 1)
    if not w.quantised:
        idx = torch.tensor(pages, dtype=torch.int64, device=inp["cache"].device)
        cache = W.bf16_to_bits(inp["cache"].index_select(0, idx)) if pages else np.zeros((1, P, 576), np.uint16)
        return cache, None, sub
    theta = w.rope_theta if rope_theta is None else rope_theta
    cache = np.zeros((npg, P, 576), np.int8 if w.int8 else np.uint8)
    sz = np.zeros((npg, P, 2) if w.int8 else (npg, P), np.float32)
    starts = np.concatenate([[0], np.cumsum(lens)])
    for b in seqs:
        a, e = int(starts[b]), int(starts[b + 1])
        c_bits = W.bf16_to_bits(inp["src_c_kv"][a:e])
        k_bits = W.bf16_to_bits(inp["src_k_pe"][a:e])
        O.append_tokens(cache, sz, sub, [b] * (e - a), list(range(e - a)), c_bits, k_bits, theta, P,
                        int8=w.int8, fp8=w.fp8)
    return cache, sz, sub


def oracle_decode(inp: dict, w: W.Workload, pairs, absorbed=False, rope_theta=None, cache_override=None):
    seqs = sorted({b for b, _ in pairs})
    cache, sz, table = cache_override if cache_override is not None else oracle_cache(inp, w, seqs, rope_theta)
    lens = inp["seq_lens"].cpu().numpy()
    return O.decode(f64(inp["q_nope"]), f64(inp["q_pe"]), cache, sz, table, lens, f64(inp["W_UK"]),
                    f64(inp["W_UV"]), inp["scale"], w.page_size, w.int8, pairs=pairs, absorbed=absorbed, fp8=w.fp8)


def gpu_decode(inp: dict, w: W.Workload, cache, sz, num_splits=0, block_table=None):
    d = dims_of(w)
    bt = (inp["block_table"] if block_table is None else block_table).cuda()
    out, lse = mla.decode(d, inp["q_nope"].cuda(), inp["q_pe"].cuda(), cache, sz, bt, inp["seq_lens"].cuda(),
                          inp["W_UK"].cuda(), inp["W_UV"].cuda(), inp["scale"], num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def assert_parity(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref: np.ndarray, lse_ref: np.ndarray, pairs,
                  what=""):
    og = out_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.cpu().numpy().astype(np.float64)
    worst_abs, worst_rel = 0.0, 0.0
    for b, h in pairs:
        ref = out_ref[b, h]
        err = np.abs(og[b, h] - ref)
        m = float(np.abs(ref).max())
        worst_abs = max(worst_abs, float(err.max()))
        if m > 0:
            worst_rel = max(worst_rel, float(err.max()) / m)
        else:
            assert float(err.max()) == 0.0, (what, b, h)
        if math.isinf(lse_ref[b, h]):
            assert math.isinf(lg[b, h]) and lg[b, h] < 0, (what, b, h, lg[b, h])
        else:
            assert abs(lg[b, h] - lse_ref[b, h]) <= LSE_ABS_TOL, (what, b, h, lg[b, h], lse_ref[b, h])
    assert worst_abs <= ABS_TOL, (what, worst_abs)
    assert worst_rel <= REL_TOL, (what, worst_rel)
    return worst_abs, worst_rel
