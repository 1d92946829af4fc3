"""GPU parity of chunked prefill (mla_prefill) against the fp64 oracle,
through the C ABI: the chunk's rows written into the paged cache (compared
with the oracle's own append) and the causal attention of the chunk's tokens
over the history and the chunk (compared element by element: the absorbed
fp64 form on every (sequence, token, head), the un-absorbed form on a seeded
sample; the two are pinned to each other in test_oracle.py)."""
import numpy as np
import pytest
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import assert_parity, f64

pytestmark = pytest.mark.gpu


def _pf(heads=16, P=64, hist=(0, 300), chunk=64, fmt="bf16", theta=10000.0, seed=41):
    g = W.generator(seed)
    B = len(hist)
    seq_lens = torch.tensor([h + chunk for h in hist], dtype=torch.int32).clamp(min=0)
    table, npg = W.draw_page_table(seq_lens, P, True, g, spare_pages=2)
    x = dict(seq_lens=seq_lens, table=table, P=P, heads=heads, chunk=chunk, fmt=fmt, theta=theta,
             scale=1.0 / np.sqrt(192.0))
    if fmt == "int8":
        x["cache"], x["sz"] = W.draw_int8_cache(npg, P, g)
    elif fmt == "fp8":
        x["cache"], x["sz"] = W.draw_fp8_cache(npg, P, g)
    else:
        x["cache"], x["sz"] = W.draw_bf16((npg, P, 576), 1.0, g), None
    x["c_kv"] = W.draw_bf16((B, chunk, 512), 1.0, g)
    x["k_pe"] = W.draw_bf16((B, chunk, 64), 1.0, g)
    x["W_UK"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    x["W_UV"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    x["q_nope"] = W.draw_bf16((B, chunk, heads, 128), 1.0, g)
    x["q_pe"] = W.draw_bf16((B, chunk, heads, 64), 1.0, g)
    return x


def _dims(x):
    return mla.dims(x["heads"], x["P"], int8=x["fmt"] == "int8", fp8=x["fmt"] == "fp8")


def _gpu(x, num_splits=0):
    d = _dims(x)
    cache = x["cache"].cuda()
    sz = x["sz"].cuda() if x["sz"] is not None else None
    B, T = x["q_nope"].shape[0], x["chunk"]
    ws = torch.empty(mla.prefill_workspace_size(d, B, T, num_splits), dtype=torch.uint8, device="cuda")
    out, lse = mla.prefill(d, cache, sz, x["table"].cuda(), x["seq_lens"].cuda(), x["c_kv"].cuda(),
                           x["k_pe"].cuda(), x["q_nope"].cuda(), x["q_pe"].cuda(), x["W_UK"].cuda(),
                           x["W_UV"].cuda(), x["scale"], rope_theta=x["theta"], num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, cache, sz, mla.read_device_status(ws)


def _oracle_cache(x):
    if x["fmt"] == "bf16":
        return W.bf16_to_bits(x["cache"]), None
    return x["cache"].numpy().copy(), x["sz"].numpy().copy()


def _oracle(x, triples=None, absorbed=False):
    cache, sz = _oracle_cache(x)
    o, l = O.prefill_chunk(cache, sz, x["table"].numpy(), x["seq_lens"].numpy(), W.bf16_to_bits(x["c_kv"]),
                           W.bf16_to_bits(x["k_pe"]), x["theta"], f64(x["q_nope"]), f64(x["q_pe"]), f64(x["W_UK"]),
                           f64(x["W_UV"]), x["scale"], x["P"], x["fmt"] == "int8", triples=triples,
                           absorbed=absorbed, fp8=x["fmt"] == "fp8")
    return o, l, cache, sz


def _check(x, num_splits=0, sample=24):
    out, lse, cache, sz, st = _gpu(x, num_splits)
    B, T, H = out.shape[0], out.shape[1], out.shape[2]
    flat = lambda a: a.reshape(B, T * H, *a.shape[3:])  # noqa: E731  rows v = t * H + h
    ref_o, ref_l, ref_cache, ref_sz = _oracle(x, absorbed=True)
    pairs = [(b, v) for b in range(B) for v in range(T * H)]
    assert_parity(flat(out), flat(lse), flat(ref_o), flat(ref_l), pairs, "prefill (absorbed oracle)")
    rng = np.random.default_rng(7)
    triples = [(int(b), int(t), int(h)) for b, t, h in
               zip(rng.integers(0, B, sample), rng.integers(0, T, sample), rng.integers(0, H, sample))]
    un_o, un_l, _, _ = _oracle(x, triples=triples)
    assert_parity(flat(out), flat(lse), flat(un_o), flat(un_l), [(b, t * H + h) for b, t, h in triples],
                  "prefill (un-absorbed oracle)")
    return out, lse, cache, sz, st, ref_cache, ref_sz


@pytest.mark.parametrize("heads,P,hist,chunk", [(16, 64, (0, 300), 64), (128, 16, (130,), 20),
                                                (16, 128, (1000, 5), 200)])
def test_prefill_bf16(cuda_lib, heads, P, hist, chunk):
    out, lse, cache, _, st, ref_cache, _ = _check(_pf(heads=heads, P=P, hist=hist, chunk=chunk))
    assert st == mla.MLA_OK
    got = W.bf16_to_bits(cache)
    np.testing.assert_array_equal(got[..., :512], ref_cache[..., :512])  # latent rows copied exactly
    r, g = O.bf16_bits_to_f64(ref_cache[..., 512:]), O.bf16_bits_to_f64(got[..., 512:])
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), 1e-30))[1] - 8)
    assert np.all(np.abs(g - r) <= ulp)                                  # RoPE key within one bf16 ulp


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_prefill_quantised_cache_rows_bit_exact(cuda_lib, fmt):
    out, lse, cache, sz, st, ref_cache, ref_sz = _check(_pf(hist=(250, 3), chunk=48, fmt=fmt, theta=0.0, seed=43))
    assert st == mla.MLA_OK
    np.testing.assert_array_equal(cache.cpu().numpy(), ref_cache)
    np.testing.assert_array_equal(sz.cpu().numpy(), ref_sz)


def test_prefill_explicit_splits(cuda_lib):
    _check(_pf(hist=(700, 0, 129), chunk=32, seed=44), num_splits=7)


def test_prefill_sequence_shorter_than_chunk(cuda_lib):
    """A sequence whose length is below the chunk has its first tokens at
    negative positions: they are not written (bounds status) and attend to
    nothing (out = 0, lse = -inf); the rest is ordinary."""
    x = _pf(hist=(-6, 40), chunk=16, seed=45)
    out, lse, _, _, st, _, _ = _check(x)
    assert st == mla.MLA_ERR_DEVICE_BOUNDS
    assert torch.all(out[0, :6] == 0) and torch.all(torch.isneginf(lse[0, :6]))
    assert torch.all(torch.isfinite(lse[0, 6:])) and torch.all(torch.isfinite(lse[1]))


def test_prefill_then_decode_reads_what_prefill_wrote(cuda_lib):
    """A decode step after the prefill, on the cache the prefill left, matches
    the oracle's decode over the oracle's prefilled cache."""
    x = _pf(hist=(90, 400), chunk=40, seed=46)
    _, _, cache, _, st = _gpu(x)
    assert st == mla.MLA_OK
    _, _, ref_cache, _ = _oracle(x, triples=[])
    g = W.generator(47)
    B, H = 2, x["heads"]
    qn, qp = W.draw_bf16((B, H, 128), 1.0, g), W.draw_bf16((B, H, 64), 1.0, g)
    out, lse = mla.decode(_dims(x), qn.cuda(), qp.cuda(), cache, None, x["table"].cuda(), x["seq_lens"].cuda(),
                          x["W_UK"].cuda(), x["W_UV"].cuda(), x["scale"])
    torch.cuda.synchronize()
    ref_o, ref_l = O.decode(f64(qn), f64(qp), ref_cache, None, x["table"].numpy(), x["seq_lens"].numpy(),
                            f64(x["W_UK"]), f64(x["W_UV"]), x["scale"], x["P"], False)
    assert_parity(out, lse, ref_o, ref_l, [(b, h) for b in range(B) for h in range(H)], "decode after prefill")


@pytest.mark.parametrize("fmt,P,heads,theta", [("fp8", 16, 128, 10000.0), ("int8", 128, 16, 10000.0),
                                               ("bf16", 32, 32, 10000.0)])
def test_prefill_formats_pages_heads(cuda_lib, fmt, P, heads, theta):
    """Quantised caches with RoPE on (the two appends may differ by a bf16
    ulp in the rotated key, so only the attention is compared), page sizes
    16 / 32 / 128, 16 to 128 heads."""
    _check(_pf(heads=heads, P=P, hist=(200, 513), chunk=24, fmt=fmt, theta=theta, seed=48 + P), sample=12)
