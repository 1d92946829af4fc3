"""GPU parity of sparse (top-k) decode (mla_decode_sparse) against the fp64
oracle's decode_sparse, through the C ABI: random selections in random
order with padding, lists longer than a sequence's selection, list lengths
that are not multiples of the gather's chunk, 16 and 128 heads, bf16 and
INT8 caches, an empty selection, a bad entry, and the all-positions case,
which must equal mla_decode bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import assert_parity, f64

pytestmark = pytest.mark.gpu


def _sp(heads=16, P=64, lens=(300,), top_k=100, fill=0.8, int8=False, seed=23, fp8=False):
    g = W.generator(seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, True, g, spare_pages=3)
    x = dict(seq_lens=seq_lens, table=table, P=P, heads=heads, int8=int8, fp8=fp8, scale=1.0 / np.sqrt(192.0))
    if int8:
        x["codes"], x["sz"] = W.draw_int8_cache(npg, P, g)
    elif fp8:
        x["codes"], x["sz"] = W.draw_fp8_cache(npg, P, g)
    else:
        x["cache"] = W.draw_bf16((npg, P, 576), 1.0, g)
    x["W_UK"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    x["W_UV"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    x["q_nope"] = W.draw_bf16((len(lens), heads, 128), 1.0, g)
    x["q_pe"] = W.draw_bf16((len(lens), heads, 64), 1.0, g)
    x["idx"] = W.draw_token_indices(seq_lens, top_k, fill, g)
    return x


def _gpu(x, num_splits=0, idx=None):
    d = mla.dims(x["heads"], x["P"], int8=x["int8"], fp8=x["fp8"])
    cache, sz = (x["codes"].cuda(), x["sz"].cuda()) if (x["int8"] or x["fp8"]) else (x["cache"].cuda(), None)
    idx = x["idx"] if idx is None else idx
    ws = torch.empty(mla.decode_sparse_workspace_size(d, len(x["seq_lens"]), idx.shape[1], num_splits),
                     dtype=torch.uint8, device="cuda")
    out, lse = mla.decode_sparse(d, x["q_nope"].cuda(), x["q_pe"].cuda(), cache, sz, x["table"].cuda(),
                                 x["seq_lens"].cuda(), idx.cuda(), x["W_UK"].cuda(), x["W_UV"].cuda(), x["scale"],
                                 num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, mla.read_device_status(ws)


def _oracle(x, idx=None):
    quantised = x["int8"] or x["fp8"]
    cache, sz = (x["codes"].numpy(), x["sz"].numpy()) if quantised else (W.bf16_to_bits(x["cache"]), None)
    return O.decode_sparse(f64(x["q_nope"]), f64(x["q_pe"]), cache, sz, x["table"].numpy(), x["seq_lens"].numpy(),
                           (x["idx"] if idx is None else idx).numpy(), f64(x["W_UK"]), f64(x["W_UV"]), x["scale"],
                           x["P"], x["int8"], fp8=x["fp8"])


def _check(x, num_splits=0):
    out, lse, st = _gpu(x, num_splits)
    assert st == mla.MLA_OK
    ref_o, ref_l = _oracle(x)
    pairs = [(b, h) for b in range(out.shape[0]) for h in range(out.shape[1])]
    assert_parity(out, lse, ref_o, ref_l, pairs, "sparse")
    return out, lse


@pytest.mark.parametrize("P,top_k", [(64, 100), (16, 2048), (128, 777)])
def test_sparse_random_selections(cuda_lib, P, top_k):
    _check(_sp(P=P, lens=(1, 300, 2500, 129, 5000), top_k=top_k, seed=P + top_k))


@pytest.mark.parametrize("heads,int8", [(128, False), (16, True), (128, True)])
def test_sparse_heads_and_int8(cuda_lib, heads, int8):
    _check(_sp(heads=heads, lens=(700, 3000), top_k=300, int8=int8, seed=heads + int8))


def test_sparse_many_splits(cuda_lib):
    _check(_sp(lens=(4000, 9000, 30), top_k=1500, seed=77), num_splits=500)


def test_sparse_all_positions_equals_dense_decode(cuda_lib):
    x = _sp(lens=(700, 129, 2000), top_k=2000, seed=88)
    L = x["seq_lens"]
    idx = torch.full((3, 2000), -1, dtype=torch.int32)
    for b in range(3):
        idx[b, : int(L[b])] = torch.arange(int(L[b]), dtype=torch.int32)
    out, lse, st = _gpu(x, idx=idx)
    assert st == mla.MLA_OK
    d = mla.dims(16, 64)
    o1, l1 = mla.decode(d, x["q_nope"].cuda(), x["q_pe"].cuda(), x["cache"].cuda(), None, x["table"].cuda(),
                        L.cuda(), x["W_UK"].cuda(), x["W_UV"].cuda(), x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(lse, l1)


def test_sparse_empty_selection_and_bad_entry(cuda_lib):
    x = _sp(lens=(500, 400), top_k=64, seed=99)
    idx = x["idx"].clone()
    idx[0] = -1                       # nothing selected
    out, lse, st = _gpu(x, idx=idx)
    assert st == mla.MLA_OK
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ref_o, ref_l = _oracle(x, idx)
    assert_parity(out, lse, ref_o, ref_l, [(1, h) for h in range(16)], "sparse")
    bad = idx.clone()
    bad[1, 3] = 400                   # == seq_len: out of range, reported and skipped
    out2, lse2, st2 = _gpu(x, idx=bad)
    assert st2 == mla.MLA_ERR_DEVICE_BOUNDS
    # the oracle skips the out-of-range entry itself: it gets the list as the library did
    ref_o, ref_l = _oracle(x, bad)
    assert_parity(out2, lse2, ref_o, ref_l, [(1, h) for h in range(16)], "sparse, bad entry skipped")


@pytest.mark.parametrize("heads", [16, 128])
def test_sparse_fp8(cuda_lib, heads):
    _check(_sp(heads=heads, lens=(700, 3000), top_k=300, fp8=True, seed=heads + 7))


@pytest.mark.parametrize("P", [16, 128])
def test_sparse_fp8_page_sizes(cuda_lib, P):
    _check(_sp(P=P, lens=(900, 2000), top_k=257, fp8=True, seed=91 + P))
