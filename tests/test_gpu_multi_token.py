"""GPU parity of multi-token decode (mla_decode_multi: q_len new tokens per
sequence, causal among themselves) against the fp64 oracle's
decode_multi_token, through the C ABI.

Cases span several tiles and ragged tails, sequences shorter than q_len
(queries that see nothing), lengths just past a tile boundary with many
splits (segments in which some queries see no token), 16/32/128 heads,
q_len up to MLA_MAX_Q_LEN, and bf16 and INT8 caches."""
import numpy as np
import pytest
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import assert_parity, f64

pytestmark = pytest.mark.gpu


def _mt(heads=16, T=2, P=64, lens=(300,), int8=False, seed=17, fp8=False):
    g = W.generator(seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, True, g, spare_pages=3)
    x = dict(seq_lens=seq_lens, table=table, P=P, heads=heads, T=T, int8=int8, fp8=fp8,
             scale=1.0 / np.sqrt(192.0))
    if int8:
        x["codes"], x["sz"] = W.draw_int8_cache(npg, P, g)
    elif fp8:
        x["codes"], x["sz"] = W.draw_fp8_cache(npg, P, g)
    else:
        x["cache"] = W.draw_bf16((npg, P, 576), 1.0, g)
    x["W_UK"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    x["W_UV"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    x["q_nope"] = W.draw_bf16((len(lens), T, heads, 128), 1.0, g)
    x["q_pe"] = W.draw_bf16((len(lens), T, heads, 64), 1.0, g)
    return x


def _gpu(x, num_splits=0):
    d = mla.dims(x["heads"], x["P"], int8=x["int8"], fp8=x["fp8"])
    if x["int8"] or x["fp8"]:
        cache, sz = x["codes"].cuda(), x["sz"].cuda()
    else:
        cache, sz = x["cache"].cuda(), None
    out, lse = mla.decode_multi(d, x["q_nope"].cuda(), x["q_pe"].cuda(), cache, sz, x["table"].cuda(),
                                x["seq_lens"].cuda(), x["W_UK"].cuda(), x["W_UV"].cuda(), x["scale"],
                                num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def _oracle(x):
    if x["int8"] or x["fp8"]:
        cache, sz = x["codes"].numpy(), x["sz"].numpy()
    else:
        cache, sz = W.bf16_to_bits(x["cache"]), None
    return O.decode_multi_token(f64(x["q_nope"]), f64(x["q_pe"]), cache, sz, x["table"].numpy(),
                                x["seq_lens"].numpy(), f64(x["W_UK"]), f64(x["W_UV"]), x["scale"], x["P"],
                                x["int8"], fp8=x["fp8"])


def _check(x, num_splits=0):
    out, lse = _gpu(x, num_splits)
    ref_o, ref_l = _oracle(x)
    B, T, H = out.shape[0], out.shape[1], out.shape[2]
    pairs = [(b, v) for b in range(B) for v in range(T * H)]
    # rows of a sequence as (token, head) pairs: v = t * H + h
    assert_parity(out.reshape(B, T * H, -1), lse.reshape(B, T * H), ref_o.reshape(B, T * H, -1),
                  ref_l.reshape(B, T * H), pairs, f"T{T} H{H}")
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("T", [2, 3, 4, 8])
def test_multi_token_ragged(cuda_lib, T):
    out, lse, _, ref_l = _check(_mt(T=T, lens=(1, 2, 3, 129, 700, 256), seed=30 + T))
    # sequences shorter than T: the queries below position 0 see nothing
    for b, L in enumerate((1, 2, 3)):
        for t in range(max(0, T - L)):
            assert torch.all(out[b, t] == 0) and torch.all(torch.isneginf(lse[b, t]))


@pytest.mark.parametrize("heads,T", [(32, 2), (128, 2), (16, 5)])
def test_multi_token_head_counts(cuda_lib, heads, T):
    _check(_mt(heads=heads, T=T, lens=(383, 130), seed=50 + heads + T))


@pytest.mark.parametrize("splits", [1, 7, 1000])
def test_multi_token_segments_with_invisible_rows(cuda_lib, splits):
    # one token past a tile boundary: with many splits that token is a
    # segment of its own, which queries t < T - 1 cannot see
    _check(_mt(T=4, lens=(129, 257, 385, 1000), seed=61), num_splits=splits)


def test_multi_token_int8(cuda_lib):
    _check(_mt(T=2, lens=(200, 1030, 3), int8=True, seed=71))


def test_single_query_is_mla_decode_bit_for_bit(cuda_lib):
    x = _mt(T=1, lens=(700, 33), seed=81)
    out, lse = _gpu(x)
    d = mla.dims(16, 64)
    o1, l1 = mla.decode(d, x["q_nope"][:, 0].contiguous().cuda(), x["q_pe"][:, 0].contiguous().cuda(),
                        x["cache"].cuda(), None, x["table"].cuda(), x["seq_lens"].cuda(), x["W_UK"].cuda(),
                        x["W_UV"].cuda(), x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], o1) and torch.equal(lse[:, 0], l1)


def test_q_len_out_of_range_is_refused(cuda_lib):
    x = _mt(T=mla.MAX_Q_LEN + 1, lens=(10,), seed=91)
    with pytest.raises(mla.MLAError) as e:
        _gpu(x)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_multi_token_fp8(cuda_lib):
    _check(_mt(T=3, lens=(200, 1030, 2), fp8=True, seed=72))


@pytest.mark.parametrize("P,T", [(128, 2), (16, 5)])
def test_multi_token_fp8_page_sizes(cuda_lib, P, T):
    _check(_mt(T=T, P=P, lens=(700, 129, 3), fp8=True, seed=73 + P))
