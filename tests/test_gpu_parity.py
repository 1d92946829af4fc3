"""GPU parity of the library against the fp64 oracle, through the C ABI.

Small cases compare every (b, h) element by element; they span several
128-token tiles, ragged tails, every page size, single- and multi-chunk
splits, 16/32/64/128 heads, bf16, INT8 and FP8 caches and the degenerate cases
(empty sequence, one token, lengths at tile boundaries)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import (assert_parity, dims_of, f64, gpu_cache, gpu_decode, oracle_cache, oracle_decode)

pytestmark = pytest.mark.gpu


def _small(heads=16, P=64, lens=(300,), int8=False, seed=7, std=1.0, shuffled=True, fp8=False):
    w = W.Workload(f"small_h{heads}_p{P}", len(lens), heads, 0, P, shuffled, std, 0.02, 1.0, seed, int8=int8,
                   fp8=fp8)
    g = W.generator(seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, shuffled, g, spare_pages=3)
    inp = dict(workload=w, seq_lens=seq_lens, block_table=table, num_pages=npg, page_size=P, scale=w.softmax_scale)
    if int8:
        codes, sz = W.draw_int8_cache(npg, P, g)
        inp["cache_i8"], inp["sz"] = codes, sz
    elif fp8:
        codes, sc = W.draw_fp8_cache(npg, P, g)
        inp["cache_i8"], inp["sz"] = codes, sc
    else:
        inp["cache"] = W.draw_bf16((npg, P, 576), std, g)
    inp["W_UK"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    inp["W_UV"] = W.draw_bf16((heads, 128, 512), 0.02, g)
    inp["q_nope"] = W.draw_bf16((len(lens), heads, 128), 1.0, g)
    inp["q_pe"] = W.draw_bf16((len(lens), heads, 64), 1.0, g)
    return w, inp


def _run_small(w, inp, num_splits=0):
    if w.quantised:
        cache, sz = inp["cache_i8"].cuda(), inp["sz"].cuda()
        oc = (inp["cache_i8"].numpy(), inp["sz"].numpy(), inp["block_table"].numpy())
    else:
        cache, sz = inp["cache"].cuda(), None
        oc = (W.bf16_to_bits(inp["cache"]), None, inp["block_table"].numpy())
    out, lse = gpu_decode(inp, w, cache, sz, num_splits=num_splits)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.heads)]
    ref_o, ref_l = oracle_decode(inp, w, pairs, cache_override=oc)
    return assert_parity(out, lse, ref_o, ref_l, pairs, w.name), out, lse


def test_tiny_workload_full_oracle(cuda_lib):
    w = W.WORKLOADS["tiny"]
    inp = W.make_decode_inputs(w)
    cache, sz = gpu_cache(inp, w)
    out, lse = gpu_decode(inp, w, cache, sz)
    pairs = [(0, h) for h in range(w.heads)]
    ref_o, ref_l = oracle_decode(inp, w, pairs)
    assert_parity(out, lse, ref_o, ref_l, pairs, w.name)


@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_page_sizes_ragged(cuda_lib, P):
    _run_small(*_small(P=P, lens=(1, 129, 700, 256)))


@pytest.mark.parametrize("heads", [16, 32, 64, 128])
def test_head_counts(cuda_lib, heads):
    _run_small(*_small(heads=heads, lens=(383, 130)))


@pytest.mark.parametrize("splits", [1, 2, 5, 64, 1000])
def test_split_counts(cuda_lib, splits):
    _run_small(*_small(lens=(1000, 5, 2500, 128)), num_splits=splits)


def test_tile_boundaries_and_empty(cuda_lib):
    w, inp = _small(lens=(0, 1, 127, 128, 129, 255, 256, 257, 0))
    (_, _), out, lse = _run_small(w, inp)
    assert torch.all(out[0] == 0) and torch.all(out[-1] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[-1]))


@pytest.mark.parametrize("heads", [16, 128])
def test_int8_cache_decode(cuda_lib, heads):
    _run_small(*_small(heads=heads, lens=(200, 1030), int8=True))


@pytest.mark.parametrize("heads", [16, 128])
def test_fp8_cache_decode(cuda_lib, heads):
    _run_small(*_small(heads=heads, lens=(200, 1030), fp8=True, seed=8))


@pytest.mark.parametrize("P", [16, 128])
def test_fp8_page_sizes_ragged(cuda_lib, P):
    _run_small(*_small(P=P, lens=(1, 129, 700), fp8=True, seed=9))


def test_fp8_tile_boundaries_empty_and_splits(cuda_lib):
    w, inp = _small(lens=(0, 1, 127, 128, 129, 257), fp8=True, seed=10)
    (_, _), out, lse = _run_small(w, inp, num_splits=7)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_fp8_accepts_float8_tensor(cuda_lib):
    """The E4M3 codes may be held as torch.float8_e4m3fn: same bits, same results."""
    w, inp = _small(lens=(300,), fp8=True, seed=11)
    codes, sc = inp["cache_i8"].cuda(), inp["sz"].cuda()
    o1, l1 = gpu_decode(inp, w, codes, sc)
    o2, l2 = gpu_decode(inp, w, codes.view(torch.float8_e4m3fn), sc)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("fmt", ["bf16", "int8", "fp8"])
def test_nan_patterns_past_the_sequence_end_do_not_reach_the_output(cuda_lib, fmt):
    """The rows of a sequence's last page past its length are never part of
    the attention; filled with NaN bit patterns (bf16 0x7FC0, E4M3 0x7F /
    0xFF; any INT8 byte is a number) they must not reach the output."""
    w, inp = _small(lens=(200, 1030, 77), int8=fmt == "int8", fp8=fmt == "fp8", seed=12)
    P = w.page_size
    table = inp["block_table"]
    for b, L in enumerate(inp["seq_lens"].tolist()):
        if L % P:
            page = int(table[b, (L - 1) // P])
            if fmt == "bf16":
                inp["cache"].view(torch.int16)[page, L % P:] = 0x7FC0
            else:
                inp["cache_i8"].view(torch.uint8)[page, L % P:, 0::2] = 0x7F
                inp["cache_i8"].view(torch.uint8)[page, L % P:, 1::2] = 0xFF
    (_, _), out, lse = _run_small(w, inp)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_shuffled_table_bit_identical_and_deterministic(cuda_lib):
    """Same rows reached through a different physical layout give bit-identical
    results for the same split plan; repeated runs are bit-identical."""
    w, inp = _small(lens=(900, 77, 1500), shuffled=False)
    cache = inp["cache"].cuda()
    out1, lse1 = gpu_decode(inp, w, cache, None, num_splits=7)
    out1b, lse1b = gpu_decode(inp, w, cache, None, num_splits=7)
    assert torch.equal(out1, out1b) and torch.equal(lse1, lse1b)
    npg = cache.shape[0]
    perm = torch.randperm(npg, generator=W.generator(99))
    cache2 = torch.empty_like(cache)
    cache2[perm.cuda()] = cache
    table2 = inp["block_table"].clone()
    m = table2 >= 0
    table2[m] = perm[table2[m].long()].to(torch.int32)
    out2, lse2 = gpu_decode(inp, w, cache2, None, num_splits=7, block_table=table2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_out_of_range_length_sets_status(cuda_lib):
    w, inp = _small(lens=(300, 200))
    d = dims_of(w)
    seq_lens = torch.tensor([300, 10 ** 6], dtype=torch.int32, device="cuda")  # second exceeds its pages
    ws = torch.empty(mla.decode_workspace_size(d, 2), dtype=torch.uint8, device="cuda")
    out, lse = mla.decode(d, inp["q_nope"].cuda(), inp["q_pe"].cuda(), inp["cache"].cuda(), None,
                          inp["block_table"].cuda(), seq_lens, inp["W_UK"].cuda(), inp["W_UV"].cuda(),
                          inp["scale"], workspace=ws)
    assert mla.read_device_status(ws) == mla.MLA_ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    # a clean call resets the status word
    mla.decode(d, inp["q_nope"].cuda(), inp["q_pe"].cuda(), inp["cache"].cuda(), None, inp["block_table"].cuda(),
               inp["seq_lens"].cuda(), inp["W_UK"].cuda(), inp["W_UV"].cuda(), inp["scale"], workspace=ws)
    assert mla.read_device_status(ws) == mla.MLA_OK


def test_combine_matches_oracle(cuda_lib):
    rng = np.random.default_rng(3)
    B, S, H = 3, 6, 16
    po = rng.normal(0, 1, (B, S, H, 512)).astype(np.float32)
    pl = rng.normal(0, 3, (B, S, H)).astype(np.float32)
    pl[0, 2] = -np.inf          # empty chunks
    pl[2, :, 5] = -np.inf       # every chunk empty for (2, 5)
    d = mla.dims(H, 64)
    o, l = mla.combine(d, torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda())
    o, l = o.cpu().numpy(), l.cpu().numpy()
    for b in range(B):
        for h in range(H):
            ro, rl = O.combine_partials(po[b, :, h].astype(np.float64), pl[b, :, h].astype(np.float64))
            np.testing.assert_allclose(o[b, h], ro, rtol=1e-5, atol=1e-6)
            if math.isinf(rl):
                assert np.isneginf(l[b, h])
            else:
                assert abs(l[b, h] - rl) < 1e-5


# ------------------------------------------------------------------ append --- #

def _append_case(int8, theta, seed=5, fp8=False):
    P, B, maxp = 16, 3, 6
    g = W.generator(seed)
    table, npg = W.draw_page_table(torch.tensor([maxp * P] * B, dtype=torch.int32), P, True, g)
    n = 150
    seq_ids = torch.randint(0, B, (n,), generator=g, dtype=torch.int32)
    pos = torch.randperm(B * maxp * P, generator=g)[:n]
    seq_ids = (pos // (maxp * P)).to(torch.int32)
    pos = (pos % (maxp * P)).to(torch.int32)
    c = W.draw_bf16((n, 512), 1.0, g)
    k = W.draw_bf16((n, 64), 1.0, g)
    d = mla.dims(16, P, int8=int8, fp8=fp8)
    if int8:
        cache = torch.zeros((npg, P, 576), dtype=torch.int8, device="cuda")
        sz = torch.zeros((npg, P, 2), dtype=torch.float32, device="cuda")
        ref = np.zeros((npg, P, 576), np.int8)
        rsz = np.zeros((npg, P, 2), np.float32)
    elif fp8:
        cache = torch.zeros((npg, P, 576), dtype=torch.uint8, device="cuda")
        sz = torch.zeros((npg, P), dtype=torch.float32, device="cuda")
        ref = np.zeros((npg, P, 576), np.uint8)
        rsz = np.zeros((npg, P), np.float32)
    else:
        cache = torch.zeros((npg, P, 576), dtype=torch.bfloat16, device="cuda")
        sz, ref, rsz = None, np.zeros((npg, P, 576), np.uint16), None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.cache_append(d, cache, sz, table.cuda(), seq_ids.cuda(), pos.cuda(), c.cuda(), k.cuda(), theta, st)
    O.append_tokens(ref, rsz, table.numpy(), seq_ids.tolist(), pos.tolist(), W.bf16_to_bits(c),
                    W.bf16_to_bits(k), theta, P, int8=int8, fp8=fp8)
    assert mla.read_status_word(st) == mla.MLA_OK
    return cache, sz, ref, rsz


def test_append_bf16_bit_exact_without_rope(cuda_lib):
    cache, _, ref, _ = _append_case(False, 0.0)
    np.testing.assert_array_equal(W.bf16_to_bits(cache), ref)


def test_append_bf16_rope_within_one_ulp(cuda_lib):
    cache, _, ref, _ = _append_case(False, 10000.0)
    got = W.bf16_to_bits(cache)
    np.testing.assert_array_equal(got[..., :512], ref[..., :512])            # latent copied exactly
    g = O.bf16_bits_to_f64(got[..., 512:])
    r = O.bf16_bits_to_f64(ref[..., 512:])
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), 1e-30))[1] - 8)
    assert np.all(np.abs(g - r) <= ulp)
    assert np.mean(g == r) > 0.99


def test_append_int8_codes_bit_exact_without_rope(cuda_lib):
    cache, sz, ref, rsz = _append_case(True, 0.0)
    np.testing.assert_array_equal(cache.cpu().numpy(), ref)
    np.testing.assert_array_equal(sz.cpu().numpy(), rsz)


def test_append_fp8_codes_bit_exact_without_rope(cuda_lib):
    cache, sz, ref, rsz = _append_case(False, 0.0, fp8=True)
    np.testing.assert_array_equal(cache.cpu().numpy(), ref)
    np.testing.assert_array_equal(sz.cpu().numpy(), rsz)


def test_append_fp8_ties_saturation_and_signed_zero(cuda_lib):
    """A row whose largest magnitude is 448 has scale 1, so its codes are the
    format's own rounding of the values: ties to the even mantissa, subnormal
    ties, -0 and negative values that round to zero."""
    P = 16
    special = [448.0, 1.0625, -1.1875, 3 * 2.0 ** -10, 2.0 ** -10, -0.0, -(2.0 ** -10), 248.0, 15 * 2.0 ** -10,
               -448.0, 1.09375, 240.0, -(2.0 ** -12), 0.5, 7 * 2.0 ** -9]
    c = torch.zeros((2, 512), dtype=torch.float32)
    c[0, :len(special)] = torch.tensor(special)
    c[1, :] = torch.linspace(-3.0, 2.0, 512)          # an ordinary row: scale 3/448
    c = c.to(torch.bfloat16)
    assert all(float(v) == x for v, x in zip(c[0, :len(special)], special))  # all exact in bf16
    k = torch.zeros((2, 64), dtype=torch.bfloat16)
    table = torch.tensor([[0]], dtype=torch.int32)
    d = mla.dims(16, P, fp8=True)
    cache = torch.zeros((1, P, 576), dtype=torch.uint8, device="cuda")
    sz = torch.zeros((1, P), dtype=torch.float32, device="cuda")
    pos = torch.tensor([0, 1], dtype=torch.int32)
    mla.cache_append(d, cache, sz, table.cuda(), torch.zeros(2, dtype=torch.int32, device="cuda"), pos.cuda(),
                     c.cuda(), k.cuda(), 0.0)
    ref = np.zeros((1, P, 576), np.uint8)
    rsz = np.zeros((1, P), np.float32)
    O.append_tokens(ref, rsz, table.numpy(), [0, 0], [0, 1], W.bf16_to_bits(c), W.bf16_to_bits(k), 0.0, P,
                    int8=False, fp8=True)
    got = cache.cpu().numpy()
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(sz.cpu().numpy(), rsz)
    assert sz[0, 0].item() == 1.0
    np.testing.assert_array_equal(got[0, 0, :len(special)], O.e4m3_encode(np.array(special, np.float32)))


def test_append_out_of_range_sets_status(cuda_lib):
    P = 16
    table = torch.tensor([[0, 1], [2, -1]], dtype=torch.int32, device="cuda")
    cache = torch.zeros((3, P, 576), dtype=torch.bfloat16, device="cuda")
    c = torch.ones((3, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((3, 64), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # token 0 ok, token 1 hits a -1 table entry, token 2 has a bad sequence id
    mla.cache_append(mla.dims(16, P), cache, None, table, torch.tensor([0, 1, 5], dtype=torch.int32, device="cuda"),
                     torch.tensor([3, 20, 0], dtype=torch.int32, device="cuda"), c, k, 0.0, st)
    assert mla.read_status_word(st) == mla.MLA_ERR_DEVICE_BOUNDS
    assert float(cache[0, 3, 0]) == 1.0 and float(cache.float().sum()) == 576.0


def test_large_batch_plan_chunks(cuda_lib):
    """More sequences than the plan CTA has threads (128): the length scan and
    the segment scan each run in several passes."""
    rng = np.random.default_rng(300)
    lens = [int(x) for x in rng.integers(0, 400, 300)]
    lens[0], lens[150], lens[299] = 0, 1, 128
    _run_small(*_small(lens=tuple(lens), seed=300), num_splits=97)


def test_256_heads(cuda_lib):
    _run_small(*_small(heads=256, lens=(700, 1), seed=256))
