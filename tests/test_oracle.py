"""Pins for the fp64 oracle: each test checks it against something other than
itself -- the pages' printed figures, closed forms, a library routine, or
invariants of the mathematics.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _bf16(x):
    return O.round_to_bf16(np.asarray(x, np.float64))


def _rand_head(L, rng, std_c=1.0, std_w=0.02):
    rows = _bf16(rng.normal(0, std_c, (L, O.ROW_DIM)))
    W_UK = _bf16(rng.normal(0, std_w, (128, 512)))
    W_UV = _bf16(rng.normal(0, std_w, (128, 512)))
    q_nope = _bf16(rng.normal(0, 1, 128))
    q_pe = _bf16(rng.normal(0, 1, 64))
    return q_nope, q_pe, rows, W_UK, W_UV


# ----------------------------------------------------------------- bf16 ---- #

def test_bf16_rounding_matches_torch_on_fp32_values():
    # For inputs that are exact fp32 values the one-step fp64 -> bf16 rounding
    # must equal torch's fp32 -> bf16 conversion (round to nearest even).
    x32 = RNG.normal(0, 3, 20000).astype(np.float32)
    x32 = np.concatenate([x32, np.float32([1e-40, -3e-39, 3.3e38, 0.0, -0.0, 1.0, 65504.0])])
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_bf16(x32.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_rounding_ties_to_even():
    assert O.round_to_bf16(1 + 2.0 ** -8) == 1.0                      # halfway, keep even 1.0
    assert O.round_to_bf16(1 + 3 * 2.0 ** -8) == 1 + 2 * 2.0 ** -7    # halfway, round up to even
    assert O.round_to_bf16(-(1 + 2.0 ** -8 + 2.0 ** -20)) == -(1 + 2.0 ** -7)
    assert np.isinf(O.round_to_bf16(3.5e38))
    bits = O.f64_to_bf16_bits(np.array([1.0, -2.0, 0.5]))
    np.testing.assert_array_equal(bits, np.array([0x3F80, 0xC000, 0x3F00], np.uint16))
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), [1.0, -2.0, 0.5])


# ------------------------------------------------------- cache footprint ---- #

def test_cache_footprint_matches_page_figures():
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))
    e = g["v2lite_latent_bytes_per_token"]
    assert O.latent_cache_bytes_per_token(e["layers"], e["latent_dim"], e["rope_dim"], e["elem_bytes"]) == e["value"]
    e = g["v2lite_latent_mib_at_32k"]
    assert O.latent_cache_bytes_per_token(e["layers"]) * e["tokens"] / 2 ** 20 == e["value_mib"]
    e = g["v2lite_per_head_mib_at_32k"]
    naive = O.per_head_cache_bytes_per_token(e["layers"], e["kv_heads"], e["key_dim"], e["value_dim"], e["elem_bytes"])
    assert naive * e["tokens"] / 2 ** 20 == e["value_mib"]
    # "Both runtimes used a ninth of the calculation"
    assert 8.5 < naive / O.latent_cache_bytes_per_token(27) < 9.5
    e = g["v3_latent_bytes_per_token_per_layer"]
    assert O.latent_cache_bytes_per_token(e["layers"]) == e["value"]
    e3 = g["v3_mha_equivalent_bytes_per_token_per_layer"]
    mha = O.per_head_cache_bytes_per_token(1, e3["kv_heads"], e3["key_dim"], e3["value_dim"], e3["elem_bytes"])
    assert mha == e3["value"] and round(mha / O.latent_cache_bytes_per_token(1)) == e3["ratio_rounded"]
    e = g["kimi_linear_7_mla_layers_mib_at_32k"]
    assert O.latent_cache_bytes_per_token(e["layers"]) * e["tokens"] / 2 ** 20 == e["value_mib"]
    e = g["llama70b_kv_bytes_at_100k"]
    b = O.per_head_cache_bytes_per_token(e["layers"], e["kv_heads"], e["head_dim"], e["head_dim"], e["elem_bytes"])
    assert round(b * e["tokens"] / 1e9) == e["value_gb"]
    for k in ("llama2_7b_kib_per_token", "falcon7b_kib_per_token"):
        e = g[k]
        b = O.per_head_cache_bytes_per_token(e["layers"], e["kv_heads"], e["head_dim"], e["head_dim"], e["elem_bytes"])
        assert b / 1024 == e["value_kib"]
    # INT8 latent row: 576 one-byte codes + fp32 scale and zero point
    assert O.latent_cache_bytes_per_token(1, elem_bytes=1, side_bytes_per_row=8) == 584


# ------------------------------------------------------------------ RoPE ---- #

def test_rope_closed_forms():
    x = np.zeros(64)
    x[0], x[32] = 1.0, 1.0
    # pair 0 turns at 1 rad per position; pair 16 at theta**(-1/2) = 0.01 rad per position
    r = O.rope_rotate(x[None], np.array([1]), 10000.0)[0]
    assert r[0] == pytest.approx(math.cos(1.0), abs=1e-15) and r[1] == pytest.approx(math.sin(1.0), abs=1e-15)
    r = O.rope_rotate(x[None], np.array([100]), 10000.0)[0]
    assert r[32] == pytest.approx(math.cos(1.0), abs=1e-13) and r[33] == pytest.approx(math.sin(1.0), abs=1e-13)
    np.testing.assert_array_equal(O.rope_rotate(x[None], np.array([0]), 10000.0)[0], x)
    np.testing.assert_array_equal(O.rope_rotate(x[None], np.array([777]), 0.0)[0], x)


def test_rope_invariants():
    q = RNG.normal(size=(64,))
    k = RNG.normal(size=(64,))
    for m, n in [(0, 0), (5, 3), (1000, 998), (1 << 20, (1 << 20) - 2)]:
        rq = O.rope_rotate(q[None], np.array([m]), 10000.0)[0]
        rk = O.rope_rotate(k[None], np.array([n]), 10000.0)[0]
        assert np.linalg.norm(rq) == pytest.approx(np.linalg.norm(q), rel=1e-12)
        # the score depends on positions only through m - n
        r0 = O.rope_rotate(q[None], np.array([m - n]), 10000.0)[0]
        assert rq @ rk == pytest.approx(r0 @ k, rel=1e-9, abs=1e-9)


# ------------------------------------------------------------------ INT8 ---- #

def test_int8_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "int8_worked_examples.json")))
    for case in g["cases"]:
        codes, s, zp = O.quantize_tokens_int8(np.array(case["row"], np.float32))
        np.testing.assert_array_equal(codes[0], np.array(case["codes"], np.int8), err_msg=case["why"])
        assert zp[0] == case["zero_point"]
        assert s[0] == np.float32(np.float32(case["scale_num"]) / np.float32(case["scale_den"]))


def test_int8_error_bound_and_zero():
    rows = (RNG.normal(0, 1, (200, 576)) * RNG.uniform(0.01, 100, (200, 1))).astype(np.float32)
    rows[:, 7] = 0.0
    rows[3] = np.abs(rows[3])   # all non-negative row
    rows[4] = -np.abs(rows[4])  # all non-positive row
    codes, s, zp = O.quantize_tokens_int8(rows)
    xh = O.dequantize_tokens_int8(codes, s, zp)
    err = np.abs(xh - rows.astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))
    np.testing.assert_array_equal(xh[:, 7], 0.0)
    assert codes.min() >= -128 and codes.max() <= 127
    # monotone: larger input never gets a smaller code
    order = np.argsort(rows, axis=1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(codes.astype(int), order, 1), axis=1) >= 0)


# ------------------------------------------------------------------- FP8 ---- #

def _fp8_golden():
    return json.load(open(os.path.join(GOLDEN, "fp8_e4m3_worked_examples.json")))


def test_fp8_e4m3_worked_values():
    g = _fp8_golden()
    for case in g["decode"]:
        v = O.e4m3_value(np.array([case["code"]], np.uint8))[0]
        if case["value"] == "nan":
            assert np.isnan(v), case["why"]
        else:
            assert v == case["value"] and np.signbit(v) == np.signbit(case["value"]), case["why"]
    for case in g["encode"]:
        c = O.e4m3_encode(np.array([case["value"]], np.float32))[0]
        assert int(c) == case["code"], case["why"]
    for case in g["quantize"]:
        codes, s = O.quantize_tokens_fp8(np.array(case["row"], np.float32))
        np.testing.assert_array_equal(codes[0], np.array(case["codes"], np.uint8), err_msg=case["why"])
        assert s[0] == np.float32(np.float32(case["scale_num"]) / np.float32(case["scale_den"]))


def test_fp8_e4m3_format_closed_forms():
    v = O.e4m3_value(np.arange(256))
    finite = ~np.isnan(v)
    assert finite.sum() == 254                      # two NaN patterns, no infinities
    assert np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # magnitudes rise with the code
    np.testing.assert_array_equal(v[0x80:0xFF], -pos)
    # each binade [2^e, 2^(e+1)) holds 8 evenly spaced values; subnormals step by 2^-9
    np.testing.assert_array_equal(np.diff(pos[:9]), np.full(8, 2.0 ** -9))
    for e in range(1, 15):
        np.testing.assert_array_equal(pos[8 * e: 8 * e + 8], 2.0 ** (e - 7) * (1 + np.arange(8) / 8))
    # every finite code survives decode -> encode
    codes = np.arange(256)[finite]
    np.testing.assert_array_equal(O.e4m3_encode(v[finite]), codes.astype(np.uint8))


def test_fp8_e4m3_encode_is_brute_force_nearest():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.normal(0, 1, 4000) * np.exp2(rng.uniform(-14, 10, 4000)),
                        rng.uniform(-500, 500, 1000)]).astype(np.float32)
    c = O.e4m3_encode(x)
    allv = O.e4m3_value(np.arange(256))
    fin = np.arange(256)[~np.isnan(allv)]
    xd = x.astype(np.float64)
    target = np.clip(xd, -448.0, 448.0)
    d_all = np.abs(target[:, None] - allv[fin][None, :])
    d_best = d_all.min(axis=1)
    got = np.abs(target - O.e4m3_value(c))
    np.testing.assert_array_equal(got, d_best)
    ties = (d_all == d_best[:, None]).sum(axis=1) > 1
    nonzero = O.e4m3_value(c) != 0
    assert np.all((c[ties & nonzero] & 1) == 0)     # ties went to the even mantissa
    assert np.all(np.signbit(O.e4m3_value(c)) == np.signbit(xd))


def test_fp8_quantize_error_bound_and_extremes():
    rows = (RNG.normal(0, 1, (200, 576)) * RNG.uniform(0.01, 100, (200, 1))).astype(np.float32)
    rows[:, 7] = 0.0
    rows[5] = 0.0                                   # an all-zero row
    codes, s = O.quantize_tokens_fp8(rows)
    xh = O.dequantize_tokens_fp8(codes, s)
    x = rows.astype(np.float64)
    sd = s[:, None].astype(np.float64)
    # half a step of E4M3 at the value (2^-4 relative in a binade, 2^-10 among
    # subnormals), plus the fp32 division's rounding
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sd * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(xh - x) <= bound)
    np.testing.assert_array_equal(xh[:, 7], 0.0)
    assert s[5] == 1.0 and np.all(codes[5] == 0)
    # the row's largest magnitude lands on +-448
    live = np.arange(200) != 5
    amax_at = np.abs(rows).argmax(axis=1)
    top = O.e4m3_value(codes[np.arange(200), amax_at])
    np.testing.assert_array_equal(np.abs(top[live]), 448.0)


# ------------------------------------------------------ paged addressing ---- #

def test_append_then_gather_roundtrip_and_injective_slots():
    P, B, maxp = 16, 3, 5
    perm = RNG.permutation(B * maxp)
    table = perm.reshape(B, maxp).astype(np.int32)
    cache = np.zeros((B * maxp, P, 576), np.uint16)
    lens = [1, 37, 80]
    seq_ids = [b for b in range(B) for _ in range(lens[b])]
    pos = [t for b in range(B) for t in range(lens[b])]
    src = _bf16(RNG.normal(0, 1, (len(pos), 576)))
    O.append_tokens(cache, None, table, seq_ids, pos, O.f64_to_bf16_bits(src[:, :512]),
                    O.f64_to_bf16_bits(src[:, 512:]), 0.0, P, int8=False)
    slots = {O.page_slot(table, b, t, P) for b, t in zip(seq_ids, pos)}
    assert len(slots) == len(pos)
    off = 0
    for b in range(B):
        rows = O.gather_rows(cache, None, table, b, lens[b], P, int8=False)
        np.testing.assert_array_equal(rows, src[off:off + lens[b]])
        off += lens[b]
    # with RoPE on, the stored key is the bf16 rounding of the fp64 rotation
    cache2 = np.zeros_like(cache)
    O.append_tokens(cache2, None, table, seq_ids, pos, O.f64_to_bf16_bits(src[:, :512]),
                    O.f64_to_bf16_bits(src[:, 512:]), 10000.0, P, int8=False)
    rows = O.gather_rows(cache2, None, table, 2, lens[2], P, int8=False)
    want = _bf16(O.rope_rotate(src[off - lens[2]:off, 512:], np.arange(lens[2]), 10000.0))
    np.testing.assert_array_equal(rows[:, 512:], want)


def _quantised_roundtrip_errors(fmt, gather):
    """Append seeded rows to a 1-byte cache through a shuffled page table with
    the oracle's own append, read them back with ``gather`` and return, per
    element, (|read back - source|, the quantiser's bound for that element).

    The bounds come from the formats alone, not from the oracle's dequantiser:
    INT8 rounds x / s to the nearest integer, so the read-back is within s / 2
    of x ("KV Cache Optimization", section 3: min/max quantisation); E4M3
    keeps 3 mantissa bits, so x / s lands within half a step of a code, i.e.
    within |x / s| * 2^-4 in the normal range and 2^-10 among the subnormals,
    and the read-back within s times that."""
    rng = np.random.default_rng(2024 if fmt == "int8" else 2025)
    P, B, maxp = 16, 3, 6
    table = rng.permutation(B * maxp).astype(np.int32).reshape(B, maxp)
    lens = [5, 41, 96]
    seq_ids = [b for b in range(B) for _ in range(lens[b])]
    pos = [t for b in range(B) for t in range(lens[b])]
    # rows of very different magnitudes, so that the per-token scales differ
    src = _bf16(rng.normal(0, 1, (len(pos), 576)) * rng.uniform(0.01, 50, (len(pos), 1)) +
                rng.uniform(-3, 3, (len(pos), 1)))
    int8 = fmt == "int8"
    cache = np.zeros((B * maxp, P, 576), np.int8 if int8 else np.uint8)
    sz = np.zeros((B * maxp, P, 2) if int8 else (B * maxp, P), np.float32)
    O.append_tokens(cache, sz, table, seq_ids, pos, O.f64_to_bf16_bits(src[:, :512]),
                    O.f64_to_bf16_bits(src[:, 512:]), 0.0, P, int8=int8, fp8=not int8)
    errs, bounds = [], []
    off = 0
    for b in range(B):
        got = gather(cache, sz, table, b, lens[b], P, int8=int8, fp8=not int8)
        x = src[off:off + lens[b]]
        if int8:  # the token's range widened to include 0, as the recipe defines it
            lo = np.minimum(x.min(axis=1), 0.0)
            hi = np.maximum(x.max(axis=1), 0.0)
            s = np.where(hi > lo, (hi - lo) / 255.0, 1.0)[:, None]
            bound = np.broadcast_to(s * (0.5 + 1e-5), x.shape)
        else:     # the token's largest magnitude maps to 448
            s = (np.abs(x).max(axis=1) / 448.0)[:, None]
            bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-5)
        errs.append(np.abs(got - x))
        bounds.append(bound)
        off += lens[b]
    return np.concatenate(errs), np.concatenate(bounds)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_quantised_gather_reads_back_within_the_quantiser_bound(fmt):
    """The 1-byte read-back branch of gather_rows: every element of every
    appended row comes back within the format's rounding bound of the source
    value, through a shuffled page table."""
    err, bound = _quantised_roundtrip_errors(fmt, O.gather_rows)
    assert np.all(err <= bound)
    assert np.mean(err) > 0  # the rows really went through the quantiser


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_quantised_gather_pin_catches_planted_mistakes(fmt):
    """Layout mistakes planted in the read-back must fail the bound: (scale,
    zero point) read in swapped order, and each token given its page
    neighbour's parameters."""
    good = O.gather_rows

    def swapped_scale_zero(cache, sz, *a, **k):
        return good(cache, sz[..., ::-1].copy(), *a, **k)

    def neighbour_params(cache, sz, *a, **k):
        return good(cache, np.roll(sz, 1, axis=1), *a, **k)

    planted = [neighbour_params] + ([swapped_scale_zero] if fmt == "int8" else [])
    for bad in planted:
        err, bound = _quantised_roundtrip_errors(fmt, bad)
        assert not np.all(err <= bound), bad.__name__


# ------------------------------------------------------------- attention ---- #

@pytest.mark.parametrize("L", [1, 2, 7, 64, 300])
def test_absorbed_equals_unabsorbed(L):
    rng = np.random.default_rng(L)
    q_nope, q_pe, rows, W_UK, W_UV = _rand_head(L, rng)
    o1, l1, _ = O.attend_unabsorbed(q_nope, q_pe, rows, W_UK, W_UV, 1 / math.sqrt(192))
    o2, l2, _ = O.attend_absorbed(q_nope, q_pe, rows, W_UK, W_UV, 1 / math.sqrt(192))
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-15)
    assert l1 == pytest.approx(l2, rel=1e-13)


def test_closed_forms():
    rng = np.random.default_rng(7)
    q_nope, q_pe, rows, W_UK, W_UV = _rand_head(9, rng)
    scale = 0.3
    # one token: the softmax weight is 1, so o = W^UV c_0 and lse = the score
    o, lse, p = O.attend_unabsorbed(q_nope, q_pe, rows[:1], W_UK, W_UV, scale)
    np.testing.assert_allclose(o, W_UV @ rows[0, :512], rtol=1e-13)
    s0 = scale * (q_nope @ (W_UK @ rows[0, :512]) + q_pe @ rows[0, 512:])
    assert lse == pytest.approx(s0, rel=1e-13) and p[0] == 1.0
    # equal rows: o = W^UV c for any query, lse = s + ln L
    eq = np.repeat(rows[:1], 9, axis=0)
    o, lse, _ = O.attend_unabsorbed(q_nope, q_pe, eq, W_UK, W_UV, scale)
    np.testing.assert_allclose(o, W_UV @ rows[0, :512], rtol=1e-12)
    assert lse == pytest.approx(s0 + math.log(9), rel=1e-12)
    # zero query: uniform weights, o = W^UV mean(c), lse = ln L
    o, lse, p = O.attend_unabsorbed(np.zeros(128), np.zeros(64), rows, W_UK, W_UV, scale)
    np.testing.assert_allclose(o, W_UV @ rows[:, :512].mean(axis=0), rtol=1e-12, atol=1e-16)
    assert lse == pytest.approx(math.log(9), rel=1e-14)
    np.testing.assert_allclose(p, np.full(9, 1 / 9), rtol=1e-14)
    # empty sequence
    o, lse, p = O.attend_unabsorbed(q_nope, q_pe, rows[:0], W_UK, W_UV, scale)
    assert np.all(o == 0) and lse == -math.inf and p.size == 0


@pytest.mark.parametrize("H,L", [(1, 1), (4, 8), (3, 33)])
def test_library_sdpa_on_expanded_keys(H, L):
    """torch's scaled_dot_product_attention in fp64 on CPU, fed explicitly
    expanded per-head keys [W^UK c_t | k_pe_t] (192) and values W^UV c_t
    (128), must equal the oracle."""
    rng = np.random.default_rng(100 + H * L)
    rows = _bf16(rng.normal(0, 1, (L, 576)))
    W_UK = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    W_UV = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    q_nope = rng.normal(0, 1, (H, 128))
    q_pe = rng.normal(0, 1, (H, 64))
    scale = 1 / math.sqrt(192)
    K = np.stack([np.concatenate([rows[:, :512] @ W_UK[h].T, rows[:, 512:]], axis=1) for h in range(H)])
    V = np.stack([rows[:, :512] @ W_UV[h].T for h in range(H)])
    Q = np.concatenate([q_nope, q_pe], axis=1)[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=scale)[0, :, 0].numpy()
    for h in range(H):
        o, _, p = O.attend_unabsorbed(q_nope[h], q_pe[h], rows, W_UK[h], W_UV[h], scale)
        np.testing.assert_allclose(o, ref[h], rtol=1e-10, atol=1e-14)
        assert abs(p.sum() - 1.0) <= 1e-12


def test_brute_force_scores_tiny():
    """<= 8 tokens: every score from plain Python loops over explicitly built keys."""
    rng = np.random.default_rng(3)
    q_nope, q_pe, rows, W_UK, W_UV = _rand_head(6, rng, std_w=0.1)
    scale = 0.25
    scores = []
    for t in range(6):
        key = [sum(W_UK[k, m] * rows[t, m] for m in range(512)) for k in range(128)] + list(rows[t, 512:])
        qv = list(q_nope) + list(q_pe)
        scores.append(scale * sum(a * b for a, b in zip(qv, key)))
    mx = max(scores)
    z = sum(math.exp(s - mx) for s in scores)
    _, lse, p = O.attend_unabsorbed(q_nope, q_pe, rows, W_UK, W_UV, scale)
    np.testing.assert_allclose(p, [math.exp(s - mx) / z for s in scores], rtol=1e-11)
    assert lse == pytest.approx(mx + math.log(z), rel=1e-12)


@pytest.mark.parametrize("bounds", [[1], [5, 6], [0, 0, 10], [3, 17, 50, 99]])
def test_split_combine_invariance(bounds):
    rng = np.random.default_rng(sum(bounds) + 1)
    q_nope, q_pe, rows, W_UK, W_UV = _rand_head(100, rng)
    o, lse, _ = O.attend_unabsorbed(q_nope, q_pe, rows, W_UK, W_UV, 0.1)
    o2, lse2 = O.attend_split(q_nope, q_pe, rows, W_UK, W_UV, 0.1, bounds)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-16)
    assert lse2 == pytest.approx(lse, rel=1e-13)
    # combine of nothing but empty parts
    oz, lz = O.combine_partials(np.zeros((3, 512)), np.full(3, -np.inf))
    assert np.all(oz == 0) and lz == -math.inf


@pytest.mark.parametrize("fmt", ["bf16", "int8", "fp8"])
def test_decode_page_permutation_invariance(fmt):
    rng = np.random.default_rng(11)
    B, H, P, maxp = 3, 2, 16, 6
    lens = [96, 1, 50]
    npg = B * maxp
    int8, fp8 = fmt == "int8", fmt == "fp8"
    if int8:
        cache = rng.integers(-128, 128, (npg, P, 576)).astype(np.int8)
        sz = np.stack([rng.uniform(0.01, 0.1, (npg, P)), rng.integers(-128, 128, (npg, P))], -1).astype(np.float32)
    elif fp8:
        cache = rng.choice(np.r_[0:0x7F, 0x80:0xFF], (npg, P, 576)).astype(np.uint8)
        sz = rng.uniform(0.001, 0.01, (npg, P)).astype(np.float32)
    else:
        cache = O.f64_to_bf16_bits(rng.normal(0, 1, (npg, P, 576)))
        sz = None
    table = np.arange(npg, dtype=np.int32).reshape(B, maxp)
    W_UK = _bf16(rng.normal(0, 0.02, (H, 128, 512)))
    W_UV = _bf16(rng.normal(0, 0.02, (H, 128, 512)))
    qn = _bf16(rng.normal(0, 1, (B, H, 128)))
    qp = _bf16(rng.normal(0, 1, (B, H, 64)))
    out1, lse1 = O.decode(qn, qp, cache, sz, table, lens, W_UK, W_UV, 0.07, P, int8, fp8=fp8)
    perm = rng.permutation(npg)          # physical page p moves to perm[p]
    cache2 = np.empty_like(cache)
    cache2[perm] = cache
    sz2 = None
    if int8 or fp8:
        sz2 = np.empty_like(sz)
        sz2[perm] = sz
    out2, lse2 = O.decode(qn, qp, cache2, sz2, perm[table].astype(np.int32), lens, W_UK, W_UV, 0.07, P, int8,
                          fp8=fp8)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)
    # absorbed cross-check over the whole batch
    out3, lse3 = O.decode(qn, qp, cache, sz, table, lens, W_UK, W_UV, 0.07, P, int8, absorbed=True, fp8=fp8)
    np.testing.assert_allclose(out3, out1, rtol=1e-11, atol=1e-15)


# ------------------------------------------------ planted-mistake checks ---- #

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check that the
    library pin above would have caught each of them."""
    rng = np.random.default_rng(5)
    H, L = 2, 5
    rows = _bf16(rng.normal(0, 1, (L, 576)))
    W_UK = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    W_UV = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    q_nope = rng.normal(0, 1, (H, 128))
    q_pe = rng.normal(0, 1, (H, 64))
    K = np.stack([np.concatenate([rows[:, :512] @ W_UK[h].T, rows[:, 512:]], axis=1) for h in range(H)])
    V = np.stack([rows[:, :512] @ W_UV[h].T for h in range(H)])
    Q = np.concatenate([q_nope, q_pe], axis=1)[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=0.2)[0, :, 0].numpy()

    def dropped_rope(qn, qp, r, wk, wv, sc):
        return O.attend_unabsorbed(qn, np.zeros_like(qp), r, wk, wv, sc)

    def swapped_weights(qn, qp, r, wk, wv, sc):
        return O.attend_unabsorbed(qn, qp, r, wv, wk, sc)

    def wrong_sign(qn, qp, r, wk, wv, sc):
        return O.attend_unabsorbed(qn, qp, r, wk, wv, -sc)

    for bad in (dropped_rope, swapped_weights, wrong_sign):
        o = np.stack([bad(q_nope[h], q_pe[h], rows, W_UK[h], W_UV[h], 0.2)[0] for h in range(H)])
        assert not np.allclose(o, ref, rtol=1e-6), bad.__name__


# ------------------------------------------------- multi-token decode ---- #

def _mt_inputs(B, T, H, P, lens, seed):
    rng = np.random.default_rng(seed)
    maxp = max(1, -(-max(lens) // P))
    npg = B * maxp
    cache = O.f64_to_bf16_bits(rng.normal(0, 1, (npg, P, 576)))
    table = rng.permutation(npg).astype(np.int32).reshape(B, maxp)
    W_UK = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    W_UV = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    qn = _bf16(rng.normal(0, 1, (B, T, H, 128)))
    qp = _bf16(rng.normal(0, 1, (B, T, H, 64)))
    return cache, table, W_UK, W_UV, qn, qp


def test_multi_token_single_query_is_decode():
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(3, 1, 2, 16, [40, 1, 17], 21)
    out, lse = O.decode_multi_token(qn, qp, cache, None, table, [40, 1, 17], W_UK, W_UV, 0.1, 16, False)
    out1, lse1 = O.decode(qn[:, 0], qp[:, 0], cache, None, table, [40, 1, 17], W_UK, W_UV, 0.1, 16, False)
    np.testing.assert_array_equal(out[:, 0], out1)
    np.testing.assert_array_equal(lse[:, 0], lse1)


@pytest.mark.parametrize("T,L", [(2, 2), (3, 9), (4, 33), (8, 20)])
def test_multi_token_library_causal_lower_right(T, L):
    """torch's scaled_dot_product_attention in fp64 with its own bottom-right
    aligned causal mask (queries are the last T positions of the keys), on
    explicitly expanded keys and values, must equal the oracle."""
    from torch.nn.attention.bias import causal_lower_right
    H, P = 2, 8
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, T, H, P, [L], 40 + T * L)
    scale = 1 / math.sqrt(192)
    rows = O.gather_rows(cache, None, table, 0, L, P, False)
    K = np.stack([np.concatenate([rows[:, :512] @ W_UK[h].T, rows[:, 512:]], axis=1) for h in range(H)])
    V = np.stack([rows[:, :512] @ W_UV[h].T for h in range(H)])
    Q = np.stack([np.concatenate([qn[0, :, h], qp[0, :, h]], axis=1) for h in range(H)])  # [H, T, 192]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=causal_lower_right(T, L), scale=scale)[0].numpy()                          # [H, T, 128]
    out, lse = O.decode_multi_token(qn, qp, cache, None, table, [L], W_UK, W_UV, scale, P, False)
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), ref, rtol=1e-10, atol=1e-14)
    assert np.all(np.isfinite(lse))


def test_multi_token_closed_forms():
    T, H, P = 4, 2, 8
    # T = L: the first query sees only token 0, so o = W^UV c_0 and lse = its score
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, T, H, P, [T], 7)
    out, lse = O.decode_multi_token(qn, qp, cache, None, table, [T], W_UK, W_UV, 0.3, P, False)
    rows = O.gather_rows(cache, None, table, 0, T, P, False)
    for h in range(H):
        np.testing.assert_allclose(out[0, 0, h], W_UV[h] @ rows[0, :512], rtol=1e-12, atol=1e-15)
        s0 = 0.3 * (qn[0, 0, h] @ (W_UK[h] @ rows[0, :512]) + qp[0, 0, h] @ rows[0, 512:])
        assert lse[0, 0, h] == pytest.approx(s0, rel=1e-12, abs=1e-14)
    # the last query sees the whole cache: single-token decode of the full sequence
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(2, T, H, P, [37, 12], 8)
    out, lse = O.decode_multi_token(qn, qp, cache, None, table, [37, 12], W_UK, W_UV, 0.3, P, False)
    full, lfull = O.decode(qn[:, -1], qp[:, -1], cache, None, table, [37, 12], W_UK, W_UV, 0.3, P, False)
    np.testing.assert_allclose(out[:, -1], full, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse[:, -1], lfull, rtol=1e-13)
    # fewer cached tokens than queries: the queries below position 0 see nothing
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, T, H, P, [2], 9)
    out, lse = O.decode_multi_token(qn, qp, cache, None, table, [2], W_UK, W_UV, 0.3, P, False)
    assert np.all(out[0, :2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.all(np.isfinite(lse[0, 2:]))


def test_multi_token_pins_catch_planted_mistakes(monkeypatch):
    """An off-by-one in the visible length, or the top-left (not bottom-right)
    alignment of the causal mask, planted in the oracle, must fail the
    library pin."""
    from torch.nn.attention.bias import causal_lower_right
    T, L, H, P = 3, 11, 1, 8
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, T, H, P, [L], 77)
    rows = O.gather_rows(cache, None, table, 0, L, P, False)
    K = np.concatenate([rows[:, :512] @ W_UK[0].T, rows[:, 512:]], axis=1)[None]
    V = (rows[:, :512] @ W_UV[0].T)[None]
    Q = np.concatenate([qn[0, :, 0], qp[0, :, 0]], axis=1)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=causal_lower_right(T, L), scale=0.2)[0, 0].numpy()
    good = O.attend_unabsorbed

    def off_by_one(qn_, qp_, r, wk, wv, sc):
        return good(qn_, qp_, r[:-1], wk, wv, sc)

    def top_left(qn_, qp_, r, wk, wv, sc):   # visible = t + 1 instead of L - T + t + 1
        return good(qn_, qp_, r[:r.shape[0] - (L - T)], wk, wv, sc)

    for bad in (off_by_one, top_left):
        monkeypatch.setattr(O.mla_oracle, "attend_unabsorbed", bad)
        out, _ = O.decode_multi_token(qn, qp, cache, None, table, [L], W_UK, W_UV, 0.2, P, False)
        monkeypatch.setattr(O.mla_oracle, "attend_unabsorbed", good)
        assert not np.allclose(out[0, :, 0], ref, rtol=1e-6), bad.__name__


# ---------------------------------------------------- sparse (top-k) decode ---- #

def test_sparse_all_positions_is_dense_decode():
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(2, 1, 2, 16, [40, 17], 101)
    idx = np.full((2, 40), -1)
    idx[0] = np.arange(40)
    idx[1, :17] = np.arange(17)
    out, lse = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [40, 17], idx, W_UK, W_UV, 0.1, 16, False)
    ref, lref = O.decode(qn[:, 0], qp[:, 0], cache, None, table, [40, 17], W_UK, W_UV, 0.1, 16, False)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, lref)


def test_sparse_library_masked_sdpa_and_order_invariance():
    """Attending to a subset of positions is SDPA over all positions with the
    unselected ones masked out (torch, fp64, boolean mask); the list order and
    padding entries do not matter."""
    H, L, P = 2, 50, 8
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, 1, H, P, [L], 102)
    rng = np.random.default_rng(5)
    chosen = rng.choice(L, 13, replace=False)
    idx = np.concatenate([chosen, [-1, -1, -1]])[None]
    out, lse = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], idx, W_UK, W_UV, 0.2, P, False)
    rows = O.gather_rows(cache, None, table, 0, L, P, False)
    K = np.stack([np.concatenate([rows[:, :512] @ W_UK[h].T, rows[:, 512:]], axis=1) for h in range(H)])
    V = np.stack([rows[:, :512] @ W_UV[h].T for h in range(H)])
    Q = np.concatenate([qn[0, 0], qp[0, 0]], axis=1)[:, None, :]
    mask = np.zeros((1, L), bool)
    mask[0, chosen] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=torch.from_numpy(mask), scale=0.2)[0, :, 0].numpy()
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-14)
    shuffled = np.concatenate([[-1], rng.permutation(chosen), [-1]])[None]
    out2, lse2 = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], shuffled, W_UK, W_UV, 0.2, P, False)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)
    # nothing selected: o = 0, lse = -inf
    o3, l3 = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], np.full((1, 4), -1), W_UK, W_UV, 0.2, P,
                             False)
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))


def test_sparse_out_of_range_entries_select_nothing():
    """An entry at or past the sequence's length, or below -1, is skipped like
    padding: the result equals that of the list without it, and a list made
    only of such entries gives o = 0, lse = -inf."""
    H, L, P = 2, 37, 8
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, 1, H, P, [L], 104)
    # the last page has slots 37..39 past the sequence's end, so a read past L would find data there
    idx = np.array([[3, 37, 17, -7, 36, 39, 1000, 0]])
    kept = np.array([[3, -1, 17, -1, 36, -1, -1, 0]])
    out, lse = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], idx, W_UK, W_UV, 0.2, P, False)
    ref, lref = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], kept, W_UK, W_UV, 0.2, P, False)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, lref)
    o2, l2 = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], np.array([[L, L + 5, -2]]), W_UK, W_UV,
                             0.2, P, False)
    assert np.all(o2 == 0) and np.all(np.isneginf(l2))


def test_sparse_pins_catch_planted_off_by_one(monkeypatch):
    """A gather that is off by one position, planted in the oracle, must fail
    the masked-SDPA pin."""
    H, L, P = 1, 30, 8
    cache, table, W_UK, W_UV, qn, qp = _mt_inputs(1, 1, H, P, [L], 103)
    chosen = np.array([3, 17, 9, 25])
    rows = O.gather_rows(cache, None, table, 0, L, P, False)
    K = np.concatenate([rows[:, :512] @ W_UK[0].T, rows[:, 512:]], axis=1)[None]
    V = (rows[:, :512] @ W_UV[0].T)[None]
    Q = np.concatenate([qn[0, 0], qp[0, 0]], axis=1)[:, None, :]
    mask = np.zeros((1, L), bool)
    mask[0, chosen] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=torch.from_numpy(mask), scale=0.2)[0, :, 0].numpy()
    good_gather = O.gather_rows

    def shifted(*a, **k):  # row i holds token i + 1
        r = good_gather(*a, **k)
        return np.concatenate([r[1:], r[:1]])

    monkeypatch.setattr(O.mla_oracle, "gather_rows", shifted)
    bad, _ = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], chosen[None], W_UK, W_UV, 0.2, P, False)
    monkeypatch.setattr(O.mla_oracle, "gather_rows", good_gather)
    good, _ = O.decode_sparse(qn[:, 0], qp[:, 0], cache, None, table, [L], chosen[None], W_UK, W_UV, 0.2, P, False)
    np.testing.assert_allclose(good[0], ref, rtol=1e-10, atol=1e-14)
    assert not np.allclose(bad[0], ref, rtol=1e-6)


# --------------------------------------------------------- chunked prefill ---- #

def _prefill_inputs(B, T, H, P, maxp, seed):
    rng = np.random.default_rng(seed)
    npg = B * maxp
    table = rng.permutation(npg).astype(np.int32).reshape(B, maxp)
    W_UK = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    W_UV = _bf16(rng.normal(0, 0.05, (H, 128, 512)))
    c_bits = O.f64_to_bf16_bits(rng.normal(0, 1, (B, T, 512)))
    k_bits = O.f64_to_bf16_bits(rng.normal(0, 1, (B, T, 64)))
    qn = _bf16(rng.normal(0, 1, (B, T, H, 128)))
    qp = _bf16(rng.normal(0, 1, (B, T, H, 64)))
    return table, W_UK, W_UV, c_bits, k_bits, qn, qp


def test_prefill_whole_prompt_is_causal_attention():
    """A prompt prefilled in one chunk from an empty cache is ordinary causal
    self-attention over the prompt: torch SDPA (fp64, is_causal) on
    explicitly expanded keys and values (RoPE off so that the stored RoPE key
    is the given one)."""
    B, T, H, P = 1, 21, 2, 16
    table, W_UK, W_UV, c_bits, k_bits, qn, qp = _prefill_inputs(B, T, H, P, 2, 3)
    cache = np.zeros((2, P, 576), np.uint16)
    out, lse = O.prefill_chunk(cache, None, table, [T], c_bits, k_bits, 0.0, qn, qp, W_UK, W_UV, 0.3, P, False)
    rows = np.concatenate([O.bf16_bits_to_f64(c_bits[0]), O.bf16_bits_to_f64(k_bits[0])], axis=1)
    for h in range(H):
        K = np.concatenate([rows[:, :512] @ W_UK[h].T, rows[:, 512:]], axis=1)
        V = rows[:, :512] @ W_UV[h].T
        Q = np.concatenate([qn[0, :, h], qp[0, :, h]], axis=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=0.3,
            is_causal=True)[0].numpy()
        np.testing.assert_allclose(out[0, :, h], ref, rtol=1e-10, atol=1e-13)


def test_prefill_in_chunks_matches_one_chunk_and_writes_the_cache():
    """Two chunks (T1 then T2) leave the cache and the second chunk's outputs
    exactly as one chunk of T1 + T2 leaves them for its last T2 tokens; the
    rows land at positions L - T .. L - 1 of each sequence."""
    B, T1, T2, H, P, maxp = 2, 9, 14, 2, 16, 4
    hist = [5, 30]
    table, W_UK, W_UV, c_bits, k_bits, qn, qp = _prefill_inputs(B, T1 + T2, H, P, maxp, 4)
    base = O.f64_to_bf16_bits(np.random.default_rng(9).normal(0, 1, (B * maxp, P, 576)))
    L = [h + T1 + T2 for h in hist]
    one = base.copy()
    o1, l1 = O.prefill_chunk(one, None, table, L, c_bits, k_bits, 1e4, qn, qp, W_UK, W_UV, 0.1, P, False)
    two = base.copy()
    O.prefill_chunk(two, None, table, [h + T1 for h in hist], c_bits[:, :T1], k_bits[:, :T1], 1e4,
                    qn[:, :T1], qp[:, :T1], W_UK, W_UV, 0.1, P, False)
    o2, l2 = O.prefill_chunk(two, None, table, L, c_bits[:, T1:], k_bits[:, T1:], 1e4, qn[:, T1:], qp[:, T1:],
                             W_UK, W_UV, 0.1, P, False)
    np.testing.assert_array_equal(one, two)
    np.testing.assert_allclose(o2, o1[:, T1:], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l2, l1[:, T1:], rtol=1e-12)
    for b in range(B):
        page, off = O.page_slot(table, b, hist[b], P)        # the chunk's first row
        np.testing.assert_array_equal(one[page, off, :512], c_bits[b, 0])
        page, off = O.page_slot(table, b, hist[b] - 1, P)    # the history before it is untouched
        np.testing.assert_array_equal(one[page, off], base[page, off])


def test_prefill_skips_tokens_without_a_page():
    """Tokens whose position is negative or whose page-table entry is -1 are
    not written anywhere (a -1 entry must not alias the last page)."""
    B, T, H, P = 2, 6, 1, 16
    table, W_UK, W_UV, c_bits, k_bits, qn, qp = _prefill_inputs(B, T, H, P, 1, 5)
    table = np.array([[0], [-1]], np.int32)     # sequence 1 has no page
    cache = np.zeros((1, P, 576), np.uint16)
    O.prefill_chunk(cache, None, table, [4, 10], c_bits, k_bits, 0.0, qn, qp, W_UK, W_UV, 0.1, P, False,
                    triples=[])
    np.testing.assert_array_equal(cache[0, :4, :512], c_bits[0, 2:])   # positions 0..3 = tokens 2..5
    assert not cache[0, 4:].any()


def test_fp8_and_prefill_pins_catch_planted_mistakes(monkeypatch):
    """Plausible mistakes planted in the oracle (on the CPU): each must fail
    the pin that guards it."""
    g = _fp8_golden()
    real_encode = O.e4m3_encode

    def truncating_encode(x):            # rounds toward zero instead of to nearest even
        v = np.asarray(x, dtype=np.float64)
        table = O.e4m3_value(np.arange(0x7F))
        a = np.minimum(np.abs(v), O.E4M3_MAX)
        code = np.clip(np.searchsorted(table, a, side="right") - 1, 0, 0x7E)
        return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)

    def ties_away(x):                    # ties away from zero instead of to even
        v = np.asarray(x, dtype=np.float64)
        c = real_encode(x).astype(np.int64)
        table = O.e4m3_value(np.arange(0x7F))
        a = np.minimum(np.abs(v), O.E4M3_MAX)
        mag = c & 0x7F
        up = np.minimum(mag + 1, 0x7E)
        tie = (np.abs(table[up] - a) == np.abs(a - table[mag])) & (up != mag)
        return np.where(tie & (table[up] > table[mag]), (c & 0x80) | up, c).astype(np.uint8)

    for bad in (truncating_encode, ties_away):
        wrong = [case for case in g["encode"]
                 if int(bad(np.array([case["value"]], np.float32))[0]) != case["code"]]
        assert wrong, bad.__name__

    # an exponent bias of 8 instead of 7 in the decoder halves every value
    def bias8(codes):
        return O.e4m3_value(codes) / 2
    wrong = [case for case in g["decode"] if case["value"] != "nan"
             and bias8(np.array([case["code"]], np.uint8))[0] != case["value"]]
    assert wrong

    # prefill: a query that also sees the next token (an off-by-one in the causal limit)
    B, T, H, P = 1, 9, 1, 16
    table, W_UK, W_UV, c_bits, k_bits, qn, qp = _prefill_inputs(B, T, H, P, 1, 6)
    cache = np.zeros((1, P, 576), np.uint16)
    good, _ = O.prefill_chunk(cache.copy(), None, table, [T], c_bits, k_bits, 0.0, qn, qp, W_UK, W_UV, 0.3, P,
                              False)
    real_multi = O.decode_multi_token

    def one_too_many(qn_, qp_, cache_, sz_, tab_, lens_, wk_, wv_, sc_, P_, int8_, triples=None, absorbed=False,
                     fp8=False):
        return real_multi(qn_, qp_, cache_, sz_, tab_, [int(l) + 1 for l in lens_], wk_, wv_, sc_, P_, int8_,
                          triples=triples, absorbed=absorbed, fp8=fp8)

    import oracle.mla_oracle as OM          # prefill_chunk looks the name up in its own module
    monkeypatch.setattr(OM, "decode_multi_token", one_too_many)
    cache2 = np.zeros((1, P, 576), np.uint16)
    bad, _ = O.prefill_chunk(cache2, None, table, [T], c_bits, k_bits, 0.0, qn, qp, W_UK, W_UV, 0.3, P, False)
    assert not np.allclose(bad, good, rtol=1e-6)
