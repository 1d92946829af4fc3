"""Seeded randomized parity: each case draws its own page size, head count,
batch, ragged lengths (with 0, 1 and tile-boundary lengths mixed in), split
count, cache type and query-token count (or a sparse selection), and checks
the library against the fp64 oracle through the C ABI.  Complements the
hand-picked cases with combinations nobody wrote down; a second family
draws row counts (heads x tokens) around the 128-row kernel's groups."""
import numpy as np
import pytest
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import assert_parity, f64

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([16, 32, 64, 128]))
    H = int(rng.choice([16, 32, 64]))
    B = int(rng.integers(1, 6))
    special = [0, 1, 127, 128, 129, 255, 256]
    lens = [int(rng.choice(special)) if rng.random() < 0.3 else int(rng.integers(1, 1500)) for _ in range(B)]
    r = rng.random()
    fmt = "int8" if r < 0.3 else "fp8" if r < 0.45 else "bf16"
    mode = rng.choice(["dense", "multi", "sparse"], p=[0.5, 0.3, 0.2])
    T = int(rng.integers(2, 5)) if mode == "multi" else 1
    splits = int(rng.choice([0, 1, 3, 17, 200]))
    return dict(P=P, H=H, lens=lens, fmt=fmt, mode=str(mode), T=T, splits=splits)


def _wide_case(seed):
    """Row counts around the 128-row kernel's groups: 32-96 heads with 1-5
    query tokens (32 to 480 rows: single and several groups, padded or not),
    shorter sequences to keep the oracle quick."""
    rng = np.random.default_rng(7000 + seed)
    P = int(rng.choice([16, 32, 64, 128]))
    H = int(rng.choice([32, 64, 96]))
    B = int(rng.integers(1, 4))
    special = [0, 1, 63, 64, 65, 127, 128, 129]
    lens = [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(1, 700)) for _ in range(B)]
    r = rng.random()
    fmt = "int8" if r < 0.3 else "fp8" if r < 0.55 else "bf16"
    T = int(rng.integers(1, 6))
    mode = "multi" if T > 1 else str(rng.choice(["dense", "sparse"], p=[0.7, 0.3]))
    splits = int(rng.choice([0, 1, 5, 40]))
    return dict(P=P, H=H, lens=lens, fmt=fmt, mode=mode, T=T, splits=splits)


@pytest.mark.parametrize("seed", range(16))
def test_random_configuration(cuda_lib, seed):
    _run_case(_case(seed), seed)


@pytest.mark.parametrize("seed", range(32))
def test_random_row_groups(cuda_lib, seed):
    _run_case(_wide_case(seed), 100 + seed)


def _run_case(c, seed):
    P, H, T = c["P"], c["H"], c["T"]
    int8, fp8 = c["fmt"] == "int8", c["fmt"] == "fp8"
    g = W.generator(5000 + seed)
    seq_lens = torch.tensor(c["lens"], dtype=torch.int32)
    B = len(c["lens"])
    table, npg = W.draw_page_table(seq_lens, P, True, g, spare_pages=2)
    if int8 or fp8:
        codes, sz = W.draw_int8_cache(npg, P, g) if int8 else W.draw_fp8_cache(npg, P, g)
        cache_d, sz_d, cache_o, sz_o = codes.cuda(), sz.cuda(), codes.numpy(), sz.numpy()
    else:
        cache = W.draw_bf16((npg, P, 576), 1.0, g)
        cache_d, sz_d, cache_o, sz_o = cache.cuda(), None, W.bf16_to_bits(cache), None
    W_UK = W.draw_bf16((H, 128, 512), 0.02, g)
    W_UV = W.draw_bf16((H, 128, 512), 0.02, g)
    qshape = (B, H) if T == 1 else (B, T, H)
    q_nope = W.draw_bf16(qshape + (128,), 1.0, g)
    q_pe = W.draw_bf16(qshape + (64,), 1.0, g)
    scale = 1.0 / np.sqrt(192.0)
    d = mla.dims(H, P, int8=int8, fp8=fp8)
    args = (d, q_nope.cuda(), q_pe.cuda(), cache_d, sz_d, table.cuda(), seq_lens.cuda())
    wts = (W_UK.cuda(), W_UV.cuda(), scale)
    oargs = (f64(q_nope), f64(q_pe), cache_o, sz_o, table.numpy(), seq_lens.numpy())
    if c["mode"] == "sparse":
        idx = W.draw_token_indices(seq_lens, int(max(1, max(c["lens"]) // 3)), 0.7, g)
        out, lse = mla.decode_sparse(*args, idx.cuda(), *wts, num_splits=c["splits"])
        ref_o, ref_l = O.decode_sparse(*oargs, idx.numpy(), f64(W_UK), f64(W_UV), scale, P, int8, fp8=fp8)
    elif c["mode"] == "multi":
        out, lse = mla.decode_multi(*args, *wts, num_splits=c["splits"])
        ref_o, ref_l = O.decode_multi_token(*oargs, f64(W_UK), f64(W_UV), scale, P, int8, fp8=fp8)
        out, lse = out.reshape(B, T * H, -1), lse.reshape(B, T * H)
        ref_o, ref_l = ref_o.reshape(B, T * H, -1), ref_l.reshape(B, T * H)
    else:
        out, lse = mla.decode(*args, *wts, num_splits=c["splits"])
        ref_o, ref_l = O.decode(*oargs, f64(W_UK), f64(W_UV), scale, P, int8, fp8=fp8)
    torch.cuda.synchronize()
    pairs = [(b, v) for b in range(B) for v in range(out.shape[1])]
    assert_parity(out, lse, ref_o, ref_l, pairs, str(c))
