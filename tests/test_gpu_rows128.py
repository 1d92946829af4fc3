"""GPU parity of the 128-row attention kernel (decode_hm.cu) against the
fp64 oracle, through the C ABI.

Every call whose rows per sequence (heads, or q_len x heads) are a multiple
of 128 runs on it, for all three cache formats.  The kernel takes the plan's
128-token tiles in halves of 64 tokens, so the lengths here sit on and
around both boundaries (63, 64, 65, 127, 128, 129, ...), for every page
size (16 and 32: several pages per half; 64: one; 128: half a page), with
split counts from one partition to one per half-tile, two row groups (256
heads), multi-token rows (16 x 8, 32 x 4, 64 x 2), and the degenerate cases
(empty sequence, one token, NaN patterns past a sequence's end).  Row counts
above 32 that are not a multiple of 128 run here too, the last group padded."""
import pytest
import torch

import mla_decode_attention_paged_gb300 as mla
from harness import gpu_decode
from test_gpu_multi_token import _check as mt_check, _mt
from test_gpu_parity import _run_small, _small

pytestmark = pytest.mark.gpu

BOUNDARY_LENS = (0, 1, 63, 64, 65, 127, 128, 129, 191, 192, 193, 700)


@pytest.mark.parametrize("fmt", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_rows128_half_tile_boundaries_and_page_sizes(cuda_lib, fmt, P):
    w, inp = _small(heads=128, P=P, lens=BOUNDARY_LENS, int8=fmt == "int8", fp8=fmt == "fp8", seed=128 + P)
    (_, _), out, lse = _run_small(w, inp)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
@pytest.mark.parametrize("splits", [1, 3, 64, 500])
def test_rows128_split_counts(cuda_lib, fmt, splits):
    # 500 partitions over these 2,400 tokens: most segments are one half-tile
    _run_small(*_small(heads=128, lens=(1000, 5, 1300, 65), int8=fmt == "int8", seed=11 + splits),
               num_splits=splits)


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
def test_rows128_two_row_groups(cuda_lib, fmt):
    _run_small(*_small(heads=256, lens=(700, 1, 130), fp8=fmt == "fp8", seed=257))


@pytest.mark.parametrize("heads,T,fmt", [(16, 8, "bf16"), (32, 4, "fp8"), (64, 2, "int8"), (128, 2, "bf16")])
def test_rows128_multi_token_rows(cuda_lib, heads, T, fmt):
    # rows v = t * heads + h: one group holds several query tokens, causal among themselves
    mt_check(_mt(heads=heads, T=T, lens=(1, 5, 64, 129, 700), int8=fmt == "int8", fp8=fmt == "fp8",
                 seed=900 + heads + T))


@pytest.mark.parametrize("heads,T,fmt", [(16, 3, "bf16"), (16, 4, "int8"), (16, 5, "fp8"), (16, 6, "bf16"),
                                          (32, 3, "int8"), (32, 5, "bf16"), (16, 7, "fp8")])
def test_rows128_padded_groups_multi_token(cuda_lib, heads, T, fmt):
    # 48 to 160 rows: one or two groups, the last padded past the sequence's
    # rows (those rows run with a zero latent query and write nothing)
    mt_check(_mt(heads=heads, T=T, lens=(1, 5, 64, 129, 700), int8=fmt == "int8", fp8=fmt == "fp8",
                 seed=1300 + heads + T), num_splits=7)


@pytest.mark.parametrize("heads,fmt", [(64, "int8"), (96, "bf16"), (96, "fp8"), (160, "bf16")])
def test_rows128_padded_groups_single_token(cuda_lib, heads, fmt):
    _run_small(*_small(heads=heads, lens=(700, 1, 130, 64), int8=fmt == "int8", fp8=fmt == "fp8", seed=400 + heads),
               num_splits=5)


def test_rows128_multi_token_invisible_segments(cuda_lib):
    # many splits: segments made only of the last new tokens, which the
    # earlier query rows of the group cannot see
    mt_check(_mt(heads=16, T=8, lens=(129, 257, 385, 1000), seed=961), num_splits=1000)


@pytest.mark.parametrize("fmt", ["bf16", "int8", "fp8"])
def test_rows128_nan_patterns_past_the_sequence_end(cuda_lib, fmt):
    w, inp = _small(heads=128, lens=(200, 1030, 77, 65), int8=fmt == "int8", fp8=fmt == "fp8", seed=13)
    P = w.page_size
    for b, L in enumerate(inp["seq_lens"].tolist()):
        if L % P:
            page = int(inp["block_table"][b, (L - 1) // P])
            if fmt == "bf16":
                inp["cache"].view(torch.int16)[page, L % P:] = 0x7FC0
            else:
                inp["cache_i8"].view(torch.uint8)[page, L % P:, 0::2] = 0x7F
                inp["cache_i8"].view(torch.uint8)[page, L % P:, 1::2] = 0xFF
                inp["sz"].view(torch.int32)[page, L % P:] = 0x7FC00000  # NaN scales too
    (_, _), out, lse = _run_small(w, inp)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_rows128_bit_identical_run_to_run_and_under_a_shuffled_table(cuda_lib):
    w, inp = _small(heads=128, lens=(900, 65, 1), seed=21)
    cache = inp["cache"].cuda()
    o1, l1 = gpu_decode(inp, w, cache, None, num_splits=9)
    o2, l2 = gpu_decode(inp, w, cache, None, num_splits=9)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # the same rows on other physical pages
    npg = cache.shape[0]
    perm = torch.randperm(npg, generator=torch.Generator().manual_seed(5))
    moved = torch.empty_like(cache)
    moved[perm.cuda()] = cache
    table = inp["block_table"].clone()
    valid = table >= 0
    table[valid] = perm[table[valid].long()].to(torch.int32)
    o3, l3 = gpu_decode(inp, w, moved, None, num_splits=9, block_table=table)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_rows128_is_the_kernel_that_runs(cuda_lib):
    """More than 32 rows take the 128-row kernel's automatic split count (one
    partition per resident pair and row group): 96 bf16 rows or 64 INT8 rows
    make one group (padded below 128), 256 rows two, each with half the
    pairs; 64 bf16 rows stay on the pair kernel as two 32-row groups."""
    one = mla.auto_num_splits(mla.dims(128, 64), 4)
    assert mla.auto_num_splits(mla.dims(96, 64), 4) == one
    assert mla.auto_num_splits(mla.dims(64, 64, int8=True), 4) == one
    assert mla.auto_num_splits(mla.dims(256, 64), 4) == one // 2
    # bf16: 64 rows stay two 32-row groups of the pair kernel, half the pairs each
    assert mla.auto_num_splits(mla.dims(64, 64), 4) == one // 2
