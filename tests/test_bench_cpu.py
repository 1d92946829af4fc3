"""bench.py's host-side arithmetic, on CPU: the roofline units it reports."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import oracle as O  # noqa: E402


def test_bytes_per_token_match_the_cache_layout():
    # one layer: 576 values, plus the per-token quantisation parameters
    assert bench.BYTES_PER_TOKEN["bf16"] == O.latent_cache_bytes_per_token(1)
    assert bench.BYTES_PER_TOKEN["int8"] == O.latent_cache_bytes_per_token(1, elem_bytes=1, side_bytes_per_row=8)
    assert bench.BYTES_PER_TOKEN["fp8"] == O.latent_cache_bytes_per_token(1, elem_bytes=1, side_bytes_per_row=4)


def test_prefill_flops_closed_forms():
    per_key = 2 * 576 + 2 * 512
    # a whole prompt as one chunk: token t sees t + 1 keys, sum = T (T + 1) / 2
    assert bench.prefill_flops([10], 10, 3) == pytest.approx(3 * per_key * 55)
    # a chunk after a history of h: token t sees h + t + 1 keys
    h, T = 100, 8
    assert bench.prefill_flops([h + T], T, 1) == pytest.approx(per_key * (T * h + T * (T + 1) // 2))
    # a sequence shorter than the chunk: tokens at negative positions see nothing
    assert bench.prefill_flops([3], 5, 1) == pytest.approx(per_key * (1 + 2 + 3))
    # sequences add up
    assert bench.prefill_flops([10, 108], 8, 2) == pytest.approx(
        bench.prefill_flops([10], 8, 2) + bench.prefill_flops([108], 8, 2))


def test_whole_job_rate_units():
    # 32 tokens in 0.25 ms on one rank
    assert bench.whole_job_rate(32, 1, 0.25) == pytest.approx(128000.0)


@pytest.mark.parametrize("fmt,rows,kernel", [
    ("bf16", 16, "decode_pair.cu"), ("bf16", 32, "decode_pair.cu"), ("bf16", 64, "decode_pair.cu"),
    ("bf16", 48, "decode_hm.cu"), ("bf16", 96, "decode_hm.cu"), ("bf16", 128, "decode_hm.cu"),
    ("bf16", 8192, "decode_hm.cu"), ("int8", 16, "decode_tc.cu"), ("int8", 32, "decode_tc.cu"),
    ("int8", 64, "decode_hm.cu"), ("fp8", 48, "decode_hm.cu"), ("fp8", 128, "decode_hm.cu"),
])
def test_attention_kernel_follows_the_library_choice(fmt, rows, kernel):
    """The source the bench hashes for its DRAM-traffic record is the kernel
    the library runs for these rows (mla_api.cu, choose_attention: more than
    32 rows on the 128-row kernel, except bf16 rows of one or two 32-row
    groups; else bf16 on CTA pairs, 1-byte caches on single CTAs)."""
    assert os.path.basename(bench.attention_kernel(fmt, rows)[0]) == kernel


@pytest.mark.parametrize("auto", [76, 64, 148])
def test_minimum_chunks_round_up_to_whole_partitions_per_unit(auto):
    """A workload that asks for a minimum number of KV chunks per sequence
    runs with a multiple of the automatic split count (every attention unit
    then walks the same number of equal partitions), never fewer chunks than
    asked, and the smallest such multiple."""
    from mla_decode_attention_paged_gb300 import workloads as W
    w = W.WORKLOADS["ctx1m"]
    s = W.num_splits_for(w, auto)
    assert s % auto == 0
    assert s >= w.min_splits_per_seq * w.batch
    assert s - auto < max(auto, w.min_splits_per_seq * w.batch)
    # workloads without a minimum keep the automatic count (0 = automatic)
    assert W.num_splits_for(W.WORKLOADS["v2lite"], auto) == 0
