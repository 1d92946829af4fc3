"""Parity at the full sizes of the benchmark workloads, in the launch
configuration bench.py times.  The oracle cannot evaluate every output at
these sizes, so each test checks a seeded sample of sequences: the
un-absorbed oracle on some heads of each sampled sequence, and the absorbed
fp64 form (pinned to the un-absorbed one in test_oracle.py) on all heads."""
import numpy as np
import pytest
import torch

import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import assert_parity, dims_of, gpu_cache, gpu_decode, oracle_cache, oracle_decode

pytestmark = pytest.mark.gpu

# workload key -> (sampled sequences rule, un-absorbed heads per sampled sequence)
SAMPLES = {
    "tiny": (None, None),
    "v2lite": ([0, 31], None),
    "ctx1m": ([1], [0, 15]),
    "ragged": ("longest+3", [0, 37, 64, 127]),
    "int8": ([0, 57, 127], [0, 31, 96, 127]),
    "fp8_v2lite": ([0, 31], [0, 15]),
}


def _sample_seqs(rule, seq_lens, batch):
    if rule is None:
        return list(range(batch))
    if rule == "longest+3":
        lens = seq_lens.cpu().numpy()
        g = np.random.default_rng(2024)
        others = g.choice([b for b in range(batch) if b != int(lens.argmax())], 3, replace=False)
        return sorted({int(lens.argmax()), *map(int, others)})
    return rule


@pytest.mark.parametrize("key", ["tiny", "v2lite", "ctx1m", "ragged", "int8", "fp8_v2lite"])
def test_full_size_workload(cuda_lib, key):
    w = W.WORKLOADS[key]
    inp = W.make_decode_inputs(w, device="cuda")
    cache, sz = gpu_cache(inp, w)
    splits = W.num_splits_for(w, mla.auto_num_splits(dims_of(w), w.batch))
    out, lse = gpu_decode(inp, w, cache, sz, num_splits=splits)
    del cache, sz
    torch.cuda.empty_cache()
    rule, heads = SAMPLES[key]
    seqs = _sample_seqs(rule, inp["seq_lens"], w.batch)
    oc = oracle_cache(inp, w, seqs)
    all_pairs = [(b, h) for b in seqs for h in range(w.heads)]
    un_pairs = all_pairs if heads is None else [(b, h) for b in seqs for h in heads]
    ref_o, ref_l = oracle_decode(inp, w, un_pairs, cache_override=oc)
    assert_parity(out, lse, ref_o, ref_l, un_pairs, w.name + " (un-absorbed oracle)")
    if heads is not None:
        ref_o, ref_l = oracle_decode(inp, w, all_pairs, absorbed=True, cache_override=oc)
        assert_parity(out, lse, ref_o, ref_l, all_pairs, w.name + " (absorbed oracle, all heads)")


@pytest.mark.parametrize("key,seq", [("v2lite_mtp2", 9), ("v2lite_mtp4", 22)])
def test_full_size_multi_token(cuda_lib, key, seq):
    """Multi-token decode at the V2-Lite size (32 x 32,768 tokens, q_len 2 or
    4), in bench.py's configuration: every (token, head) of one sampled
    sequence against the un-absorbed oracle."""
    import oracle as O
    from harness import f64
    w = W.WORKLOADS[key]
    inp = W.make_decode_inputs(w, device="cuda")
    d = dims_of(w)
    T, H = w.q_len, w.heads
    d_rows = mla.dims(H * T, w.page_size)
    splits = mla.auto_num_splits(d_rows, w.batch)
    out, lse = mla.decode_multi(d, inp["q_nope"], inp["q_pe"], inp["cache"], None, inp["block_table"],
                                inp["seq_lens"], inp["W_UK"], inp["W_UV"], inp["scale"], num_splits=splits)
    torch.cuda.synchronize()
    cache, sz, table = oracle_cache(inp, w, [seq])
    ref_o, ref_l = O.decode_multi_token(f64(inp["q_nope"]), f64(inp["q_pe"]), cache, sz, table,
                                        inp["seq_lens"].cpu().numpy(), f64(inp["W_UK"]), f64(inp["W_UV"]),
                                        inp["scale"], w.page_size, False,
                                        triples=[(seq, t, h) for t in range(T) for h in range(H)])
    B = w.batch
    pairs = [(seq, v) for v in range(T * H)]
    assert_parity(out.reshape(B, T * H, -1), lse.reshape(B, T * H), ref_o.reshape(B, T * H, -1),
                  ref_l.reshape(B, T * H), pairs, w.name)


def test_full_size_sparse_topk(cuda_lib):
    """Sparse decode at the V2-Lite size with DeepSeek Sparse Attention's
    top-2048 selection per sequence, in bench.py's configuration: every head
    of two sampled sequences against the un-absorbed oracle."""
    import oracle as O
    from harness import f64
    w = W.WORKLOADS["v2lite_topk2048"]
    inp = W.make_decode_inputs(w, device="cuda")
    d = dims_of(w)
    out, lse = mla.decode_sparse(d, inp["q_nope"], inp["q_pe"], inp["cache"], None, inp["block_table"],
                                 inp["seq_lens"], inp["token_indices"], inp["W_UK"], inp["W_UV"], inp["scale"],
                                 num_splits=mla.auto_num_splits(d, w.batch))
    torch.cuda.synchronize()
    seqs = [4, 27]
    cache, sz, table = oracle_cache(inp, w, seqs)
    pairs = [(b, h) for b in seqs for h in range(w.heads)]
    ref_o, ref_l = O.decode_sparse(f64(inp["q_nope"]), f64(inp["q_pe"]), cache, sz, table,
                                   inp["seq_lens"].cpu().numpy(), inp["token_indices"].cpu().numpy(),
                                   f64(inp["W_UK"]), f64(inp["W_UV"]), inp["scale"], w.page_size, False, pairs=pairs)
    assert_parity(out, lse, ref_o, ref_l, pairs, w.name)


def test_full_size_prefill_chunk(cuda_lib):
    """Chunked prefill at the bench's size (4 sequences, a 512-token chunk
    after 8,192 cached tokens, 16 heads), in bench.py's configuration: the
    chunk's first, middle and last tokens of two sampled sequences, every
    head, against the un-absorbed oracle, which appends the chunk to its own
    copy of the history first."""
    import oracle as O
    from harness import f64
    w = W.WORKLOADS["v2lite_prefill512"]
    inp = W.make_decode_inputs(w, device="cuda")
    d = dims_of(w)
    T, H = w.chunk, w.heads
    splits = mla.auto_num_splits(mla.dims(H * T, w.page_size), w.batch)
    seqs = [0, 3]
    cache, sz, table = oracle_cache(inp, w, seqs)      # the history as drawn, before the GPU writes the chunk
    gpu_cache = inp["cache"].cuda()
    out, lse = mla.prefill(d, gpu_cache, None, inp["block_table"], inp["seq_lens"], inp["chunk_c_kv"],
                           inp["chunk_k_pe"], inp["q_nope"], inp["q_pe"], inp["W_UK"], inp["W_UV"], inp["scale"],
                           rope_theta=w.rope_theta, num_splits=splits)
    torch.cuda.synchronize()
    triples = [(b, t, h) for b in seqs for t in (0, T // 2, T - 1) for h in range(H)]
    ref_o, ref_l = O.prefill_chunk(cache, sz, table, inp["seq_lens"].cpu().numpy(),
                                   W.bf16_to_bits(inp["chunk_c_kv"]), W.bf16_to_bits(inp["chunk_k_pe"]),
                                   w.rope_theta, f64(inp["q_nope"]), f64(inp["q_pe"]), f64(inp["W_UK"]),
                                   f64(inp["W_UV"]), inp["scale"], w.page_size, False, triples=triples)
    B = w.batch
    pairs = [(b, t * H + h) for b, t, h in triples]
    assert_parity(out.reshape(B, T * H, -1), lse.reshape(B, T * H), ref_o.reshape(B, T * H, -1),
                  ref_l.reshape(B, T * H), pairs, w.name)
