"""The decode step inside a CUDA graph: cache append + mla_decode (and
mla_decode_multi) captured once on a side stream and replayed must give
bit-identical results to eager calls.  Checks that the library does nothing
during a call that stream capture forbids (no allocation, no host
synchronisation, no device-wide calls), including its programmatic
dependent launches, which the graph keeps as programmatic edges."""
import pytest
import torch

import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(T, seed):
    g = W.generator(seed)
    B, H, P = 4, 16, 64
    seq_lens = torch.tensor([700, 129, 2000, 64], dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, True, g, spare_pages=2)
    qshape = (B, H) if T == 1 else (B, T, H)
    x = dict(cache=W.draw_bf16((npg, P, 576), 1.0, g).cuda(), table=table.cuda(), lens=seq_lens.cuda(),
             W_UK=W.draw_bf16((H, 128, 512), 0.02, g).cuda(), W_UV=W.draw_bf16((H, 128, 512), 0.02, g).cuda(),
             q_nope=W.draw_bf16(qshape + (128,), 1.0, g).cuda(), q_pe=W.draw_bf16(qshape + (64,), 1.0, g).cuda(),
             new_c=W.draw_bf16((B * T, 512), 1.0, g).cuda(), new_k=W.draw_bf16((B * T, 64), 1.0, g).cuda())
    x["ids"] = torch.arange(B, dtype=torch.int32, device="cuda").repeat_interleave(T)
    x["pos"] = (x["lens"].repeat_interleave(T) - T + torch.arange(T, dtype=torch.int32, device="cuda").repeat(B)).int()
    x["out"] = torch.empty(qshape + (128,), dtype=torch.bfloat16, device="cuda")
    x["lse"] = torch.empty(qshape, dtype=torch.float32, device="cuda")
    x["ws"] = torch.empty(mla.decode_multi_workspace_size(mla.dims(H, P), B, T, 0), dtype=torch.uint8, device="cuda")
    return mla.dims(H, P), x


def _step(d, x, T, stream):
    mla.cache_append(d, x["cache"], None, x["table"], x["ids"], x["pos"], x["new_c"], x["new_k"], 10000.0,
                     stream=stream)
    fn = mla.decode if T == 1 else mla.decode_multi
    fn(d, x["q_nope"], x["q_pe"], x["cache"], None, x["table"], x["lens"], x["W_UK"], x["W_UV"], 0.0721,
       workspace=x["ws"], out=x["out"], lse_out=x["lse"], stream=stream)


@pytest.mark.parametrize("T", [1, 3])
def test_graph_replay_matches_eager(cuda_lib, T):
    d, x = _inputs(T, 5 + T)
    _step(d, x, T, None)  # first calls: one-time attribute setup happens outside the capture
    torch.cuda.synchronize()
    ref_out, ref_lse = x["out"].clone(), x["lse"].clone()
    x["out"].zero_()
    x["lse"].zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        _step(d, x, T, s)
    for _ in range(3):
        x["out"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(x["out"], ref_out) and torch.equal(x["lse"], ref_lse)
    assert mla.read_device_status(x["ws"]) == mla.MLA_OK


def _capture_and_check(step, outs, ws):
    """Run ``step`` eagerly once, capture it in a graph on a side stream, and
    check three replays against the eager results."""
    step(None)
    torch.cuda.synchronize()
    refs = [o.clone() for o in outs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for _ in range(3):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            assert torch.equal(o, r)
    assert mla.read_device_status(ws) == mla.MLA_OK


def test_graph_fp8_decode_step(cuda_lib):
    """An FP8 cache: the quantising append and the 1-byte decode path in a graph."""
    g = W.generator(21)
    B, H, P = 3, 16, 64
    lens = torch.tensor([900, 64, 1300], dtype=torch.int32)
    table, npg = W.draw_page_table(lens, P, True, g)
    d = mla.dims(H, P, fp8=True)
    codes, sc = W.draw_fp8_cache(npg, P, g)
    x = dict(cache=codes.cuda(), sc=sc.cuda(), table=table.cuda(), lens=lens.cuda(),
             W_UK=W.draw_bf16((H, 128, 512), 0.02, g).cuda(), W_UV=W.draw_bf16((H, 128, 512), 0.02, g).cuda(),
             q_nope=W.draw_bf16((B, H, 128), 1.0, g).cuda(), q_pe=W.draw_bf16((B, H, 64), 1.0, g).cuda(),
             new_c=W.draw_bf16((B, 512), 1.0, g).cuda(), new_k=W.draw_bf16((B, 64), 1.0, g).cuda())
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    pos = (x["lens"] - 1).int()
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(mla.decode_workspace_size(d, B, 0), dtype=torch.uint8, device="cuda")

    def step(stream):
        mla.cache_append(d, x["cache"], x["sc"], x["table"], ids, pos, x["new_c"], x["new_k"], 10000.0, stream=stream)
        mla.decode(d, x["q_nope"], x["q_pe"], x["cache"], x["sc"], x["table"], x["lens"], x["W_UK"], x["W_UV"],
                   0.0721, workspace=ws, out=out, lse_out=lse, stream=stream)

    _capture_and_check(step, [out, lse], ws)


def test_graph_prefill_chunk(cuda_lib):
    """A prefill chunk (append by position + causal attention) in a graph."""
    g = W.generator(22)
    B, H, P, T = 2, 16, 64, 40
    lens = torch.tensor([300, 41], dtype=torch.int32)
    table, npg = W.draw_page_table(lens, P, True, g)
    d = mla.dims(H, P)
    x = dict(cache=W.draw_bf16((npg, P, 576), 1.0, g).cuda(), table=table.cuda(), lens=lens.cuda(),
             W_UK=W.draw_bf16((H, 128, 512), 0.02, g).cuda(), W_UV=W.draw_bf16((H, 128, 512), 0.02, g).cuda(),
             q_nope=W.draw_bf16((B, T, H, 128), 1.0, g).cuda(), q_pe=W.draw_bf16((B, T, H, 64), 1.0, g).cuda(),
             c_kv=W.draw_bf16((B, T, 512), 1.0, g).cuda(), k_pe=W.draw_bf16((B, T, 64), 1.0, g).cuda())
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, T, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(mla.prefill_workspace_size(d, B, T, 0), dtype=torch.uint8, device="cuda")

    def step(stream):
        mla.prefill(d, x["cache"], None, x["table"], x["lens"], x["c_kv"], x["k_pe"], x["q_nope"], x["q_pe"],
                    x["W_UK"], x["W_UV"], 0.0721, rope_theta=10000.0, workspace=ws, out=out, lse_out=lse,
                    stream=stream)

    _capture_and_check(step, [out, lse], ws)
