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
