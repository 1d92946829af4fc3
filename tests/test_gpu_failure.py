"""Device-side failure detection, without a GPU fault.

Every wait in the attention kernels is bounded.  The test hook
mla_test_inject_wait_timeout makes each CTA's first cache-page barrier
expect 16 bytes more than its copies deliver, so that wait cannot complete:
the kernel must record MLA_ERR_DEVICE_TIMEOUT in the workspace status word,
release its tensor memory and return, and the context must stay usable (the
next decode in the same process is correct).  Nothing faults, traps or
hangs: the wait ends at its ~2 s limit."""
import numpy as np
import pytest
import torch

import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(fmt: str, heads=16, lens=(700, 129), P=64, seed=31):
    g = W.generator(seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, True, g)
    x = dict(seq_lens=seq_lens.cuda(), table=table.cuda(), W_UK=W.draw_bf16((heads, 128, 512), 0.02, g).cuda(),
             W_UV=W.draw_bf16((heads, 128, 512), 0.02, g).cuda(),
             q_nope=W.draw_bf16((len(lens), heads, 128), 1.0, g).cuda(),
             q_pe=W.draw_bf16((len(lens), heads, 64), 1.0, g).cuda(), sz=None)
    if fmt != "bf16":
        codes, sz = W.draw_int8_cache(npg, P, g) if fmt == "int8" else W.draw_fp8_cache(npg, P, g)
        x["cache"], x["sz"] = codes.cuda(), sz.cuda()
    else:
        x["cache"] = W.draw_bf16((npg, P, 576), 1.0, g).cuda()
    return mla.dims(heads, P, int8=fmt == "int8", fp8=fmt == "fp8"), x


def _decode(d, x, ws):
    out, lse = mla.decode(d, x["q_nope"], x["q_pe"], x["cache"], x["sz"], x["table"], x["seq_lens"], x["W_UK"],
                          x["W_UV"], 1.0 / np.sqrt(192.0), num_splits=8, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("heads", [16, 128], ids=["16-heads", "128-rows"])
@pytest.mark.parametrize("fmt", ["bf16", "int8", "fp8"], ids=["bf16-pairs", "int8", "fp8"])
def test_unsatisfiable_wait_reports_timeout_and_context_survives(cuda_lib, fmt, heads):
    d, x = _inputs(fmt, heads=heads)
    ws = torch.empty(mla.decode_workspace_size(d, 2, 8), dtype=torch.uint8, device="cuda")
    ref_out, ref_lse = _decode(d, x, ws)
    assert mla.read_device_status(ws) == mla.MLA_OK
    try:
        mla.test_inject_wait_timeout(True)
        _decode(d, x, ws)
        assert mla.read_device_status(ws) == mla.MLA_ERR_DEVICE_TIMEOUT
    finally:
        mla.test_inject_wait_timeout(False)
    out, lse = _decode(d, x, ws)
    assert mla.read_device_status(ws) == mla.MLA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
