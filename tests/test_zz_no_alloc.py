"""mla_decode_no_alloc: the decode entry point for callers that cannot
allocate device memory (for example a serving loop that must not call
cudaMalloc on its decode path, or a C host whose device memory is budgeted up
front).  It runs on the library's fixed scratch array instead of a caller
workspace.  These checks call it through the C ABI twice in a row and compare
each result with mla_decode's, and check that a shape needing more scratch
than the array holds is refused.  Kept in a file collected last."""
import numpy as np
import pytest
import torch

import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import ABS_TOL, LSE_ABS_TOL, REL_TOL

pytestmark = pytest.mark.gpu


def _inputs(heads=16, lens=(3000, 129, 4096, 1), P=64, seed=21):
    g = W.generator(seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, True, g)
    d = dict(seq_lens=seq_lens.cuda(), table=table.cuda(), num_pages=npg,
             cache=W.draw_bf16((npg, P, 576), 1.0, g).cuda(), W_UK=W.draw_bf16((heads, 128, 512), 0.02, g).cuda(),
             W_UV=W.draw_bf16((heads, 128, 512), 0.02, g).cuda(),
             q_nope=W.draw_bf16((len(lens), heads, 128), 1.0, g).cuda(),
             q_pe=W.draw_bf16((len(lens), heads, 64), 1.0, g).cuda())
    return mla.dims(heads, P), d


def _close(a_out, a_lse, b_out, b_lse):
    a, b = a_out.float().cpu().numpy(), b_out.float().cpu().numpy()
    err = np.abs(a - b)
    assert err.max() <= ABS_TOL
    row_max = np.abs(b).max(axis=-1)
    assert np.all(err.max(axis=-1) <= REL_TOL * np.maximum(row_max, 1e-30))
    assert np.abs(a_lse.cpu().numpy() - b_lse.cpu().numpy()).max() <= LSE_ABS_TOL


def test_no_alloc_matches_decode_on_two_calls(cuda_lib):
    d, x = _inputs()
    scale = 1.0 / np.sqrt(192.0)
    ref_out, ref_lse = mla.decode(d, x["q_nope"], x["q_pe"], x["cache"], None, x["table"], x["seq_lens"], x["W_UK"],
                                  x["W_UV"], scale, num_splits=40)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for _ in range(2):
        lse = torch.empty_like(ref_lse)
        out, _ = mla.decode_no_alloc(d, x["q_nope"], x["q_pe"], x["cache"], None, x["table"], x["seq_lens"],
                                     x["W_UK"], x["W_UV"], scale, num_splits=40, lse_out=lse, device_status=status)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)
        assert int(status.item()) == mla.MLA_OK


def test_no_alloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    d, x = _inputs()
    batch = 4096  # (splits + batch) * H * 2 KB of partials alone exceeds the fixed array
    assert mla.decode_workspace_size(d, batch, 152) > mla.NO_ALLOC_WORKSPACE_BYTES
    q = torch.zeros((batch, 16, 128), dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros((batch, 16, 64), dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(batch, dtype=torch.int32, device="cuda")
    table = torch.zeros((batch, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_no_alloc(d, q, qp, x["cache"], None, table, lens, x["W_UK"], x["W_UV"], 0.1, num_splits=152)
    assert e.value.status == mla.MLA_ERR_WORKSPACE
