"""mla_decode_no_alloc: the decode entry point for callers that cannot
allocate device memory (for example a serving loop that must not call
cudaMalloc on its decode path, because the call can synchronise the device,
or a C host whose device memory is budgeted up front by someone else).  It
runs on the library's fixed scratch array instead of a caller workspace.

These checks call it through the C ABI twice in a row for each cache format
and require both results to be bit-identical to mla_decode's with the same
split count (the same kernels run on the same inputs), check one of them
against the fp64 oracle, check that a device-side status (a bounded wait
that ran out) is copied out of the shared scratch and that the next call is
clean again, and check that a shape needing more scratch than the array
holds is refused.  Kept in a file collected last."""
import numpy as np
import pytest
import torch

import oracle as O
import mla_decode_attention_paged_gb300 as mla
from mla_decode_attention_paged_gb300 import workloads as W
from harness import assert_parity, f64

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(192.0)
SPLITS = 40


def _inputs(fmt, heads=16, lens=(3000, 129, 4096, 1), P=64, seed=21):
    g = W.generator(seed)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    table, npg = W.draw_page_table(seq_lens, P, True, g)
    x = dict(seq_lens=seq_lens, table=table, W_UK=W.draw_bf16((heads, 128, 512), 0.02, g),
             W_UV=W.draw_bf16((heads, 128, 512), 0.02, g), q_nope=W.draw_bf16((len(lens), heads, 128), 1.0, g),
             q_pe=W.draw_bf16((len(lens), heads, 64), 1.0, g), sz=None, P=P)
    if fmt == "bf16":
        x["cache"] = W.draw_bf16((npg, P, 576), 1.0, g)
    else:
        x["cache"], x["sz"] = W.draw_int8_cache(npg, P, g) if fmt == "int8" else W.draw_fp8_cache(npg, P, g)
    return mla.dims(heads, P, int8=fmt == "int8", fp8=fmt == "fp8"), x


def _dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _decode(d, x):
    out, lse = mla.decode(d, x["q_nope"], x["q_pe"], x["cache"], x["sz"], x["table"], x["seq_lens"], x["W_UK"],
                          x["W_UV"], SCALE, num_splits=SPLITS)
    torch.cuda.synchronize()
    return out, lse


def _no_alloc(d, x, status):
    lse = torch.empty((x["q_nope"].shape[0], d.num_heads), dtype=torch.float32, device="cuda")
    out, _ = mla.decode_no_alloc(d, x["q_nope"], x["q_pe"], x["cache"], x["sz"], x["table"], x["seq_lens"],
                                 x["W_UK"], x["W_UV"], SCALE, num_splits=SPLITS, lse_out=lse, device_status=status)
    torch.cuda.synchronize()
    return out, lse


def _oracle(fmt, x):
    cache = W.bf16_to_bits(x["cache"]) if fmt == "bf16" else x["cache"].numpy()
    sz = None if x["sz"] is None else x["sz"].numpy()
    return O.decode(f64(x["q_nope"]), f64(x["q_pe"]), cache, sz, x["table"].numpy(), x["seq_lens"].numpy(),
                    f64(x["W_UK"]), f64(x["W_UV"]), SCALE, x["P"], fmt == "int8", fp8=fmt == "fp8")


@pytest.mark.parametrize("fmt,heads", [("bf16", 16), ("int8", 16), ("fp8", 16), ("bf16", 128), ("int8", 128)])
def test_no_alloc_equals_decode_on_two_calls(cuda_lib, fmt, heads):
    # 16 heads: the pair (bf16) and single-CTA (1-byte) kernels; 128 heads: the 128-row kernel
    d, host = _inputs(fmt, heads=heads, lens=(3000, 129, 4096, 1) if heads == 16 else (700, 129, 65, 1))
    assert mla.decode_workspace_size(d, 4, SPLITS) <= mla.NO_ALLOC_WORKSPACE_BYTES
    x = _dev(host)
    ref_out, ref_lse = _decode(d, x)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for call in range(2):
        out, lse = _no_alloc(d, x, status)
        assert int(status.item()) == mla.MLA_OK, call
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), call
    ref_o, ref_l = _oracle(fmt, host)
    B, H = ref_o.shape[:2]
    assert_parity(out, lse, ref_o, ref_l, [(b, h) for b in range(B) for h in range(H)], f"no-alloc {fmt} {heads}")


def test_no_alloc_reports_device_status_and_recovers(cuda_lib):
    """A bounded wait that runs out inside the attention kernel (the library's
    test hook, as for mla_decode) is reported through device_status; the next
    call on the same scratch reports MLA_OK and gives the same results as
    before."""
    d, host = _inputs("bf16", lens=(700, 129))
    x = _dev(host)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ref_out, ref_lse = _no_alloc(d, x, status)
    assert int(status.item()) == mla.MLA_OK
    try:
        mla.test_inject_wait_timeout(True)
        _no_alloc(d, x, status)
        assert int(status.item()) == mla.MLA_ERR_DEVICE_TIMEOUT
    finally:
        mla.test_inject_wait_timeout(False)
    out, lse = _no_alloc(d, x, status)
    assert int(status.item()) == mla.MLA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_no_alloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    d, host = _inputs("bf16")
    x = _dev(host)
    batch = 4096  # (splits + batch) * H * 2 KB of partials alone exceeds the fixed array
    assert mla.decode_workspace_size(d, batch, 152) > mla.NO_ALLOC_WORKSPACE_BYTES
    q = torch.zeros((batch, 16, 128), dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros((batch, 16, 64), dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(batch, dtype=torch.int32, device="cuda")
    table = torch.zeros((batch, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_no_alloc(d, q, qp, x["cache"], None, table, lens, x["W_UK"], x["W_UV"], 0.1, num_splits=152)
    assert e.value.status == mla.MLA_ERR_WORKSPACE
