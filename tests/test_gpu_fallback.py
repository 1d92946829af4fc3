"""The single-CTA attention kernel: the fallback for devices on which the
CTA-pair kernels cannot be placed.  GB300 always places the pairs, so the
test hook mla_test_force_single_cta routes decodes (bf16, INT8 and FP8
caches) to the fallback and these cases check it against the fp64 oracle."""
import pytest
import torch

import mla_decode_attention_paged_gb300 as mla
from harness import assert_parity
from test_gpu_parity import _run_small, _small

pytestmark = pytest.mark.gpu


@pytest.fixture
def single_cta(cuda_lib):
    mla.test_force_single_cta(True)
    try:
        yield
    finally:
        mla.test_force_single_cta(False)


@pytest.mark.parametrize("heads,P,lens", [(16, 64, (1, 129, 700, 256)), (32, 16, (383, 130)),
                                          (128, 64, (0, 255, 1030)), (64, 128, (2500, 5))])
def test_single_cta_bf16_parity(single_cta, heads, P, lens):
    _run_small(*_small(heads=heads, P=P, lens=lens, seed=heads + P))


@pytest.mark.parametrize("splits", [1, 7, 300])
def test_single_cta_bf16_splits(single_cta, splits):
    _run_small(*_small(lens=(1000, 5, 2500, 128), seed=splits), num_splits=splits)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_single_cta_one_byte_parity(single_cta, fmt):
    _run_small(*_small(lens=(1, 129, 700, 2000), int8=fmt == "int8", fp8=fmt == "fp8", seed=77))
