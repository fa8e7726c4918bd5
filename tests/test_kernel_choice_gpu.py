"""The kernel variant each layer kind takes by default, as td_kernel_name
reports it on the device: the automatic choices follow the measured rules
(tensor cores for G = 4, 8 with 16 tokens per warp on full layers and the
shared-memory ring on sparse layers; CUDA cores for G = 1, 2 with rows staged
through cp.async when every CTA gathers one round or less)."""
import pytest
import torch

import sparse_attention_td_gb300 as td

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_default_kernel_choices():
    gqa = td.make_shape(4, 32, 8, 32768)
    assert td.td_kernel_name(gqa, 0, False).startswith("attention_mma16_kernel (tensor cores, 16 tokens per warp)")
    assert td.td_kernel_name(gqa, 2048, True).startswith("attention_mma_ring_kernel")  # 8 splits
    serving = td.make_shape(32, 32, 8, 16384)
    assert td.td_kernel_name(serving, 4096, True).startswith("attention_mma_ring_kernel")
    assert td.td_kernel_name(serving, 1024, True).startswith("attention_mma_ring_kernel")
    assert td.td_kernel_name(serving, 256, True).startswith("attention_mma_ring_kernel")
    mha = td.make_shape(1, 32, 32, 10240)
    assert "cp.async" in td.td_kernel_name(mha, 512, True)          # 32 x 512 rows: one round a CTA
    assert "register-streamed" in td.td_kernel_name(mha, 0, False)
    long_mha = td.make_shape(1, 32, 32, 102400)
    assert "register-streamed" in td.td_kernel_name(long_mha, 4096, True)


def test_tuning_overrides_are_reported():
    mha = td.make_shape(1, 32, 32, 102400)
    try:
        td.td_set_tuning("sparse_staged", 2)
        assert "TMA row gathers" in td.td_kernel_name(mha, 4096, True)
        td.td_set_tuning("mma", 0)
        assert td.td_kernel_name(td.make_shape(4, 32, 8, 32768), 0, False).startswith("attention_kernel")
    finally:
        td.td_set_tuning("sparse_staged", -1)
        td.td_set_tuning("mma", -1)
