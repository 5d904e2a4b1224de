"""Kernel-level GPU parity: the FP8 weight quantisation is byte work and must
be bit-exact against the oracle's own quantiser."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ads():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import ar_decode_step_gb300.build as b
    b.build()
    import ar_decode_step_gb300 as m
    m.load()
    return m


@pytest.mark.parametrize("shape,stream", [((6144, 2560), 901), ((2560, 9728), 902), ((37, 272), 903)])
def test_quantize_fp8_weight_bit_exact(ads, shape, stream):
    import torch
    W = synth.normal_bf16(0, stream, shape, std=0.02)
    W[3] = 0                     # zero row: scale 1, all-zero codes
    W[5, :4] = [0x43E0, 0xC3E0, 0x3F80, 0x0001]  # 448, -448, 1, a subnormal
    q_ref, s_ref = oracle.quant_weight(W)
    wd = torch.from_numpy(W.view(np.int16)).cuda()
    q, s = ads.quantize_fp8_weight(wd)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
