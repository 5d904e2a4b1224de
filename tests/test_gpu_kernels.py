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


def _oracle_attention_layer(qkv, qn, kn, K, V, n_q, n_kv, pos, eps=1e-6, theta=1e6):
    """The oracle's building blocks composed for one layer at position pos:
    q/k RMSNorm + RoPE, bf16 KV write at pos, GQA attention over [0, pos]."""
    D = 128
    q = np.array([oracle.rope(oracle.rmsnorm(qkv[h * D:(h + 1) * D], qn, eps), pos, theta) for h in range(n_q)])
    K, V = K.copy(), V.copy()
    for j in range(n_kv):
        k = oracle.rope(oracle.rmsnorm(qkv[(n_q + j) * D:(n_q + j + 1) * D], kn, eps), pos, theta)
        v = qkv[(n_q + n_kv + j) * D:(n_q + n_kv + j + 1) * D]
        K[j, pos] = [oracle.f64_to_bf16(x) for x in k]
        V[j, pos] = [oracle.f64_to_bf16(x) for x in v]
    return oracle.attention(q, K, V, pos + 1).reshape(-1), K, V


@pytest.mark.parametrize("n_q,n_kv,max_pos,pos", [(32, 8, 300, 0), (32, 8, 300, 15), (32, 8, 300, 16),
                                                 (32, 8, 300, 211), (32, 8, 300, 299), (8, 8, 64, 40),
                                                 (16, 2, 1100, 1099)])
def test_attention_op_matches_oracle(ads, n_q, n_kv, max_pos, pos):
    import torch
    D = 128
    qkv = synth.normal_f32(5, 1000 + pos, ((n_q + 2 * n_kv) * D,), std=1.5)
    qn = synth.normal_bf16(3, 1, (D,), std=0.02, mean=1.0)
    kn = synth.normal_bf16(3, 2, (D,), std=0.02, mean=1.0)
    K = synth.normal_bf16(1, 11, (n_kv, max_pos, D))
    V = synth.normal_bf16(1, 12, (n_kv, max_pos, D))
    ref, K_ref, V_ref = _oracle_attention_layer(qkv.astype(np.float64), qn, kn, K, V, n_q, n_kv, pos)
    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    kd, vd = dev(K.copy()), dev(V.copy())
    out = torch.zeros(n_q * D, dtype=torch.float32, device="cuda")
    ads.attention_decode(dev(qkv), dev(qn), dev(kn), kd, vd, out, n_q, n_kv, pos)
    got = out.cpu().numpy().astype(np.float64)
    assert np.allclose(got, ref, rtol=1e-3, atol=2e-3), np.abs(got - ref).max()
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kh, vh = kd.cpu().numpy().view(np.uint16), vd.cpu().numpy().view(np.uint16)
    assert np.allclose(f(kh[:, pos]), f(K_ref[:, pos]), rtol=2 ** -7, atol=1e-6)
    assert np.array_equal(vh[:, pos], V_ref[:, pos])       # v is only rounded: bit-exact
    kh[:, pos] = K[:, pos]
    vh[:, pos] = V[:, pos]
    assert np.array_equal(kh, K) and np.array_equal(vh, V)  # nothing else written


def test_attention_op_rejects_bad_args(ads):
    import torch
    z = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(ads.TtsError) as e:
        ads._call("tts_attention_decode", z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                  z.data_ptr(), 32, 8, 64, 64, 1e-6, 1e6, None)
    assert e.value.status == -3
    with pytest.raises(ads.TtsError) as e:
        ads._call("tts_attention_decode", z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                  z.data_ptr(), 24, 8, 64, 3, 1e-6, 1e6, None)
    assert e.value.status == -1
