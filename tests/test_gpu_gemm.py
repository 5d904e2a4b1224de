"""The tensor-core GEMM of the batched prefill (tts_gemm_bf16) against the CPU
oracle's linear layer (fp64 sums of the same bf16 operands): plain store,
additive epilogue with split-K, and the fused gate/up + SwiGLU epilogue, on
shapes with ragged M (rows past M are masked), several N tiles and several
k-blocks, covering the 64-, 80-, 128- and 192-column tile widths."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import ar_decode_step_gb300.build as b
    b.build()
    import ar_decode_step_gb300 as m
    m.load()
    return m, torch


def bf16_dev(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def ref_rows(Wb, Ab):
    """Oracle linear layer applied to every row of A: [M][N] fp64."""
    return np.stack([oracle.linear_bf16(Wb, f64(Ab[i])) for i in range(Ab.shape[0])])


@pytest.mark.parametrize("M,N,K", [(37, 128, 64), (200, 256, 512), (300, 384, 2560), (260, 640, 512),
                                   (512, 2560, 256)])
def test_gemm_store(env, M, N, K):
    ads, torch = env
    Ab = synth.normal_bf16(2, 101, (M, K))
    Wb = synth.normal_bf16(2, 102, (N, K), std=0.02)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ads.gemm_bf16(bf16_dev(torch, Ab), bf16_dev(torch, Wb), C, epi=0)
    torch.cuda.synchronize()
    got = C.cpu().numpy().astype(np.float64)
    ref = ref_rows(Wb, Ab)
    assert np.isfinite(got).all()
    assert np.allclose(got, ref, rtol=1e-4, atol=1e-4 * np.abs(ref).max())


@pytest.mark.parametrize("splits", [1, 3])
def test_gemm_add_split_k(env, splits):
    ads, torch = env
    M, N, K = 150, 256, 1024
    Ab = synth.normal_bf16(2, 103, (M, K))
    Wb = synth.normal_bf16(2, 104, (N, K), std=0.02)
    base = synth.normal_f32(2, 105, (M, N))
    C = torch.from_numpy(base.copy()).cuda()
    ads.gemm_bf16(bf16_dev(torch, Ab), bf16_dev(torch, Wb), C, epi=1, splits=splits)
    torch.cuda.synchronize()
    got = C.cpu().numpy().astype(np.float64)
    ref = base.astype(np.float64) + ref_rows(Wb, Ab)
    assert np.allclose(got, ref, rtol=1e-4, atol=2e-4 * np.abs(ref).max())


def test_gemm_swiglu(env):
    ads, torch = env
    M, N, K = 130, 256, 512
    Ab = synth.normal_bf16(2, 106, (M, K))
    Wb = synth.normal_bf16(2, 107, (2 * N, K), std=0.05)
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    ads.gemm_bf16(bf16_dev(torch, Ab), bf16_dev(torch, Wb), out, epi=2)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    gu = ref_rows(Wb, Ab)
    g, u = gu[:, :N], gu[:, N:]
    ref = g / (1.0 + np.exp(-g)) * u
    # one bf16 rounding of an fp32 value: within 2^-8 relative (plus tiny values)
    assert np.allclose(got, ref, rtol=2 ** -7, atol=1e-3 * np.abs(ref).max())


def fp8_operands(torch, seed, rows, K, std):
    """E4M3 rows with a per-row scale (the oracle's quantisation of bf16 draws)."""
    Wb = synth.normal_bf16(2, seed, (rows, K), std=std)
    q, sw = oracle.quant_weight(Wb)
    return q, sw, torch.from_numpy(np.ascontiguousarray(q)).cuda(), torch.from_numpy(np.ascontiguousarray(sw)).cuda()


def ref_fp8(q_a, sa, q_w, sw):
    """Oracle FP8 projection per row: bf16(fp32(sum a8 w8) * fp32(sa * sw[n]))."""
    return np.stack([oracle.linear_fp8(q_w, sw, q_a[i], float(sa[i])) for i in range(q_a.shape[0])])


@pytest.mark.parametrize("M,N,K,epi", [(37, 128, 256, 0), (300, 384, 2560, 0), (130, 256, 512, 1), (260, 256, 1024, 2)])
def test_gemm_fp8(env, M, N, K, epi):
    ads, torch = env
    qa, sa, qa_d, sa_d = fp8_operands(torch, 111, M, K, 1.0)
    rows = 2 * N if epi == 2 else N
    qw, sw, qw_d, sw_d = fp8_operands(torch, 112, rows, K, 0.02)
    if epi == 2:
        C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    elif epi == 1:
        base = synth.normal_f32(2, 113, (M, N))
        C = torch.from_numpy(base.copy()).cuda()
    else:
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ads.gemm_fp8(qa_d, qw_d, sa_d, sw_d, C, epi=epi)
    torch.cuda.synchronize()
    got = C.float().cpu().numpy().astype(np.float64)
    y = ref_fp8(qa, sa, qw, sw)
    if epi == 2:
        g, u = y[:, :N], y[:, N:]
        silu = g / (1.0 + np.exp(-g))
        ref = silu * u
        assert np.allclose(got, ref, rtol=2 ** -6, atol=2e-3 * np.abs(ref).max())
    else:
        ref = y if epi == 0 else base.astype(np.float64) + y
        # bf16 outputs: the GPU's fp32 sum may round to the neighbouring bf16 value
        assert np.allclose(got, ref, rtol=2 ** -7, atol=1e-6 * np.abs(ref).max())
