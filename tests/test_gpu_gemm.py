"""The tensor-core GEMM of the batched prefill (tts_gemm_bf16, tts_gemm_fp8,
tts_gemm_tiled) against the CPU oracle's linear layer (fp64 sums of the same
operands): plain store, additive epilogue, and the fused gate/up + SwiGLU
epilogue, on shapes with ragged M (rows past M are masked), several N tiles
and several k-blocks, covering every tile width, 128- and 256-row tiles and
the cluster split of the K range (its partial sums added in a fixed order:
bit-identical from run to run)."""
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


TILED = [  # M, N, K, epi, tile rows, tile columns, K split
    (300, 320, 512, 1, 256, 160, 4),
    (300, 384, 1024, 0, 256, 192, 2),
    (37, 256, 1024, 1, 128, 128, 3),
    (200, 160, 256, 0, 256, 80, 1),
    (260, 256, 512, 2, 256, 128, 1),
    (130, 192, 512, 1, 256, 64, 1),
    (90, 320, 768, 0, 128, 160, 3),
]


@pytest.mark.parametrize("M,N,K,epi,rows,cols,splits", TILED)
def test_gemm_tiled_bf16(env, M, N, K, epi, rows, cols, splits):
    ads, torch = env
    Ab = synth.normal_bf16(2, 121, (M, K))
    Wb = synth.normal_bf16(2, 122, ((2 * N if epi == 2 else N), K), std=0.05 if epi == 2 else 0.02)
    base = synth.normal_f32(2, 123, (M, N))
    runs = []
    for _ in range(2):
        if epi == 2:
            C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        elif epi == 1:
            C = torch.from_numpy(base.copy()).cuda()
        else:
            C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        ads.gemm_tiled(bf16_dev(torch, Ab), bf16_dev(torch, Wb), C, epi, rows, cols, splits)
        torch.cuda.synchronize()
        runs.append(C.float().cpu().numpy())
    assert np.array_equal(runs[0], runs[1]), "split sums must be deterministic"
    got = runs[0].astype(np.float64)
    y = ref_rows(Wb, Ab)
    if epi == 2:
        g, u = y[:, :N], y[:, N:]
        ref = g / (1.0 + np.exp(-g)) * u
        assert np.allclose(got, ref, rtol=2 ** -7, atol=1e-3 * np.abs(ref).max())
    else:
        ref = y if epi == 0 else base.astype(np.float64) + y
        assert np.isfinite(got).all()
        assert np.allclose(got, ref, rtol=1e-4, atol=2e-4 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K,epi,rows,cols,splits", [
    (300, 320, 1024, 1, 256, 160, 4),
    (300, 384, 1024, 0, 256, 192, 2),
    (260, 256, 512, 2, 256, 128, 1),
    (45, 192, 512, 0, 128, 64, 2),
])
def test_gemm_tiled_fp8(env, M, N, K, epi, rows, cols, splits):
    ads, torch = env
    qa, sa, qa_d, sa_d = fp8_operands(torch, 131, M, K, 1.0)
    qw, sw, qw_d, sw_d = fp8_operands(torch, 132, 2 * N if epi == 2 else N, K, 0.02)
    base = synth.normal_f32(2, 133, (M, N))
    if epi == 2:
        C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    elif epi == 1:
        C = torch.from_numpy(base.copy()).cuda()
    else:
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ads.gemm_tiled(qa_d, qw_d, C, epi, rows, cols, splits, a_scale_dev=sa_d, b_scale_dev=sw_d)
    torch.cuda.synchronize()
    got = C.float().cpu().numpy().astype(np.float64)
    y = ref_fp8(qa, sa, qw, sw)
    if epi == 2:
        g, u = y[:, :N], y[:, N:]
        ref = g / (1.0 + np.exp(-g)) * u
        assert np.allclose(got, ref, rtol=2 ** -6, atol=2e-3 * np.abs(ref).max())
    else:
        ref = y if epi == 0 else base.astype(np.float64) + y
        assert np.allclose(got, ref, rtol=2 ** -7, atol=1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("rows,cols,splits", [(192, 128, 1), (128, 96, 1), (256, 128, 5), (128, 64, 17)])
def test_gemm_tiled_rejects_bad_tiles(env, rows, cols, splits):
    """Tiles the kernel does not build (row count, width, split count, a split
    with no k-block) are refused before any launch."""
    ads, torch = env
    A = torch.zeros((64, 1024), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((128, 1024), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(ads.TtsError):
        ads.gemm_tiled(A, B, C, 0, rows, cols, splits)
