"""Pins for the CPU oracle: each building block is checked against something
other than itself -- library routines (torch CPU casts, rms_norm, SDPA, numpy
float64 matmul), closed forms, invariants, exact integer arithmetic and brute
force on tiny inputs -- so that a dropped term, a wrong sign or index, or a
transposed operand fails one of them.  No GPU."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

pytestmark = pytest.mark.usefixtures("oracle_lib")

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit images with torch's own bfloat16 type (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def f32_to_bf16_bits_torch(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def e4m3_decode_torch(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e4m3_encode_torch(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# ----------------------------------------------------------------------------
# Scalar formats
# ----------------------------------------------------------------------------

def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = e4m3_decode_torch(codes)
    got = np.array([oracle.e4m3_decode(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # only S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_spec_values():
    # OCP 8-bit FP spec, E4M3: max normal 448, min normal 2^-6, min subnormal 2^-9.
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0xB8) == -1.0
    # round-trip of every finite code
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        enc = oracle.e4m3_encode(v)
        if v == 0.0:
            assert enc in (0x00, 0x80)
        else:
            assert enc == c, (c, v, enc)
    # ties go to the even mantissa
    assert oracle.e4m3_encode(1.0625) == 0x38   # between 1.0 (m=0) and 1.125 (m=1)
    assert oracle.e4m3_encode(1.1875) == 0x3A   # between 1.125 (m=1) and 1.25 (m=2)
    assert oracle.e4m3_encode(3.0 * 2.0 ** -10) == 0x02  # subnormal tie 1.5 -> 2
    # saturation of finite overflow
    assert oracle.e4m3_encode(448.0 * (1 + 2.0 ** -4)) == 0x7E
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1234)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 50,
        rng.uniform(-448, 448, 200_000).astype(np.float32),
        (rng.standard_normal(100_000) * 2.0 ** -7).astype(np.float32),  # subnormal region
    ])
    ref = e4m3_encode_torch(x)
    enc = np.vectorize(oracle.e4m3_encode, otypes=[np.uint8])
    got = enc(x)
    # +-0 may differ in sign only for values that round to zero; compare values
    ref_v = e4m3_decode_torch(ref)
    got_v = e4m3_decode_torch(got)
    assert np.array_equal(ref_v, got_v)


def test_bf16_rounding():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100_000) * 10.0 ** rng.uniform(-8, 8, 100_000)).astype(np.float32)
    ref = f32_to_bf16_bits_torch(x)
    got = np.array([oracle.f32_to_bf16(v) for v in x], np.uint16)
    assert np.array_equal(ref, got)
    # direct rounding from fp64: a value just above a bf16 midpoint rounds up,
    # which a two-step fp64 -> fp32 -> bf16 rounding would get wrong.
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80          # exact tie -> even
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie 1.5 ulp -> even (2)
    assert oracle.f64_to_bf16(-2.0) == 0xC000
    bits = np.arange(0, 65536, 97, dtype=np.uint16)
    vals = bf16_bits_to_f64(bits)
    for b, v in zip(bits, vals):
        if np.isfinite(v):
            assert oracle.bf16_to_f64(b) == v


# ----------------------------------------------------------------------------
# RMSNorm
# ----------------------------------------------------------------------------

def test_rmsnorm_against_torch_and_invariants():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(2560) * 3.0
    g = synth.normal_bf16(3, 1, (2560,), std=0.02, mean=1.0)
    y = oracle.rmsnorm(x, g, 1e-6)
    ref = F.rms_norm(torch.from_numpy(x), (2560,), torch.from_numpy(bf16_bits_to_f64(g)), eps=1e-6).numpy()
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)
    ones = np.full(2560, 0x3F80, np.uint16)
    y1 = oracle.rmsnorm(x, ones, 1e-6)
    assert abs(math.sqrt(np.mean(y1 ** 2)) - 1.0) < 1e-6
    assert np.allclose(oracle.rmsnorm(7.5 * x, ones, 0.0), oracle.rmsnorm(x, ones, 0.0), rtol=1e-13)
    # gamma is applied per element (a dropped or transposed gamma fails this)
    assert np.allclose(y, y1 * bf16_bits_to_f64(g), rtol=1e-13)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def test_rope_invariants_and_closed_forms():
    rng = np.random.default_rng(1)
    D, theta = 128, 1e6
    x = rng.standard_normal(D)
    assert np.array_equal(oracle.rope(x, 0, theta), x)  # position 0 is the identity
    for pos in (1, 5, 141, 4000, 8191):
        y = oracle.rope(x, pos, theta)
        # each (i, i+64) pair keeps its norm
        n0 = x[:64] ** 2 + x[64:] ** 2
        n1 = y[:64] ** 2 + y[64:] ** 2
        assert np.allclose(n0, n1, rtol=1e-12)
        # pair 0 has inverse frequency 1: its angle is the position itself
        c, s = math.cos(pos), math.sin(pos)
        assert abs(y[0] - (x[0] * c - x[64] * s)) < 1e-12
        assert abs(y[64] - (x[64] * c + x[0] * s)) < 1e-12
        # pair 63 has inverse frequency theta^(-126/128)
        a = pos * theta ** (-126.0 / 128.0)
        assert abs(y[63] - (x[63] * math.cos(a) - x[127] * math.sin(a))) < 1e-12
    # <RoPE(q, m), RoPE(k, n)> depends only on m - n
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for m, n in ((5, 0), (4000, 3995), (8000, 7995)):
        d0 = np.dot(oracle.rope(q, m, theta), oracle.rope(k, n, theta))
        d1 = np.dot(oracle.rope(q, m - n, theta), k)
        assert abs(d0 - d1) < 1e-9


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------

def _rand_cache(rng, n_kv, max_pos, D):
    k = synth.normal_bf16(1, int(rng.integers(1 << 30)), (n_kv, max_pos, D))
    v = synth.normal_bf16(1, int(rng.integers(1 << 30)), (n_kv, max_pos, D))
    return k, v


def test_attention_single_key_returns_v():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((32, 128)) * 5
    K, V = _rand_cache(rng, 8, 16, 128)
    out = oracle.attention(q, K, V, 1)
    Vd = bf16_bits_to_f64(V)
    for h in range(32):
        assert np.array_equal(out[h], Vd[h // 4, 0])


def test_attention_equal_keys_mean_and_grouping_and_causality():
    rng = np.random.default_rng(3)
    n_q, n_kv, D, T = 32, 8, 128, 40
    K, V = _rand_cache(rng, n_kv, 64, D)
    Keq = K.copy()
    Keq[:, :T] = K[:, :1]
    q = rng.standard_normal((n_q, D))
    out = oracle.attention(q, Keq, V, T)
    Vd = bf16_bits_to_f64(V)
    for h in range(n_q):
        assert np.allclose(out[h], Vd[h // 4, :T].mean(axis=0), rtol=1e-12, atol=1e-14)
    # head grouping: kv head j's distinctive V reaches q heads 4j..4j+3 only
    Vmark = np.zeros_like(V)
    for j in range(n_kv):
        Vmark[j, :, :] = np.uint16(0x3F80 + j)  # bf16 1.0 + j ulps: distinct per kv head
    out = oracle.attention(q, K, Vmark, T)
    for h in range(n_q):
        assert np.allclose(out[h], bf16_bits_to_f64(np.array([0x3F80 + h // 4], np.uint16))[0])
    # causality: entries at positions >= len do not matter
    K2, V2 = K.copy(), V.copy()
    K2[:, T:] = 0x4000
    V2[:, T:] = 0xC000
    assert np.array_equal(oracle.attention(q, K, V, T), oracle.attention(q, K2, V2, T))


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(4)
    n_q, n_kv, D, T = 8, 2, 32, 37
    K, V = _rand_cache(rng, n_kv, 48, D)
    q = rng.standard_normal((n_q, D))
    out = oracle.attention(q, K, V, T)
    Kt = torch.from_numpy(bf16_bits_to_f64(K[:, :T])).repeat_interleave(n_q // n_kv, 0)
    Vt = torch.from_numpy(bf16_bits_to_f64(V[:, :T])).repeat_interleave(n_q // n_kv, 0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], Kt, Vt)[:, 0, :].numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# Projections
# ----------------------------------------------------------------------------

def test_linear_bf16_brute_force():
    rng = np.random.default_rng(5)
    W = synth.normal_bf16(0, 77, (24, 40), std=0.5)
    x = rng.standard_normal(40)
    y = oracle.linear_bf16(W, x)
    assert np.allclose(y, bf16_bits_to_f64(W) @ x, rtol=1e-13, atol=1e-13)
    # identity / one-hot rows pick single inputs (a transposed W fails this)
    eye = np.zeros((40, 40), np.uint16)
    eye[np.arange(40), (np.arange(40) * 7) % 40] = 0x3F80
    assert np.array_equal(oracle.linear_bf16(eye, x), x[(np.arange(40) * 7) % 40])


def test_linear_fp8_exact_integer_arithmetic():
    rng = np.random.default_rng(6)
    N, K = 8, 16
    W8 = rng.integers(0, 256, (N, K), dtype=np.uint8)
    W8[(W8 & 0x7F) == 0x7F] = 0x10  # no NaN codes
    a8 = rng.integers(0, 256, K, dtype=np.uint8)
    a8[(a8 & 0x7F) == 0x7F] = 0x22
    sw = rng.uniform(0.001, 0.01, N).astype(np.float32)
    sa = np.float32(0.0123)
    y = oracle.linear_fp8(W8, sw, a8, float(sa))
    # every e4m3 value is an integer multiple of 2^-9: sum products exactly in integers
    wi = (e4m3_decode_torch(W8) * 512).astype(np.int64)
    ai = (e4m3_decode_torch(a8) * 512).astype(np.int64)
    for n in range(N):
        acc_int = sum(int(wi[n, k]) * int(ai[k]) for k in range(K))  # acc * 2^18
        acc32 = np.float32(acc_int / 2.0 ** 18)
        v = np.float32(acc32 * np.float32(sa * sw[n]))
        ref = bf16_bits_to_f64(f32_to_bf16_bits_torch(np.array([v])))[0]
        assert y[n] == ref


def test_quant_weight_and_act_match_torch_cast():
    W = synth.normal_bf16(0, 91, (64, 256), std=0.02)
    W[5] = 0  # an all-zero row takes scale 1
    q, s = oracle.quant_weight(W)
    Wf = torch.from_numpy(bf16_bits_to_f64(W).astype(np.float32))
    amax = Wf.abs().amax(dim=1)
    s_ref = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert np.array_equal(s, s_ref.numpy())
    q_ref = (Wf / s_ref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, q_ref)
    # the row maximum maps to +-448 exactly
    for n in range(64):
        if n != 5:
            assert np.abs(e4m3_decode_torch(q[n])).max() == 448.0
    x = np.random.default_rng(8).standard_normal(2560) * 2.0
    qa, sa = oracle.quant_act(x)
    x32 = torch.from_numpy(x.astype(np.float32))
    sa_ref = torch.clamp(x32.abs().amax(), min=1e-12) / 448.0
    assert sa == sa_ref.item()
    assert np.array_equal(qa, (x32 / sa_ref).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(oracle.silu(-1.0) + math.exp(-1.0) / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    z = torch.linspace(-20, 20, 1001, dtype=torch.float64)
    ref = F.silu(z).numpy()
    got = np.array([oracle.silu(float(v)) for v in z])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)


# ----------------------------------------------------------------------------
# Embedding, argmax, delay pattern
# ----------------------------------------------------------------------------

def test_embed_one_hot_rows():
    C, V, H = 8, 1026, 2560
    E = np.zeros((C, V, H), np.uint16)
    codes = np.array([0, 17, 1023, 1024, 1025, 5, 512, 999], np.int32)
    for k in range(C):
        for c in range(V):
            E[k, c, (k * 37 + c) % H] = 0x3F80
    x = oracle.embed(E, codes)
    ref = np.zeros(H)
    for k in range(C):
        ref[(k * 37 + codes[k]) % H] += 1.0
    assert np.array_equal(x, ref)


def test_argmax_ties_lowest_index():
    v = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert oracle.argmax(v) == 1
    assert oracle.argmax(np.full(1026, 3.25)) == 0
    w = np.zeros(1026)
    w[1025] = 1e-300
    assert oracle.argmax(w) == 1025


def _read_delay_golden():
    rows = {}
    with open(f"{GOLDEN}/delay_pattern.txt") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            t, rest = line.split(":")
            rows[int(t)] = [x.strip() for x in rest.split()]
    return rows


def test_delay_pattern_table():
    """Brute-force table for frames 0..10 with codebook 0 emitting EOC at frame 2
    (tests/golden/delay_pattern.txt); 'A' marks the argmax (live) entries."""
    table = _read_delay_golden()
    assert sorted(table) == list(range(11))
    eoc = 2
    for t, row in table.items():
        for k, want in enumerate(row):
            got = oracle.delay_code(k, t, eoc, 77)
            if want == "A":
                assert got == 77, (t, k)
            else:
                assert got == int(want), (t, k)
    # no EOC yet: only the BOS region is forced
    for t in range(12):
        for k in range(8):
            assert oracle.delay_code(k, t, -1, 5) == (1024 if t < k else 5)


def test_undelay_round_trip():
    """Row i of codebook k in the delayed stream is frame i - k of the
    un-delayed stream; shifting back recovers the frames."""
    rng = np.random.default_rng(9)
    T, C = 12, 8
    frames = rng.integers(0, 1024, (T, C))
    delayed = np.full((T + C - 1, C), 1024)
    for k in range(C):
        delayed[k:k + T, k] = frames[:, k]
    back = np.stack([delayed[k:k + T, k] for k in range(C)], axis=1)
    assert np.array_equal(back, frames)
    for t in range(C):
        for k in range(C):
            if t < k:
                assert delayed[t, k] == oracle.delay_code(k, t, -1, -5)
