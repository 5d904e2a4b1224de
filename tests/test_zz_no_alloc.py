"""The allocation-free attention entry point, called through the C ABI.

Some callers cannot allocate device memory when they call in (a fixed memory
budget owned by another runtime, a loop that must never block in cudaMalloc).
tts_attention_decode_noalloc serves them from a static device array.  Both
entry points run the same kernel with the same split count and merge order,
so here the allocation-free output must equal tts_attention_decode's (which
takes its scratch from the stream-ordered allocator) bit for bit, on calls in
a row -- including a call at a small context after one at a large context,
whose leftovers in the shared array must not leak into the result -- and must
meet the CPU oracle's attention.  This file is collected last so that a
failure here comes after every other test."""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import ar_decode_step_gb300.build as b
    b.build()
    import ar_decode_step_gb300 as m
    return m.load()


def _inputs(n_q, n_kv, max_pos, seed):
    qkv = synth.normal_f32(5, seed, ((n_q + 2 * n_kv) * D,), std=1.5)
    qn = synth.normal_bf16(3, seed + 1, (D,), std=0.02, mean=1.0)
    kn = synth.normal_bf16(3, seed + 2, (D,), std=0.02, mean=1.0)
    K = synth.normal_bf16(1, seed + 3, (n_kv, max_pos, D))
    V = synth.normal_bf16(1, seed + 4, (n_kv, max_pos, D))
    return qkv, qn, kn, K, V


def _dev(a):
    import torch
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def _call(lib, name, qkv, qn, kn, kd, vd, out, n_q, n_kv, max_pos, pos):
    f = getattr(lib, name)
    return f(ctypes.c_void_p(qkv.data_ptr()), ctypes.c_void_p(qn.data_ptr()), ctypes.c_void_p(kn.data_ptr()),
             ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(vd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
             n_q, n_kv, max_pos, pos, ctypes.c_float(1e-6), ctypes.c_float(1e6), None)


def _oracle_attention(qkv, qn, kn, K, V, n_q, n_kv, pos, eps=1e-6, theta=1e6):
    """The oracle's q/k RMSNorm + RoPE, bf16 KV write at pos and GQA attention
    over [0, pos], composed for one layer."""
    q = np.array([oracle.rope(oracle.rmsnorm(qkv[h * D:(h + 1) * D], qn, eps), pos, theta) for h in range(n_q)])
    K, V = K.copy(), V.copy()
    for j in range(n_kv):
        k = oracle.rope(oracle.rmsnorm(qkv[(n_q + j) * D:(n_q + j + 1) * D], kn, eps), pos, theta)
        K[j, pos] = [oracle.f64_to_bf16(x) for x in k]
        V[j, pos] = [oracle.f64_to_bf16(x) for x in qkv[(n_q + n_kv + j) * D:(n_q + n_kv + j + 1) * D]]
    return oracle.attention(q, K, V, pos + 1).reshape(-1)


# (n_q, n_kv, max_pos, [(pos, seed), ...]): each case's calls run in a row; the
# second and third calls of the first case follow a large context with small ones
CASES = [(32, 8, 2048, [(1900, 71), (17, 72), (0, 73)]),
         (16, 2, 2048, [(2047, 81), (5, 82)])]


@pytest.mark.parametrize("n_q,n_kv,max_pos,calls", CASES)
def test_noalloc_matches_allocating_entry_point_and_oracle(lib, n_q, n_kv, max_pos, calls):
    import torch
    for pos, seed in calls:
        qkv, qn, kn, K, V = _inputs(n_q, n_kv, max_pos, seed)
        dq, dqn, dkn = _dev(qkv), _dev(qn), _dev(kn)
        k_a, v_a, k_b, v_b = _dev(K.copy()), _dev(V.copy()), _dev(K.copy()), _dev(V.copy())
        out_a = torch.full((n_q * D,), float("nan"), dtype=torch.float32, device="cuda")
        out_b = torch.full((n_q * D,), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(lib, "tts_attention_decode", dq, dqn, dkn, k_a, v_a, out_a, n_q, n_kv, max_pos, pos) == 0
        assert _call(lib, "tts_attention_decode_noalloc", dq, dqn, dkn, k_b, v_b, out_b, n_q, n_kv, max_pos,
                     pos) == 0
        assert torch.equal(out_a, out_b), f"pos {pos}: max diff {(out_a - out_b).abs().max().item()}"
        assert torch.equal(k_a, k_b) and torch.equal(v_a, v_b)
        ref = _oracle_attention(qkv.astype(np.float64), qn, kn, K, V, n_q, n_kv, pos)
        got = out_b.cpu().numpy().astype(np.float64)
        assert np.allclose(got, ref, rtol=1e-3, atol=2e-3), f"pos {pos}: {np.abs(got - ref).max()}"


def test_noalloc_rejects_oversized_request(lib):
    import torch
    z = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 64 query heads at max_pos 65536 need more than the 2 MiB static array
    rc = _call(lib, "tts_attention_decode_noalloc", z, z, z, z, z, z, 64, 8, 65536, 10)
    assert rc == -1
