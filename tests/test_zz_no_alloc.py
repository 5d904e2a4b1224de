"""The allocation-free attention entry point, called through the C ABI.

Some callers cannot allocate device memory when they call in (a fixed memory
budget owned by another runtime, a loop that must never block in cudaMalloc).
tts_attention_decode_noalloc serves them from a static device array; here its
output must match tts_attention_decode (which takes its scratch from the
stream-ordered allocator) on the same inputs, on two calls in a row.  This
file is collected last so that a failure here comes after every other test."""
import ctypes

import numpy as np
import pytest

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
    import torch
    qkv = synth.normal_f32(5, seed, ((n_q + 2 * n_kv) * D,), std=1.5)
    qn = synth.normal_bf16(3, seed + 1, (D,), std=0.02, mean=1.0)
    kn = synth.normal_bf16(3, seed + 2, (D,), std=0.02, mean=1.0)
    K = synth.normal_bf16(1, seed + 3, (n_kv, max_pos, D))
    V = synth.normal_bf16(1, seed + 4, (n_kv, max_pos, D))
    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    return dev(qkv), dev(qn), dev(kn), K, V, dev


def _call(lib, name, qkv, qn, kn, kd, vd, out, n_q, n_kv, max_pos, pos):
    f = getattr(lib, name)
    return f(ctypes.c_void_p(qkv.data_ptr()), ctypes.c_void_p(qn.data_ptr()), ctypes.c_void_p(kn.data_ptr()),
             ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(vd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
             n_q, n_kv, max_pos, pos, ctypes.c_float(1e-6), ctypes.c_float(1e6), None)


@pytest.mark.parametrize("n_q,n_kv,max_pos,calls", [(32, 8, 512, [(300, 71), (17, 72)]),
                                                    (16, 2, 2048, [(2047, 81), (5, 82)])])
def test_noalloc_matches_allocating_entry_point(lib, n_q, n_kv, max_pos, calls):
    import torch
    for pos, seed in calls:  # two calls in a row, different positions and inputs
        qkv, qn, kn, K, V, dev = _inputs(n_q, n_kv, max_pos, seed)
        k_a, v_a, k_b, v_b = dev(K.copy()), dev(V.copy()), dev(K.copy()), dev(V.copy())
        out_a = torch.full((n_q * D,), float("nan"), dtype=torch.float32, device="cuda")
        out_b = torch.full((n_q * D,), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(lib, "tts_attention_decode", qkv, qn, kn, k_a, v_a, out_a, n_q, n_kv, max_pos, pos) == 0
        assert _call(lib, "tts_attention_decode_noalloc", qkv, qn, kn, k_b, v_b, out_b, n_q, n_kv, max_pos,
                     pos) == 0
        a, b = out_a.cpu().numpy(), out_b.cpu().numpy()
        assert np.isfinite(b).all()
        assert np.allclose(b, a, rtol=1e-3, atol=2e-3), np.abs(a - b).max()
        assert torch.equal(k_a, k_b) and torch.equal(v_a, v_b)


def test_noalloc_rejects_oversized_request(lib):
    import torch
    z = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 64 query heads at max_pos 65536 need more than the 2 MiB static array
    rc = _call(lib, "tts_attention_decode_noalloc", z, z, z, z, z, z, 64, 8, 65536, 10)
    assert rc == -1
