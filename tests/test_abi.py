"""The C-ABI library (no GPU needed): it builds, loads, exports every symbol
include/*.h declares, and rejects bad arguments on the host before any CUDA
call."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import ar_decode_step_gb300.build as b
    b.build()
    import ar_decode_step_gb300 as m
    return m.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(tts_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tts_init", "tts_prefill", "tts_decode_step", "tts_reset", "tts_shutdown",
                     "tts_decode_steps", "tts_quantize_fp8_weight"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    import ar_decode_step_gb300 as m
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in m.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    import ar_decode_step_gb300 as m
    assert m.status_str(0) == "ok"
    assert m.status_str(-3) == "context full"
    assert m.status_str(12345) == "unknown status"


def test_host_validation_rejects_bad_config(lib):
    import ar_decode_step_gb300 as m
    cfg = m.tts_config(36, 2560, 32, 8, 128, 9728, 8, 1026, 256, 1e-6, 1e6, 0, None, 0)
    w = m.tts_weights()
    ctx = ctypes.c_void_p()
    # NULL weights
    assert lib.tts_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(ctx)) == -1
    assert lib.tts_init(None, ctypes.byref(w), ctypes.byref(ctx)) == -1
    assert lib.tts_init(ctypes.byref(cfg), ctypes.byref(w), None) == -1
    for field, bad in (("head_dim", 64), ("n_q_heads", 30), ("hidden", 2500), ("max_pos", 0),
                       ("precision", 3), ("n_codebooks", 9), ("inter", 20000), ("options", 4)):
        c2 = m.tts_config.from_buffer_copy(cfg)
        setattr(c2, field, bad)
        assert lib.tts_init(ctypes.byref(c2), ctypes.byref(w), ctypes.byref(ctx)) == -1, field
    assert not ctx.value


def test_calls_without_context(lib):
    out = np.zeros(8, np.int32)
    assert lib.tts_decode_step(None, None, out.ctypes.data) == -6
    assert lib.tts_decode_steps(None, 1, None) == -6
    assert lib.tts_prefill(None, None, 0) == -6
    assert lib.tts_reset(None) == -6
    assert lib.tts_shutdown(None) == 0
    assert lib.tts_quantize_fp8_weight(None, 4, 4, None, None, None) == -1


def test_gemm_tiled_rejects_bad_tiles_before_any_device_call(lib):
    """Host validation of tts_gemm_tiled: pointers are checked for NULL and
    16-byte alignment, the tile (rows, width, K split, one k-block per
    split) against the shape; none of these reach the device."""
    P = ctypes.c_void_p(0x1000)  # aligned stand-ins, never dereferenced
    f = lib.tts_gemm_tiled
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 8 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    ok_shape = (256, 1024)  # N, K
    bad = [
        (192, 128, 1),   # 192-row tile
        (128, 96, 1),    # width not built
        (256, 128, 5),   # K split over 5
        (128, 64, 17),   # more splits than k-blocks (16)
        (256, 192, 1),   # N = 256 not a multiple of 192
    ]
    for rows, cols, splits in bad:
        assert f(P, P, None, None, P, 64, ok_shape[0], ok_shape[1], 0, 0, rows, cols, splits, None) == -1, (rows, cols)
    # SwiGLU: 128 + 128 columns only, no K split
    assert f(P, P, None, None, P, 64, 256, 1024, 2, 0, 128, 64, 1, None) == -1
    assert f(P, P, None, None, P, 64, 256, 1024, 2, 0, 128, 128, 2, None) == -1
    # E4M3: scales required, K a multiple of 128
    assert f(P, P, None, None, P, 64, 256, 1024, 0, 1, 128, 128, 1, None) == -1
    assert f(P, P, P, P, P, 64, 256, 1088, 0, 1, 128, 128, 1, None) == -1
    # misaligned or NULL operands
    assert f(ctypes.c_void_p(0x1008), P, None, None, P, 64, 256, 1024, 0, 0, 128, 128, 1, None) == -1
    assert f(None, P, None, None, P, 64, 256, 1024, 0, 0, 128, 128, 1, None) == -1
