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
    cfg = m.tts_config(36, 2560, 32, 8, 128, 9728, 8, 1026, 256, 1e-6, 1e6, 0, None)
    w = m.tts_weights()
    ctx = ctypes.c_void_p()
    # NULL weights
    assert lib.tts_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(ctx)) == -1
    assert lib.tts_init(None, ctypes.byref(w), ctypes.byref(ctx)) == -1
    assert lib.tts_init(ctypes.byref(cfg), ctypes.byref(w), None) == -1
    for field, bad in (("head_dim", 64), ("n_q_heads", 30), ("hidden", 2500), ("max_pos", 0),
                       ("precision", 3), ("n_codebooks", 9), ("inter", 20000)):
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
