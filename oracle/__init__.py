"""CPU oracle for the batch-1 decode step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It wraps ``oracle.c`` (plain C, fp64) through
ctypes and shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (fp64, no FMA contraction, OpenMP)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_layers", "hidden", "n_q", "n_kv", "head_dim", "inter", "n_cb", "cb_vocab", "max_pos")] + \
               [("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double), ("precision", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class _Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p)] + \
               [(n, _PP) for n in ("wqkv", "wo", "wgu", "wd", "qqkv", "qo", "qgu", "qd",
                                   "sqkv", "so", "sgu", "sd", "ln_in", "ln_post", "q_norm", "k_norm")] + \
               [("act_scales", ctypes.c_void_p)]


class _State(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_int),
                ("t", ctypes.c_int), ("eoc", ctypes.c_int), ("amax_acc", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i32, dbl, flt = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float
            sig = {
                "or_bf16_to_f64": (dbl, [ctypes.c_uint16]),
                "or_f64_to_bf16": (ctypes.c_uint16, [dbl]),
                "or_f32_to_bf16": (ctypes.c_uint16, [flt]),
                "or_e4m3_decode": (dbl, [ctypes.c_uint8]),
                "or_e4m3_encode": (ctypes.c_uint8, [flt]),
                "or_rmsnorm": (None, [vp, vp, i32, dbl, vp]),
                "or_linear_bf16": (None, [vp, i32, i32, vp, vp]),
                "or_quant_act": (None, [vp, i32, vp, vp]),
                "or_quant_act_static": (None, [vp, i32, flt, vp]),
                "or_linear_fp8": (None, [vp, vp, i32, i32, vp, flt, vp]),
                "or_quant_weight": (None, [vp, i32, i32, vp, vp]),
                "or_rope": (None, [vp, i32, i32, dbl]),
                "or_silu": (dbl, [dbl]),
                "or_attention": (None, [vp, vp, vp, i32, i32, i32, i32, i32, vp]),
                "or_embed": (None, [vp, i32, i32, i32, vp, vp]),
                "or_argmax": (i32, [vp, i32]),
                "or_delay_code": (i32, [i32, i32, i32, i32, i32]),
                "or_philox4x32_10": (None, [vp, vp, vp]),
                "or_sample_code": (i32, [vp, i32, dbl, ctypes.c_uint64, i32, i32, vp]),
                "or_decode_step": (i32, [ctypes.POINTER(_Dims), ctypes.POINTER(_Weights),
                                         ctypes.POINTER(_State), vp, vp, vp, vp]),
                "or_prefill": (i32, [ctypes.POINTER(_Dims), ctypes.POINTER(_Weights),
                                     ctypes.POINTER(_State), vp, i32, i32]),
                "or_layer": (i32, [ctypes.POINTER(_Dims), ctypes.POINTER(_Weights),
                                   ctypes.POINTER(_State), i32, i32, vp, i32]),
                "or_head": (i32, [ctypes.POINTER(_Dims), ctypes.POINTER(_Weights),
                                  ctypes.POINTER(_State), vp, vp, vp, vp]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# ---- thin wrappers over the building blocks (used by the pin tests) ----

def bf16_to_f64(bits: int) -> float:
    return lib().or_bf16_to_f64(int(bits))


def f64_to_bf16(x: float) -> int:
    return lib().or_f64_to_bf16(float(x))


def f32_to_bf16(x: float) -> int:
    return lib().or_f32_to_bf16(float(x))


def e4m3_decode(b: int) -> float:
    return lib().or_e4m3_decode(int(b))


def e4m3_encode(x: float) -> int:
    return lib().or_e4m3_encode(float(x))


def rmsnorm(x: np.ndarray, gamma_bf16: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    g = np.ascontiguousarray(gamma_bf16, np.uint16)
    y = np.empty_like(x)
    lib().or_rmsnorm(_p(x), _p(g), x.size, eps, _p(y))
    return y


def linear_bf16(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, np.uint16)
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty(W.shape[0], np.float64)
    lib().or_linear_bf16(_p(W), W.shape[0], W.shape[1], _p(x), _p(y))
    return y


def quant_act(x: np.ndarray):
    x = np.ascontiguousarray(x, np.float64)
    q = np.empty(x.size, np.uint8)
    s = ctypes.c_float()
    lib().or_quant_act(_p(x), x.size, _p(q), ctypes.addressof(s))
    return q, s.value


def quant_act_static(x: np.ndarray, scale: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    q = np.empty(x.size, np.uint8)
    lib().or_quant_act_static(_p(x), x.size, float(scale), _p(q))
    return q


def linear_fp8(W8: np.ndarray, sw: np.ndarray, a8: np.ndarray, sa: float) -> np.ndarray:
    W8 = np.ascontiguousarray(W8, np.uint8)
    sw = np.ascontiguousarray(sw, np.float32)
    a8 = np.ascontiguousarray(a8, np.uint8)
    y = np.empty(W8.shape[0], np.float64)
    lib().or_linear_fp8(_p(W8), _p(sw), W8.shape[0], W8.shape[1], _p(a8), float(sa), _p(y))
    return y


def quant_weight(W: np.ndarray):
    W = np.ascontiguousarray(W, np.uint16)
    q = np.empty(W.shape, np.uint8)
    s = np.empty(W.shape[0], np.float32)
    lib().or_quant_weight(_p(W), W.shape[0], W.shape[1], _p(q), _p(s))
    return q, s


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    y = np.array(x, np.float64, copy=True)
    lib().or_rope(_p(y), y.size, int(pos), float(theta))
    return y


def silu(z: float) -> float:
    return lib().or_silu(float(z))


def attention(q: np.ndarray, Kc: np.ndarray, Vc: np.ndarray, length: int) -> np.ndarray:
    """q [n_q][D] fp64; Kc, Vc bf16 bits [n_kv][max_pos][D]."""
    q = np.ascontiguousarray(q, np.float64)
    Kc = np.ascontiguousarray(Kc, np.uint16)
    Vc = np.ascontiguousarray(Vc, np.uint16)
    n_q, D = q.shape
    n_kv, max_pos, _ = Kc.shape
    out = np.empty((n_q, D), np.float64)
    lib().or_attention(_p(q), _p(Kc), _p(Vc), n_q, n_kv, D, max_pos, int(length), _p(out))
    return out


def embed(E: np.ndarray, codes) -> np.ndarray:
    E = np.ascontiguousarray(E, np.uint16)
    c = np.ascontiguousarray(codes, np.int32)
    x = np.empty(E.shape[2], np.float64)
    lib().or_embed(_p(E), E.shape[0], E.shape[1], E.shape[2], _p(c), _p(x))
    return x


def argmax(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, np.float64)
    return lib().or_argmax(_p(v), v.size)


def delay_code(k: int, t: int, eoc: int, am: int, V: int = 1026) -> int:
    return lib().or_delay_code(k, t, eoc, am, V)


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, np.uint32)
    kk = np.ascontiguousarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().or_philox4x32_10(_p(c), _p(kk), _p(out))
    return [int(x) for x in out]


def sample_code(logits, T: float, seed: int, t: int, k: int):
    """(code, margin): the temperature draw of one codebook, and how far
    u * total lies from the nearest running sum (relative to the total)."""
    v = np.ascontiguousarray(logits, np.float64)
    m = np.zeros(1, np.float64)
    c = lib().or_sample_code(_p(v), v.size, float(T), int(seed) & 0xFFFFFFFFFFFFFFFF, t, k, _p(m))
    return c, float(m[0])


# ---- the whole step ----

class Oracle:
    """Holds a model (host bf16 images from ``synth.make_weights``), its own
    FP8 quantisation when precision == 1, and a KV cache."""

    def __init__(self, weights, max_pos: int, precision: int = 0, share: "Oracle" = None):
        """share: another Oracle of the same weights and precision whose FP8
        weight quantisation this one reuses (saves the quantisation pass and
        its memory; each instance keeps its own cache and state)."""
        d = weights.dims
        self.dims = d
        self.w = weights
        self.max_pos = max_pos
        self.precision = precision
        L = d.n_layers
        self._keep = []
        self.cdims = _Dims(d.n_layers, d.hidden, d.n_q, d.n_kv, d.head_dim, d.inter, d.n_cb,
                           d.cb_vocab, max_pos, d.rms_eps, d.rope_theta, precision)

        def parr(arrs):
            a = (ctypes.c_void_p * L)(*[_p(x) for x in arrs])
            self._keep.append(a)
            return ctypes.cast(a, _PP)

        cw = _Weights()
        cw.embed, cw.head, cw.final_norm = _p(weights.embed), _p(weights.head), _p(weights.final_norm)
        cw.wqkv, cw.wo, cw.wgu, cw.wd = (parr(weights.wqkv), parr(weights.wo),
                                         parr(weights.wgu), parr(weights.wd))
        if precision == 1:
            if share is not None:
                assert share.w is weights and share.precision == 1
                self.q = share.q
            else:
                self.q = {}
                for name in ("wqkv", "wo", "wgu", "wd"):
                    self.q[name] = [quant_weight(m) for m in getattr(weights, name)]
            cw.qqkv, cw.qo, cw.qgu, cw.qd = (parr([x[0] for x in self.q[n]])
                                             for n in ("wqkv", "wo", "wgu", "wd"))
            cw.sqkv, cw.so, cw.sgu, cw.sd = (parr([x[1] for x in self.q[n]])
                                             for n in ("wqkv", "wo", "wgu", "wd"))
        cw.ln_in, cw.ln_post = parr(weights.ln_in), parr(weights.ln_post)
        cw.q_norm, cw.k_norm = parr(weights.q_norm), parr(weights.k_norm)
        self.cw = cw
        shape = (L, d.n_kv, max_pos, d.head_dim)
        self.k = np.zeros(shape, np.uint16)
        self.v = np.zeros(shape, np.uint16)
        self.st = _State(_p(self.k), _p(self.v), 0, 0, -1, None)
        self._scales = None
        self._amax = None

    # state
    @property
    def pos(self):
        return self.st.pos

    def reset(self):
        self.st.pos, self.st.t, self.st.eoc = 0, 0, -1

    def set_fp8_scales(self, scales=None):
        """Static activation scales [n_layers][4] (precision 1; 0 = per-token
        for that site), or None for per-token everywhere."""
        if scales is None:
            self._scales = None
            self.cw.act_scales = None
        else:
            self._scales = np.ascontiguousarray(scales, np.float32).reshape(self.dims.n_layers, 4)
            self.cw.act_scales = _p(self._scales)

    def start_calibration(self):
        """Record the largest input amax of every activation site from now on."""
        self._amax = np.zeros((self.dims.n_layers, 4), np.float32)
        self.st.amax_acc = _p(self._amax)

    def stop_calibration(self) -> np.ndarray:
        self.st.amax_acc = None
        a, self._amax = self._amax, None
        return a

    def set_frame(self, t: int, eoc: int = -1):
        self.st.t, self.st.eoc = t, eoc

    def set_kv(self, k: np.ndarray, v: np.ndarray, length: int):
        """Copy a [L][n_kv][>=length][D] bf16 prefix into the cache and set pos."""
        self.k[:, :, :length] = k[:, :, :length]
        self.v[:, :, :length] = v[:, :, :length]
        self.st.pos = length

    def decode_step(self, codes_in):
        c = np.ascontiguousarray(codes_in, np.int32)
        out = np.empty(self.dims.n_cb, np.int32)
        logits = np.empty((self.dims.n_cb, self.dims.cb_vocab), np.float64)
        gaps = np.empty(self.dims.n_cb, np.float64)
        rc = lib().or_decode_step(ctypes.byref(self.cdims), ctypes.byref(self.cw),
                                  ctypes.byref(self.st), _p(c), _p(out), _p(logits), _p(gaps))
        if rc:
            raise ValueError(f"or_decode_step failed ({rc})")
        return out, logits, gaps

    def embed(self, codes_in) -> np.ndarray:
        """The step's input residual stream for these codes."""
        return embed(self.w.embed, codes_in)

    def layer(self, layer: int, pos: int, h, a16: bool = False) -> np.ndarray:
        """Layer `layer` at position pos applied to the residual stream h
        (returns the layer's output; writes that layer's K/V at pos).  a16 as
        in prefill."""
        x = np.ascontiguousarray(h, np.float64).copy()
        rc = lib().or_layer(ctypes.byref(self.cdims), ctypes.byref(self.cw), ctypes.byref(self.st),
                            int(layer), int(pos), _p(x), int(a16))
        if rc:
            raise ValueError(f"or_layer failed ({rc})")
        return x

    def head(self, h):
        """(codes, logits, gaps) of the head on the final residual stream h at
        the current frame (no state change)."""
        x = np.ascontiguousarray(h, np.float64)
        out = np.empty(self.dims.n_cb, np.int32)
        logits = np.empty((self.dims.n_cb, self.dims.cb_vocab), np.float64)
        gaps = np.empty(self.dims.n_cb, np.float64)
        rc = lib().or_head(ctypes.byref(self.cdims), ctypes.byref(self.cw), ctypes.byref(self.st), _p(x),
                           _p(out), _p(logits), _p(gaps))
        if rc:
            raise ValueError(f"or_head failed ({rc})")
        return out, logits, gaps

    def prefill(self, codes, a16: bool = False):
        c = np.ascontiguousarray(codes, np.int32)
        rc = lib().or_prefill(ctypes.byref(self.cdims), ctypes.byref(self.cw),
                              ctypes.byref(self.st), _p(c), c.shape[0], int(a16))
        if rc:
            raise ValueError(f"or_prefill failed ({rc})")
