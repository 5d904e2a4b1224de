"""Python binding of the GB300 batch-1 TTS decode-step library (libtts_decode.so).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI declared in ``include/tts_decode.h``.  PyTorch is used
for device memory and streams.  There is no fallback: importing this package
raises if the CUDA library has not been built, and every call raises
``TtsError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtts_decode.so")

TTS_BF16 = 0
TTS_FP8 = 1

_STATUS = {0: "ok", -1: "bad argument", -2: "code out of range", -3: "context full",
           -4: "CUDA error", -5: "device error flag set", -6: "not initialised", -7: "unsupported"}


class TtsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} -> {status} ({_STATUS.get(status, 'unknown')})")
        self.status = status


class tts_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "inter",
                 "n_codebooks", "cb_vocab", "max_pos")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("precision", ctypes.c_int), ("stream", ctypes.c_void_p), ("options", ctypes.c_int)]


# tts_config.options bits
OPT_SEPARATE_KERNELS = 1
OPT_PREFILL_STEPS = 2


_PP = ctypes.POINTER(ctypes.c_void_p)


class tts_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p)] + \
               [(n, _PP) for n in ("wqkv", "wo", "wgu", "wd", "sqkv", "so", "sgu", "sd",
                                   "ln_in", "ln_post", "q_norm", "k_norm")]


# Every symbol include/tts_decode.h declares, with its ctypes signature.
_I, _VP, _F = ctypes.c_int, ctypes.c_void_p, ctypes.c_float
SIGNATURES = {
    "tts_init": (_I, [ctypes.POINTER(tts_config), ctypes.POINTER(tts_weights), ctypes.POINTER(_VP)]),
    "tts_shutdown": (_I, [_VP]),
    "tts_reset": (_I, [_VP]),
    "tts_prefill": (_I, [_VP, _VP, _I]),
    "tts_decode_step": (_I, [_VP, _VP, _VP]),
    "tts_decode_steps": (_I, [_VP, _I, _VP]),
    "tts_rewind": (_I, [_VP, _I, _I]),
    "tts_set_input": (_I, [_VP, _VP]),
    "tts_set_sampling": (_I, [_VP, ctypes.c_float, ctypes.c_ulonglong]),
    "tts_decode_until_eoc": (_I, [_VP, _I, _VP, _VP]),
    "tts_prefix_save": (_I, [_VP]),
    "tts_set_fp8_scales": (_I, [_VP, _VP]),
    "tts_fp8_calibrate": (_I, [_VP, _I, _VP]),
    "tts_prefix_restore": (_I, [_VP]),
    "tts_set_kv": (_I, [_VP, _VP, _VP, _I, _I]),
    "tts_get_kv": (_I, [_VP, _VP, _VP, _I, _I]),
    "tts_get_logits": (_I, [_VP, _VP]),
    "tts_get_hidden": (_I, [_VP, _VP]),
    "tts_set_frame": (_I, [_VP, _I, _I]),
    "tts_get_state": (_I, [_VP, _VP, _VP, _VP]),
    "tts_last_steps_ms": (_I, [_VP, _VP]),
    "tts_time_gemv": (_I, [_VP, _I, _I, _VP]),
    "tts_trace_step": (_I, [_VP, _VP, _I, _VP, _VP]),
    "tts_debug_layer_states": (_I, [_VP, _VP, _VP, _VP, _I]),
    "tts_gemm_bf16": (_I, [_VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "tts_gemm_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "tts_gemm_tiled": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "tts_debug_prefill_states": (_I, [_VP, _VP, _I, _VP, ctypes.c_longlong]),
    "tts_debug_expire_wait": (_I, [_VP]),
    "tts_quantize_fp8_weight": (_I, [_VP, _I, _I, _VP, _VP, _VP]),
    "tts_attention_decode": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _F, _VP]),
    "tts_attention_decode_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _F, _VP]),
    "tts_status_str": (ctypes.c_char_p, [_I]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtts_decode.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -m ar_decode_step_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _call(name: str, *args) -> None:
    rc = getattr(load(), name)(*args)
    if rc != 0:
        raise TtsError(name, rc)


def status_str(code: int) -> str:
    return load().tts_status_str(code).decode()


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------
# Device weights (torch is only the allocator here)
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _to_dev_u16(a: np.ndarray, device):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device, non_blocking=False)


def gemm_bf16(a_dev, b_dev, c_dev, epi: int = 0, splits: int = 0, stream=None):
    """C = A . B^T on the tensor cores (see tts_gemm_bf16): a_dev [M][K] and
    b_dev [N][K] (epi 2: [2N][K]) bf16 CUDA tensors; c_dev fp32 [M][N]
    (epi 0, 1) or bf16 [M][N] (epi 2); splits 0 lets the library choose the
    K split, n > 0 fixes it."""
    M, K = a_dev.shape
    N = c_dev.shape[1]
    _call("tts_gemm_bf16", a_dev.data_ptr(), b_dev.data_ptr(), c_dev.data_ptr(), M, N, K, epi, splits, stream)


def gemm_fp8(a8_dev, b8_dev, a_scale_dev, b_scale_dev, c_dev, epi: int = 0, stream=None):
    """tts_gemm_fp8: a8_dev [M][K] and b8_dev [N][K] (epi 2: [2N][K]) uint8
    E4M3 CUDA tensors with fp32 scales [M] and [N] (epi 2: [2N]); c_dev fp32
    [M][N] (epi 0, 1) or bf16 [M][N] (epi 2)."""
    M, K = a8_dev.shape
    N = c_dev.shape[1]
    _call("tts_gemm_fp8", a8_dev.data_ptr(), b8_dev.data_ptr(), a_scale_dev.data_ptr(), b_scale_dev.data_ptr(),
          c_dev.data_ptr(), M, N, K, epi, stream)


def gemm_tiled(a_dev, b_dev, c_dev, epi: int, tile_rows: int, tile_cols: int, splits: int,
               a_scale_dev=None, b_scale_dev=None, stream=None):
    """tts_gemm_tiled: tts_gemm_bf16 (uint8 operands with scales: tts_gemm_fp8)
    with an explicit tile of tile_rows (128 or 256) x tile_cols output
    columns and the K range split over `splits` CTAs."""
    M, K = a_dev.shape
    N = c_dev.shape[1]
    fp8 = a_scale_dev is not None
    _call("tts_gemm_tiled", a_dev.data_ptr(), b_dev.data_ptr(), a_scale_dev.data_ptr() if fp8 else None,
          b_scale_dev.data_ptr() if fp8 else None, c_dev.data_ptr(), M, N, K, epi, 1 if fp8 else 0,
          tile_rows, tile_cols, splits, stream)


def quantize_fp8_weight(w_dev, stream=None):
    """Per-row E4M3 quantisation on the GPU; w_dev: int16 (bf16 bits) [N][K].
    Returns (uint8 [N][K], float32 [N]) device tensors."""
    torch = _torch()
    N, K = w_dev.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w_dev.device)
    s = torch.empty((N,), dtype=torch.float32, device=w_dev.device)
    _call("tts_quantize_fp8_weight", w_dev.data_ptr(), N, K, q.data_ptr(), s.data_ptr(),
          stream if stream is not None else None)
    return q, s


def attention_decode(qkv, q_norm, k_norm, k_cache, v_cache, out, n_q: int, n_kv: int, pos: int,
                     eps: float = 1e-6, rope_theta: float = 1e6, stream=None) -> None:
    """tts_attention_decode on torch device tensors (fp32 qkv/out, int16 bf16 bits)."""
    max_pos = k_cache.shape[-2]
    _call("tts_attention_decode", qkv.data_ptr(), q_norm.data_ptr(), k_norm.data_ptr(), k_cache.data_ptr(),
          v_cache.data_ptr(), out.data_ptr(), n_q, n_kv, max_pos, pos, eps, rope_theta, stream)


@dataclass
class Dims:
    n_layers: int = 36
    hidden: int = 2560
    n_q: int = 32
    n_kv: int = 8
    head_dim: int = 128
    inter: int = 9728
    n_cb: int = 8
    cb_vocab: int = 1026
    rms_eps: float = 1e-6
    rope_theta: float = 1e6


class DeviceWeights:
    """Device copies of a weight set.  ``host`` is any object with the
    attributes embed, head, final_norm and per-layer lists wqkv, wo, wgu, wd,
    ln_in, ln_post, q_norm, k_norm holding bf16 bit images (uint16 numpy).
    For FP8 the four projection matrices of each layer are quantised on the
    GPU by tts_quantize_fp8_weight and only the E4M3 copies are kept."""

    def __init__(self, host, precision: int = TTS_BF16, device="cuda"):
        torch = _torch()
        self.precision = precision
        d = lambda a: _to_dev_u16(a, device)
        self.embed, self.head, self.final_norm = d(host.embed), d(host.head), d(host.final_norm)
        self.mats = {n: [] for n in ("wqkv", "wo", "wgu", "wd")}
        self.scales = {n: [] for n in ("wqkv", "wo", "wgu", "wd")}
        for name in ("wqkv", "wo", "wgu", "wd"):
            for m in getattr(host, name):
                t = d(m)
                if precision == TTS_FP8:
                    q, s = quantize_fp8_weight(t)
                    del t
                    self.mats[name].append(q)
                    self.scales[name].append(s)
                else:
                    self.mats[name].append(t)
        self.norms = {n: [d(x) for x in getattr(host, n)] for n in ("ln_in", "ln_post", "q_norm", "k_norm")}
        torch.cuda.synchronize()
        self.n_layers = len(self.mats["wqkv"])

    def struct(self) -> tts_weights:
        L = self.n_layers
        keep = []

        def arr(ts):
            a = (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
            keep.append(a)
            return ctypes.cast(a, _PP)

        w = tts_weights()
        w.embed, w.head, w.final_norm = self.embed.data_ptr(), self.head.data_ptr(), self.final_norm.data_ptr()
        w.wqkv, w.wo, w.wgu, w.wd = (arr(self.mats[n]) for n in ("wqkv", "wo", "wgu", "wd"))
        if self.precision == TTS_FP8:
            w.sqkv, w.so, w.sgu, w.sd = (arr(self.scales[n]) for n in ("wqkv", "wo", "wgu", "wd"))
        w.ln_in, w.ln_post, w.q_norm, w.k_norm = (arr(self.norms[n]) for n in ("ln_in", "ln_post", "q_norm", "k_norm"))
        self._keep = keep
        return w


# ----------------------------------------------------------------------------
# The decoder context
# ----------------------------------------------------------------------------

class Decoder:
    """One tts_ctx: KV cache, scratch and the captured decode-step graph."""

    def __init__(self, dims, weights: DeviceWeights, max_pos: int, stream=None, options: int = 0):
        self.dims = dims
        self.weights = weights
        cfg = tts_config(dims.n_layers, dims.hidden, dims.n_q, dims.n_kv, dims.head_dim, dims.inter,
                         dims.n_cb, dims.cb_vocab, max_pos, dims.rms_eps, dims.rope_theta,
                         weights.precision, stream, options)
        self._cfg = cfg
        self._w = weights.struct()
        self._ctx = ctypes.c_void_p()
        _call("tts_init", ctypes.byref(cfg), ctypes.byref(self._w), ctypes.byref(self._ctx))
        self.max_pos = max_pos

    @property
    def handle(self):
        return self._ctx

    def close(self):
        if self._ctx:
            _call("tts_shutdown", self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        _call("tts_reset", self._ctx)

    def prefill(self, codes: np.ndarray):
        c = np.ascontiguousarray(codes, np.int32)
        _call("tts_prefill", self._ctx, _ptr(c), c.shape[0])

    def decode_step(self, codes_in=None) -> np.ndarray:
        out = np.empty(self.dims.n_cb, np.int32)
        if codes_in is None:
            _call("tts_decode_step", self._ctx, None, _ptr(out))
        else:
            c = np.ascontiguousarray(codes_in, np.int32)
            _call("tts_decode_step", self._ctx, _ptr(c), _ptr(out))
        return out

    def decode_steps(self, n: int) -> np.ndarray:
        out = np.empty((n, self.dims.n_cb), np.int32)
        _call("tts_decode_steps", self._ctx, n, _ptr(out))
        return out

    def set_sampling(self, temperature: float, seed: int = 0):
        """tts_set_sampling: 0 = greedy argmax; > 0 = seeded categorical draws
        from softmax(logits / temperature)."""
        _call("tts_set_sampling", self._ctx, float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF)

    def decode_until_eoc(self, max_frames: int) -> np.ndarray:
        """tts_decode_until_eoc: free-running frames with one frame of
        lookahead until the last codebook's EOC; returns the codes [n][n_cb]."""
        out = np.empty((max_frames, self.dims.n_cb), np.int32)
        n = ctypes.c_int()
        _call("tts_decode_until_eoc", self._ctx, max_frames, _ptr(out), ctypes.byref(n))
        return out[:n.value]

    def set_fp8_scales(self, scales=None):
        """tts_set_fp8_scales: static activation scales [n_layers][4] (0 =
        dynamic for that site), or None for all dynamic."""
        if scales is None:
            _call("tts_set_fp8_scales", self._ctx, None)
            return
        a = np.ascontiguousarray(scales, np.float32).reshape(self.dims.n_layers, 4)
        _call("tts_set_fp8_scales", self._ctx, _ptr(a))

    def fp8_calibrate(self, n_frames: int) -> np.ndarray:
        """tts_fp8_calibrate: per-site amax [n_layers][4] over n_frames
        discarded free-running frames."""
        out = np.zeros((self.dims.n_layers, 4), np.float32)
        _call("tts_fp8_calibrate", self._ctx, n_frames, _ptr(out))
        return out

    def prefix_save(self):
        """tts_prefix_save: snapshot the cache rows [0, pos) and the state."""
        _call("tts_prefix_save", self._ctx)

    def prefix_restore(self):
        """tts_prefix_restore: back to the saved prefix (cache rows and state)."""
        _call("tts_prefix_restore", self._ctx)

    def set_input(self, codes):
        """tts_set_input: the next step's input frame (host codes [n_cb])."""
        c = np.ascontiguousarray(codes, np.int32)
        _call("tts_set_input", self._ctx, _ptr(c))

    def rewind(self, pos: int, t: int = 0):
        _call("tts_rewind", self._ctx, pos, t)

    def set_kv(self, k_dev, v_dev, length: int, len_stride: int | None = None):
        _call("tts_set_kv", self._ctx, k_dev.data_ptr(), v_dev.data_ptr(), length,
              length if len_stride is None else len_stride)

    def get_kv(self, p0: int, p1: int):
        d = self.dims
        shape = (d.n_layers, d.n_kv, p1 - p0, d.head_dim)
        k = np.empty(shape, np.uint16)
        v = np.empty(shape, np.uint16)
        _call("tts_get_kv", self._ctx, _ptr(k), _ptr(v), p0, p1)
        return k, v

    def get_logits(self) -> np.ndarray:
        out = np.empty((self.dims.n_cb, self.dims.cb_vocab), np.float32)
        _call("tts_get_logits", self._ctx, _ptr(out))
        return out

    def get_hidden(self) -> np.ndarray:
        out = np.empty(self.dims.hidden, np.float32)
        _call("tts_get_hidden", self._ctx, _ptr(out))
        return out

    def set_frame(self, t: int, eoc: int = -1):
        _call("tts_set_frame", self._ctx, t, eoc)

    def state(self):
        p, t, e = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _call("tts_get_state", self._ctx, ctypes.byref(p), ctypes.byref(t), ctypes.byref(e))
        return p.value, t.value, e.value

    def time_gemv(self, kind: int, reps: int = 1) -> float:
        """Mean device ms of one launch of projection `kind` (0 QKV, 1 O, 2 gate/up, 3 down, 4 head)."""
        ms = ctypes.c_float()
        _call("tts_time_gemv", self._ctx, kind, reps, ctypes.byref(ms))
        return ms.value

    def trace_step(self, n_sms_max: int = 1024):
        """One decode step with the persistent kernel's phase trace: uint64 ns
        stamps shaped [n_cta][stride]."""
        cap = n_sms_max * (8 + 31 * self.dims.n_layers) + 2 * 4 * 2048
        buf = np.zeros(cap, np.uint64)
        st, nc = ctypes.c_int(), ctypes.c_int()
        _call("tts_trace_step", self._ctx, _ptr(buf), cap, ctypes.byref(st), ctypes.byref(nc))
        n = st.value * nc.value
        self.last_stage_trace = buf[n: n + 2 * 4 * 2048].reshape(2, 2048, 4)
        return buf[:n].reshape(nc.value, st.value)

    def layer_states(self, codes_in=None):
        """One decode step (as decode_step) through the traced step kernel,
        returning (codes, hidden states [n_layers + 1][hidden]): the residual
        stream after the embedding and after each layer."""
        n = (self.dims.n_layers + 1) * self.dims.hidden
        buf = np.zeros(n, np.float32)
        out = np.empty(self.dims.n_cb, np.int32)
        c = None if codes_in is None else np.ascontiguousarray(codes_in, np.int32)
        _call("tts_debug_layer_states", self._ctx, None if c is None else _ptr(c), _ptr(out), _ptr(buf), n)
        return out, buf.reshape(self.dims.n_layers + 1, self.dims.hidden)

    def prefill_states(self, codes):
        """prefill(codes) on the batched path, returning the residual stream of
        every row after the embedding and after each layer: [n_layers + 1][P][hidden]."""
        c = np.ascontiguousarray(codes, np.int32)
        P = c.shape[0]
        n = (self.dims.n_layers + 1) * P * self.dims.hidden
        buf = np.zeros(n, np.float32)
        _call("tts_debug_prefill_states", self._ctx, _ptr(c), P, _ptr(buf), n)
        return buf.reshape(self.dims.n_layers + 1, P, self.dims.hidden)

    def debug_expire_wait(self) -> int:
        """tts_debug_expire_wait: one step launch whose first wait (for the
        embedding, never stored) cannot complete and whose waits give up
        after 1 ms; returns the status code (TTS_ERR_DEVICE, -5, when the
        timeout was detected)."""
        return int(load().tts_debug_expire_wait(self._ctx))

    def last_steps_ms(self) -> float:
        ms = ctypes.c_float()
        _call("tts_last_steps_ms", self._ctx, ctypes.byref(ms))
        return ms.value
