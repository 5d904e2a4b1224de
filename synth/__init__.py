"""Seeded synthetic inputs for the decode step: weights, KV prefixes and codes.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It holds no arithmetic of the decode step itself: it only draws
numbers (Philox4x32-10 counter-based generator, Box-Muller normals; see
``synth.c``) and lays them out in the tensor shapes the model uses.

Seeds (one per kind of input): weights 0, KV prefix 1, codes 2, norm-gain
variant 3.  Every tensor has its own Philox stream id, so tensors do not
overlap and any one of them can be regenerated alone.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

SEED_WEIGHTS = 0
SEED_KV = 1
SEED_CODES = 2
SEED_GAMMA = 3

BOS = 1024  # BOS-pad code
EOC = 1025  # end-of-codes code
N_ACOUSTIC = 1024  # ordinary acoustic codes are 0..1023


def build(force: bool = False) -> str:
    """Compile libsynth.so with gcc (OpenMP) if it is missing or stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.synth_normal_f32.argtypes = [u64, u64, dbl, dbl, vp, i64]
            lib.synth_normal_bf16.argtypes = [u64, u64, dbl, dbl, vp, i64]
            lib.synth_normal_bf16_strided.argtypes = [u64, u64, dbl, dbl, vp, i64, i64, i64]
            lib.synth_uniform_int.argtypes = [u64, u64, i32, i32, vp, i64]
            lib.synth_raw_u32.argtypes = [u64, u64, u64, vp]
            for f in (lib.synth_normal_f32, lib.synth_normal_bf16, lib.synth_normal_bf16_strided,
                      lib.synth_uniform_int, lib.synth_raw_u32):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def raw_u32(seed: int, stream: int, idx: int) -> np.ndarray:
    out = np.zeros(4, np.uint32)
    _load().synth_raw_u32(seed, stream, idx, _ptr(out))
    return out


def normal_f32(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().synth_normal_f32(seed, stream, mean, std, _ptr(out), out.size)
    return out


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0,
                out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit images (uint16) of N(mean, std) draws."""
    if out is None:
        out = np.empty(shape, np.uint16)
    assert out.dtype == np.uint16 and out.size == int(np.prod(shape))
    _load().synth_normal_bf16(seed, stream, mean, std, _ptr(out), out.size)
    return out


def normal_bf16_rows(seed: int, stream: int, rows: int, cols: int, out: np.ndarray,
                     std: float = 1.0) -> None:
    """Write a [rows][cols] bf16 N(0, std) tensor into the leading rows of a
    row-strided 2-D view ``out`` (its row stride may exceed ``cols``)."""
    assert out.dtype == np.uint16 and out.ndim == 2 and out.strides[1] == 2
    ld = out.strides[0] // 2
    _load().synth_normal_bf16_strided(seed, stream, 0.0, std, out.ctypes.data, rows, cols, ld)


def uniform_int(seed: int, stream: int, shape, lo: int, hi: int) -> np.ndarray:
    out = np.empty(shape, np.int32)
    _load().synth_uniform_int(seed, stream, lo, hi, _ptr(out), out.size)
    return out


# ----------------------------------------------------------------------------
# Model-shaped inputs
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Dims:
    """Backbone dimensions.  The defaults are the Qwen3-4B-shaped backbone."""
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

    @property
    def qkv_rows(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    @property
    def attn_dim(self) -> int:
        return self.n_q * self.head_dim


FULL = Dims()


# Philox stream ids: global tensors below 16, per-layer tensors at 16 + 16*layer + kind.
_S_EMBED, _S_HEAD, _S_FINAL_NORM = 1, 2, 3
_K_WQKV, _K_WO, _K_WGU, _K_WD, _K_LN_IN, _K_LN_POST, _K_QN, _K_KN = range(8)
_K_KCACHE, _K_VCACHE = 8, 9


def _lstream(layer: int, kind: int) -> int:
    return 16 + 16 * layer + kind


@dataclass
class Weights:
    """Host bf16 bit images (uint16) of every weight tensor, row-major [out][in].

    wqkv rows: q heads (h*D+d), then k heads, then v heads.
    wgu rows: the gate matrix [inter][hidden] followed by the up matrix.
    head rows: codebook k, code v at row k*cb_vocab + v.
    """
    dims: Dims
    embed: np.ndarray                      # [n_cb][cb_vocab][hidden]
    head: np.ndarray                       # [n_cb*cb_vocab][hidden]
    final_norm: np.ndarray                 # [hidden]
    wqkv: list = field(default_factory=list)
    wo: list = field(default_factory=list)
    wgu: list = field(default_factory=list)
    wd: list = field(default_factory=list)
    ln_in: list = field(default_factory=list)
    ln_post: list = field(default_factory=list)
    q_norm: list = field(default_factory=list)
    k_norm: list = field(default_factory=list)


BF16_ONE = np.uint16(0x3F80)


def make_weights(d: Dims, seed: int = SEED_WEIGHTS, std: float = 0.02,
                 gamma_variant: bool = False) -> Weights:
    """Matrices and embeddings ~ N(0, std) from ``seed``; norm gains are ones,
    or 1 + N(0, 0.02) drawn from seed 3 when ``gamma_variant`` is set."""
    H, D = d.hidden, d.head_dim

    def gamma(stream, n):
        if gamma_variant:
            return normal_bf16(SEED_GAMMA, stream, (n,), std=0.02, mean=1.0)
        return np.full((n,), BF16_ONE, np.uint16)

    w = Weights(
        dims=d,
        embed=normal_bf16(seed, _S_EMBED, (d.n_cb, d.cb_vocab, H), std),
        head=normal_bf16(seed, _S_HEAD, (d.n_cb * d.cb_vocab, H), std),
        final_norm=gamma(_S_FINAL_NORM, H),
    )
    for l in range(d.n_layers):
        w.wqkv.append(normal_bf16(seed, _lstream(l, _K_WQKV), (d.qkv_rows, H), std))
        w.wo.append(normal_bf16(seed, _lstream(l, _K_WO), (H, d.attn_dim), std))
        w.wgu.append(normal_bf16(seed, _lstream(l, _K_WGU), (2 * d.inter, H), std))
        w.wd.append(normal_bf16(seed, _lstream(l, _K_WD), (H, d.inter), std))
        w.ln_in.append(gamma(_lstream(l, _K_LN_IN), H))
        w.ln_post.append(gamma(_lstream(l, _K_LN_POST), H))
        w.q_norm.append(gamma(_lstream(l, _K_QN), D))
        w.k_norm.append(gamma(_lstream(l, _K_KN), D))
    return w


def make_kv_prefix(d: Dims, length: int, max_pos: int, seed: int = SEED_KV):
    """K and V caches [n_layers][n_kv][max_pos][head_dim] (bf16 bits) whose first
    ``length`` positions hold N(0, 1) draws; later positions are zero."""
    shape = (d.n_layers, d.n_kv, max_pos, d.head_dim)
    k = np.zeros(shape, np.uint16)
    v = np.zeros(shape, np.uint16)
    for l in range(d.n_layers):
        for j in range(d.n_kv):
            if length:
                normal_bf16_rows(seed, _lstream(l, _K_KCACHE) * 64 + j, length, d.head_dim, k[l, j])
                normal_bf16_rows(seed, _lstream(l, _K_VCACHE) * 64 + j, length, d.head_dim, v[l, j])
    return k, v


def random_codes(n_frames: int, n_cb: int = 8, seed: int = SEED_CODES, stream: int = 0) -> np.ndarray:
    """Uniform acoustic codes in [0, 1024), shape [n_frames][n_cb]."""
    return uniform_int(seed, 100 + stream, (n_frames, n_cb), 0, N_ACOUSTIC)


def delayed_prompt_codes(P: int, n_cb: int = 8, seed: int = SEED_CODES, stream: int = 0) -> np.ndarray:
    """Prompt codes under the delay pattern: codebook k is BOS-pad (1024) at
    positions p < k, otherwise a uniform acoustic code.  Shape [P][n_cb]."""
    c = uniform_int(seed, 200 + stream, (P, n_cb), 0, N_ACOUSTIC)
    for k in range(n_cb):
        c[: min(k, P), k] = BOS
    return c
