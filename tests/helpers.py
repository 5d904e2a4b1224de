"""Shared test helpers: parity metrics and oracle/GPU set-up for one weight set."""
from __future__ import annotations

import numpy as np

import synth

# Acceptance for the decode step's logits: cosine >= 0.9999 and max-abs error
# <= 2e-2 in BF16, cosine >= 0.999 in FP8; codes must match wherever the
# oracle's top-2 logit gap exceeds 1e-2.
BF16_COS, BF16_MAXABS = 0.9999, 2e-2
FP8_COS = 0.999
GAP = 1e-2


def cosine(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def check_frame(gpu_codes, gpu_logits, or_codes, or_logits, or_gaps, fp8: bool, t: int, eoc: int,
                where: str = ""):
    """Assert one frame's parity.  t / eoc: the frame index and EOC frame the
    step ran with (codes the delay mask forces must match exactly).  Returns
    (cos, maxabs, number of codes checked)."""
    gpu_logits = np.asarray(gpu_logits, np.float64).reshape(or_logits.shape)
    cos = cosine(gpu_logits, or_logits)
    maxabs = float(np.abs(gpu_logits - or_logits).max())
    if fp8:
        assert cos >= FP8_COS, f"{where}: cos {cos}"
    else:
        assert cos >= BF16_COS, f"{where}: cos {cos}"
        assert maxabs <= BF16_MAXABS, f"{where}: max-abs {maxabs}"
    n = 0
    for k in range(len(or_codes)):
        forced = t < k or (eoc >= 0 and t >= eoc + k)
        if forced or or_gaps[k] > GAP:
            assert gpu_codes[k] == or_codes[k], (
                f"{where}: codebook {k}: gpu {gpu_codes[k]} oracle {or_codes[k]} gap {or_gaps[k]}")
            n += 1
    return cos, maxabs, n


def reduced_dims(n_layers=2):
    """Smaller backbone with the same structure (G = 4 query heads per kv head)."""
    return synth.Dims(n_layers=n_layers, hidden=512, n_q=8, n_kv=2, head_dim=128, inter=1024,
                      n_cb=8, cb_vocab=1026)


def to_binding_dims(d: synth.Dims):
    import ar_decode_step_gb300 as ads
    return ads.Dims(d.n_layers, d.hidden, d.n_q, d.n_kv, d.head_dim, d.inter, d.n_cb, d.cb_vocab,
                    d.rms_eps, d.rope_theta)


def upload_kv(k: np.ndarray, v: np.ndarray, length: int):
    import torch
    kd = torch.from_numpy(np.ascontiguousarray(k[:, :, :length]).view(np.int16)).cuda()
    vd = torch.from_numpy(np.ascontiguousarray(v[:, :, :length]).view(np.int16)).cuda()
    return kd, vd


def bf16_f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def check_kv_rows(gpu_bits, oracle_bits, where: str = ""):
    """K/V rows written by a W16A16 prefill run end to end on both sides, per
    layer: cosine >= 0.9999 and no entry off by more than 0.1 * max(1,
    |oracle|).  Both sides round every projection input to bf16, so an
    activation that falls on the other side of a bf16 boundary shifts later
    layers' values by about an ulp; the elementwise bar applies layer by layer
    from identical inputs (test_gpu_prefill's layer-level check).  Returns
    (worst cosine, worst scaled error)."""
    worst_cos, worst_err = 1.0, 0.0
    for l in range(gpu_bits.shape[0]):
        a, b = bf16_f64(gpu_bits[l]).ravel(), bf16_f64(oracle_bits[l]).ravel()
        cos = cosine(a, b)
        err = np.abs(a - b) / np.maximum(1.0, np.abs(b))
        tail = float(np.mean(err > BF16_MAXABS))
        assert cos >= BF16_COS, f"{where}: layer {l}: cos {cos}"
        assert err.max() <= 0.1, f"{where}: layer {l}: {tail} beyond 2e-2, max {err.max()}"
        worst_cos, worst_err = min(worst_cos, cos), max(worst_err, float(err.max()))
    return worst_cos, worst_err


def adopt_gpu_cache(dec, orc, length: int):
    """Give the oracle the GPU's K/V rows [0, length): the next decode frames
    are then compared from the same cache (the prefill is checked on its own)."""
    gk, gv = dec.get_kv(0, length)
    orc.k[:, :, :length] = gk
    orc.v[:, :, :length] = gv
