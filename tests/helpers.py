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
