"""How far fp32 arithmetic moves the 36-layer FP8 W8A8 step from the oracle.

The oracle evaluates the step in fp64; each FP8 projection's sum is exact
there (every e4m3 product and partial sum of a row fits 53 bits).  A GPU
computes in fp32.  The float32 restatement in fp8_restatement.py computes the
same step in three variants: projection sums taken exactly (so only the fp32
rounding of norms, attention, SwiGLU and residual adds remains), in BLAS
order, and in a GPU-like chunked order.  Through one or two layers every
variant agrees with the oracle to the bf16 output rounding.  Over the 36
full-width layers of the FP8 benchmark model, the bf16-rounded projection
outputs and the per-token E4M3 re-quantisation of every layer amplify any
rounding difference: a flipped E4M3 code moves an activation by 6-12 %, which
flips further bf16 and E4M3 roundings downstream.  Every variant -- even with
exact sums -- then misses the 0.999 logits cosine bar on some frames.  The
GPU's full-depth FP8 frames are held to this measured spread instead
(test_gpu_full.py), and its layers to the strict per-layer bar.  No GPU."""
import numpy as np
import pytest

import oracle
import synth
from fp8_restatement import ORDERS, Fp8Fp32Step, frame_stats, layerwise_spread
from helpers import reduced_dims

FRAMES = 4
KV = 1024


def teacher_forced_inputs(n_cb: int, frames: int):
    """All-BOS, then seeded random codes (the inputs test_gpu_full uses)."""
    return [np.full(n_cb, 1024, np.int32)] + list(synth.random_codes(frames - 1, seed=2, stream=9))


def test_restatement_matches_oracle_through_two_layers():
    """At tiny width and two layers every order agrees with the oracle to the
    bf16 output rounding: the restatement is the same step."""
    d = synth.Dims(n_layers=2, hidden=256, n_q=4, n_kv=2, head_dim=128, inter=512)
    w = synth.make_weights(d, gamma_variant=True)
    max_pos = 24
    k, v = synth.make_kv_prefix(d, 16, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=1)
    orc.set_kv(k, v, 16)
    refs = []
    for order in ORDERS:
        r = Fp8Fp32Step(w, max_pos, order)
        r.set_kv(k, v, 16)
        refs.append(r)
    for cin in teacher_forced_inputs(d.n_cb, 3):
        o, ol, og = orc.decode_step(cin)
        for r in refs:
            c, lg = r.step(cin)
            cos, n, bad = frame_stats(lg, ol, c, o, og)
            assert cos > 0.9999, (r.order, cos)
            assert bad == 0, (r.order, c, o)


@pytest.fixture(scope="module")
def full36():
    d = synth.Dims(n_layers=36)
    return d, synth.make_weights(d)


def measure_spread(w, d, frames: int):
    """Per order, per teacher-forced frame: (cos, codes checked, codes
    differing) of the float32 restatement against the oracle, at the FP8
    benchmark workload (36 layers, 1024 cached positions of N(0, 1) K/V)."""
    max_pos = KV + frames + 1
    k, v = synth.make_kv_prefix(d, KV, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=1)
    orc.set_kv(k, v, KV)
    refs = {}
    for order in ORDERS:
        refs[order] = Fp8Fp32Step(w, max_pos, order, share=refs.get(ORDERS[0]))
        refs[order].set_kv(k, v, KV)
    stats = {o: [] for o in ORDERS}
    for cin in teacher_forced_inputs(d.n_cb, frames):
        o, ol, og = orc.decode_step(cin)
        for order, r in refs.items():
            c, lg = r.step(cin)
            stats[order].append(frame_stats(lg, ol, c, o, og))
    return stats


def test_fp32_order_spread_at_36_layers(full36):
    """The reading that FP8 parity at full depth is checked against the
    spread of fp32 implementations, not the 0.999 bar: the exact-sum variant
    (fp32 only outside the projection sums) already misses the bar on some
    frame, none falls apart (cos stays above 0.95), and codes with a clear
    top-2 gap mostly still agree."""
    d, w = full36
    stats = measure_spread(w, d, FRAMES)
    for order, s in stats.items():
        print(f"fp32 order {order:10s}: cos " + " ".join(f"{c:.5f}" for c, _, _ in s) +
              f"; codes differing {sum(b for _, _, b in s)} of {sum(n for _, n, _ in s)}")
    worst = min(c for s in stats.values() for c, _, _ in s)
    assert min(c for c, _, _ in stats["exact"]) < 0.999, \
        "fp32 outside the sums met the 0.999 bar: hold the GPU to it at frame level"
    assert worst > 0.95
    checked = sum(n for s in stats.values() for _, n, _ in s)
    differing = sum(b for s in stats.values() for _, _, b in s)
    assert differing <= 0.25 * checked


def test_fp32_spread_of_the_batched_fp8_prefill_rows():
    """The FP8 prefill check's reading: 480 prompt rows after 24 cached
    positions at reduced width (2 layers), each row's layer contribution
    compared with the oracle's layer from the same input (the protocol of
    test_gpu_prefill.py).  The float32 restatement -- even with exact
    projection sums -- leaves some rows below 0.999: the per-row bar cannot
    be the plain 0.999, it is the measured spread."""
    d = reduced_dims(2)
    w = synth.make_weights(d, gamma_variant=True)
    P, prefix = 480, 24
    max_pos = prefix + P + 4
    prompt = synth.delayed_prompt_codes(P, stream=7)
    k, v = synth.make_kv_prefix(d, prefix, max_pos)
    r = Fp8Fp32Step(w, max_pos, "exact")
    r.set_kv(k, v, prefix)
    orc = oracle.Oracle(w, max_pos, precision=1)
    orc.set_kv(k, v, prefix)
    rows = []
    for p in range(P):
        rows.append([h.numpy() for h in r.layer_states(prompt[p])])
        r.pos += 1
    R = layerwise_spread(orc, rows, prefix, d.n_layers)
    print(f"fp32 prefill rows: min {R.min():.6f} mean {R.mean():.7f} below 0.999: {(R < 0.999).sum()}")
    assert R.min() < 0.999
    assert R.min() > 0.995 and R.mean() > 0.9995
