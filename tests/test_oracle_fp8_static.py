"""The oracle's static FP8 activation scales ("Higgs Audio v3 TTS-4B on
FlashRT", FP8 W8A8 and section 5: per-tensor scales calibrated as amax / 448)
and its calibration record, pinned without the GPU: saturation, agreement with
the per-token path when the static scale equals the per-token one, and the
calibration maximum over frames."""
import numpy as np

import oracle
import synth

TINY = synth.Dims(n_layers=2, hidden=64, n_q=4, n_kv=2, head_dim=16, inter=96, n_cb=8, cb_vocab=1026)


def test_static_quant_saturates_and_matches_per_token():
    x = np.array([0.0, 1.0, -2.5, 1000.0, -1e6, 3e-3, 448.0])
    q = oracle.quant_act_static(x, 1.0)
    dec = [oracle.e4m3_decode(int(b)) for b in q]
    assert dec[3] == 448.0 and dec[4] == -448.0 and dec[6] == 448.0  # beyond +-448 s: saturated
    assert dec[0] == 0.0 and dec[1] == 1.0 and dec[2] == -2.5
    # a static scale equal to the per-token one gives the per-token codes
    rng = np.random.default_rng(3)
    v = rng.normal(size=777)
    q_dyn, s_dyn = oracle.quant_act(v)
    assert np.array_equal(oracle.quant_act_static(v, s_dyn), q_dyn)
    # a larger scale quantises x / s: every code decodes to within e4m3 rounding of x / s
    s = 4 * s_dyn
    back = np.array([oracle.e4m3_decode(int(b)) for b in oracle.quant_act_static(v, s)])
    assert np.all(np.abs(back - v / s) <= np.abs(v / s) * 2 ** -4 + 2 ** -9)


def make(weights):
    o = oracle.Oracle(weights, 32, precision=1)
    o.prefill(synth.delayed_prompt_codes(5))
    return o


def test_calibrated_scales_reproduce_the_frame():
    w = synth.make_weights(TINY, gamma_variant=True)
    bos = np.full(TINY.n_cb, 1024, np.int32)
    a = make(w)
    a.start_calibration()
    c1, l1, _ = a.decode_step(bos)
    amax = a.stop_calibration()
    assert amax.shape == (TINY.n_layers, 4) and (amax > 0).all()
    # every site's static scale = that frame's per-token scale: the same frame again
    scales = np.maximum(amax, np.float32(1e-12)) / np.float32(448.0)
    b = make(w)
    b.set_fp8_scales(scales)
    c2, l2, _ = b.decode_step(bos)
    assert np.array_equal(c1, c2) and np.array_equal(l1, l2)
    # halving every scale changes the quantised activations, hence the logits
    c = make(w)
    c.set_fp8_scales(scales / 2)
    _, l3, _ = c.decode_step(bos)
    assert not np.array_equal(l1, l3)


def test_calibration_keeps_the_largest_amax():
    w = synth.make_weights(TINY, gamma_variant=True)
    frames = [np.full(TINY.n_cb, 1024, np.int32)] + list(synth.random_codes(2, seed=2, stream=41))
    each = []
    o = make(w)
    for f in frames:
        o.start_calibration()
        o.decode_step(f)
        each.append(o.stop_calibration())
    p = make(w)
    p.start_calibration()
    for f in frames:
        p.decode_step(f)
    assert np.array_equal(p.stop_calibration(), np.max(np.stack(each), axis=0))
