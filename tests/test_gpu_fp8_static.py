"""Static FP8 activation scales and the calibration run on the GPU
(tts_set_fp8_scales, tts_fp8_calibrate; "Higgs Audio v3 TTS-4B on FlashRT",
FP8 W8A8 and section 5) against the oracle.  The scales the parity frames use
come from the oracle's own calibration, never from the GPU; the GPU's
calibration is compared with the oracle's record of the same frame."""
import numpy as np
import pytest

import oracle
import synth
from helpers import check_frame, reduced_dims, to_binding_dims

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ads():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import ar_decode_step_gb300.build as b
    b.build()
    import ar_decode_step_gb300 as m
    m.load()
    return m


@pytest.fixture(scope="module")
def model():
    d = reduced_dims(2)
    return d, synth.make_weights(d, gamma_variant=True)


PROMPT = synth.delayed_prompt_codes(5)


def pair(ads, d, w):
    dw = ads.DeviceWeights(w, precision=1)
    dec = ads.Decoder(to_binding_dims(d), dw, 32)
    dec.prefill(PROMPT)
    orc = oracle.Oracle(w, 32, precision=1)
    orc.prefill(PROMPT)
    return dec, dw, orc


def test_calibration_matches_oracle_and_leaves_state(ads, model):
    d, w = model
    dec, dw, orc = pair(ads, d, w)
    before = dec.state()
    amax = dec.fp8_calibrate(1)  # the next frame: all-BOS input after the prompt
    assert dec.state() == before
    orc.start_calibration()
    orc.decode_step(np.full(d.n_cb, 1024, np.int32))
    ref = orc.stop_calibration()
    assert np.allclose(amax, ref, rtol=2e-2, atol=0), (amax, ref)
    # the discarded frame does not change what the next real frame computes
    fresh, fw, _ = pair(ads, d, w)
    assert np.array_equal(dec.decode_steps(2), fresh.decode_steps(2))
    dec.close()
    fresh.close()


def test_static_scales_parity(ads, model):
    d, w = model
    # scales: the oracle's calibration over three frames, with 25 % headroom
    cal = oracle.Oracle(w, 32, precision=1)
    cal.prefill(PROMPT)
    frames = [np.full(d.n_cb, 1024, np.int32)] + list(synth.random_codes(2, seed=2, stream=42))
    cal.start_calibration()
    for f in frames:
        cal.decode_step(f)
    scales = (cal.stop_calibration() * np.float32(1.25)) / np.float32(448.0)
    dec, dw, orc = pair(ads, d, w)
    dec.set_fp8_scales(scales)
    orc.set_fp8_scales(scales)
    checked = 0
    for f, cin in enumerate(synth.random_codes(4, seed=2, stream=43)):
        t, eoc = orc.st.t, orc.st.eoc
        g = dec.decode_step(cin)
        o_codes, o_logits, o_gaps = orc.decode_step(cin)
        checked += check_frame(g, dec.get_logits(), o_codes, o_logits, o_gaps, True, t, eoc, f"static frame {f}")[2]
    assert checked >= 20
    # all sites dynamic again: the frames of a context that never had scales
    dec.set_fp8_scales(None)
    plain, pw, _ = pair(ads, d, w)
    dec.rewind(5)
    assert np.array_equal(dec.decode_steps(2), plain.decode_steps(2))
    dec.close()
    plain.close()


def test_static_scale_errors(ads, model):
    d, w = model
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, 16)
    with pytest.raises(ads.TtsError):
        dec.set_fp8_scales(np.ones((d.n_layers, 4)))  # a BF16 context
    with pytest.raises(ads.TtsError):
        dec.fp8_calibrate(1)
    dec.close()
    dec8, dw8, _ = pair(ads, d, w)
    bad = np.ones((d.n_layers, 4), np.float32)
    bad[1, 2] = -1.0
    with pytest.raises(ads.TtsError):
        dec8.set_fp8_scales(bad)
    dec8.close()
