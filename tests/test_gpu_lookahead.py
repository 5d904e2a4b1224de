"""The lookahead decode loop (tts_decode_until_eoc): it must produce exactly
the frames of the plain device loop (tts_decode_steps), stop after the frame
in which the last codebook emits EOC (the delay pattern's frame eoc + n_cb -
1), undo the frame it queued past the stop, and leave a state from which the
next step continues as if no frame had been queued ahead."""
import numpy as np
import pytest

import synth
from helpers import reduced_dims, to_binding_dims

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
def setup(ads):
    d = reduced_dims(2)
    w = synth.make_weights(d, gamma_variant=True)
    return d, ads.DeviceWeights(w, precision=0)


def decoder(ads, d, dw, eoc):
    dec = ads.Decoder(to_binding_dims(d), dw, 64)
    dec.prefill(synth.delayed_prompt_codes(5))
    dec.set_frame(0, eoc)
    return dec


def test_stops_after_last_codebook_eoc(ads, setup):
    d, dw = setup
    eoc = 3  # codebook k emits EOC from frame 3 + k on: the last one at frame 3 + 7 = 10
    a = decoder(ads, d, dw, eoc)
    got = a.decode_until_eoc(40)
    assert got.shape == (eoc + d.n_cb, d.n_cb)
    assert a.state() == (5 + 11, 11, eoc)
    assert (got[-1] == d.cb_vocab - 1).all()
    b = decoder(ads, d, dw, eoc)
    ref = b.decode_steps(11)
    assert np.array_equal(got, ref)
    # the frame queued past the stop was undone: the next step matches
    assert np.array_equal(a.decode_steps(2), b.decode_steps(2))
    ka, va = a.get_kv(0, 18)
    kb, vb = b.get_kv(0, 18)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    a.close()
    b.close()


def test_max_frames_and_full_cache(ads, setup):
    d, dw = setup
    a = decoder(ads, d, dw, -1)
    got = a.decode_until_eoc(6)
    b = decoder(ads, d, dw, -1)
    assert np.array_equal(got, b.decode_steps(6))
    assert a.state() == b.state() == (11, 6, -1)
    # the cache (64 positions) ends the loop: 53 more frames fit
    rest = a.decode_until_eoc(100)
    assert rest.shape[0] == 53 and a.state()[0] == 64
    with pytest.raises(ads.TtsError):
        a.decode_until_eoc(1)
    a.close()
    b.close()
