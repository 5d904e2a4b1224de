"""The lookahead decode loop (tts_decode_until_eoc): it must produce exactly
the frames of the plain device loop (tts_decode_steps), stop after the frame
in which the last codebook emits EOC (the delay pattern's frame eoc + n_cb -
1), undo the frame it queued past the stop, and leave a state from which the
next step continues as if no frame had been queued ahead."""
import numpy as np
import pytest

import oracle
import synth
from helpers import GAP, adopt_gpu_cache, check_frame, reduced_dims, to_binding_dims

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
    return d, ads.DeviceWeights(w, precision=0), w


def decoder(ads, d, dw, eoc):
    dec = ads.Decoder(to_binding_dims(d), dw, 64)
    dec.prefill(synth.delayed_prompt_codes(5))
    dec.set_frame(0, eoc)
    return dec


def test_stops_after_last_codebook_eoc(ads, setup):
    d, dw, _ = setup
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
    d, dw, _ = setup
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


@pytest.mark.parametrize("eoc", [-1, 4])
def test_lookahead_frames_match_the_oracle(ads, setup, eoc):
    """The frames the lookahead loop returns, against the CPU oracle run
    teacher-forced on the same inputs (frame 0: all-BOS; frame f: the GPU's
    codes of frame f - 1) from the same cache: every code whose oracle top-2
    gap exceeds 1e-2, and every code the delay mask forces, must match.  The
    state after the stop continues as the oracle does (full frame check)."""
    d, dw, w = setup
    n = 14  # with eoc 4 the loop stops at frame 11 and undoes the frame queued past it
    dec = decoder(ads, d, dw, eoc)
    orc = oracle.Oracle(w, 64)
    orc.prefill(synth.delayed_prompt_codes(5), a16=True)
    adopt_gpu_cache(dec, orc, 5)
    orc.set_frame(0, eoc)
    got = dec.decode_until_eoc(n)
    assert got.shape[0] == (eoc + d.n_cb if eoc >= 0 else n)
    cin = np.full(d.n_cb, d.cb_vocab - 2, np.int32)
    checked = 0
    for f in range(got.shape[0]):
        t, e = orc.st.t, orc.st.eoc
        o, _, og = orc.decode_step(cin)
        for k in range(d.n_cb):
            forced = t < k or (e >= 0 and t >= e + k)
            if forced or og[k] > GAP:
                assert got[f, k] == o[k], (f, k, got[f], o, og)
                checked += 1
        cin = got[f]
    assert checked >= got.shape[0] * d.n_cb // 2
    assert dec.state() == (orc.pos, orc.st.t, orc.st.eoc)
    # the next frame, with its logits
    t, e = orc.st.t, orc.st.eoc
    g = dec.decode_step(cin)
    o, ol, og = orc.decode_step(cin)
    check_frame(g, dec.get_logits(), o, ol, og, False, t, e, "frame after the lookahead loop")
    dec.close()
