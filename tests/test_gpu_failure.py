"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every spin-wait of the step kernel (its waits for data other CTAs exchange,
the ring's mbarrier waits) gives up after a time limit, records the timeout
in the device error word and winds the launch down.  tts_debug_expire_wait
launches the step with an embedding that is never stored, so the first
layer's wait for it cannot complete, and a 1 ms limit.  The host must see TTS_ERR_DEVICE, the context must stay usable with
its state unchanged, and the next steps -- also after tts_reset -- must meet
the oracle's parity bar."""
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


@pytest.mark.parametrize("precision", [0, 1])
def test_expired_wait_is_reported_and_the_context_recovers(ads, precision):
    d = reduced_dims(n_layers=2)
    w = synth.make_weights(d, gamma_variant=True)
    max_pos = 40
    dw = ads.DeviceWeights(w, precision=precision)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=precision)
    prompt = synth.delayed_prompt_codes(6)
    dec.prefill(prompt)
    orc.prefill(prompt, a16=True)
    gk, gv = dec.get_kv(0, 6)
    orc.k[:, :, :6], orc.v[:, :, :6] = gk, gv  # frames compared from the same cache
    codes = synth.random_codes(4, seed=2, stream=41)
    fp8 = precision == 1

    def frame(cin, where):
        t, eoc = orc.st.t, orc.st.eoc
        g = dec.decode_step(cin)
        o, ol, og = orc.decode_step(cin)
        return check_frame(g, dec.get_logits(), o, ol, og, fp8, t, eoc, where)

    frame(codes[0], "before")
    before = dec.state()
    rc = dec.debug_expire_wait()
    assert rc == -5, f"expected TTS_ERR_DEVICE, got {rc}"
    assert dec.state() == before  # the aborted launch advanced nothing
    frame(codes[1], "after the expired wait")
    # a second expiry in a row behaves the same
    assert dec.debug_expire_wait() == -5
    frame(codes[2], "after a second expired wait")
    # reset recovers the whole context as well
    dec.reset()
    orc.reset()
    assert dec.state() == (0, 0, -1)
    dec.prefill(prompt)
    orc.k[:] = 0
    orc.v[:] = 0
    orc.prefill(prompt, a16=True)
    gk, gv = dec.get_kv(0, 6)
    orc.k[:, :, :6], orc.v[:, :, :6] = gk, gv
    frame(codes[3], "after reset")
    dec.close()
