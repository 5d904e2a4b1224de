"""Prefix reuse (tts_prefix_save / tts_prefix_restore; "Higgs Audio v3 TTS-4B
on FlashRT", section 4 and Performance "prompt prefill": a resident system
prompt's KV is reused and each request prefills only its suffix,
bit-identically).  A request served after a restore -- even after the cache
rows of the prefix were overwritten in between -- must give the same K/V
rows and the same codes, bit for bit, as the same request served right after
the prefix, and as a fresh context that prefills the prefix and the suffix."""
import numpy as np
import pytest

import oracle
import synth
from helpers import adopt_gpu_cache, check_frame, check_kv_rows, reduced_dims, to_binding_dims

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


def request(dec, suffix, frames):
    dec.prefill(suffix)
    codes = dec.decode_steps(frames)
    return codes, dec.state()


def test_prefix_restore_is_bit_identical(ads, model):
    d, w = model
    dw = ads.DeviceWeights(w, precision=0)
    system = synth.delayed_prompt_codes(13)
    suf_a = synth.random_codes(7, seed=2, stream=31)
    suf_b = synth.random_codes(5, seed=2, stream=32)
    end = 13 + 7 + 4

    dec = ads.Decoder(to_binding_dims(d), dw, 64)
    dec.prefill(system)
    dec.prefix_save()
    a1, st1 = request(dec, suf_a, 4)
    ka1, va1 = dec.get_kv(0, end)
    # another request, then one that overwrites the prefix rows themselves
    dec.prefix_restore()
    request(dec, suf_b, 3)
    dec.rewind(0)
    dec.prefill(suf_b)
    dec.prefix_restore()
    assert dec.state() == (13, 0, -1)
    a2, st2 = request(dec, suf_a, 4)
    ka2, va2 = dec.get_kv(0, end)
    assert np.array_equal(a1, a2) and st1 == st2
    assert np.array_equal(ka1, ka2) and np.array_equal(va1, va2)
    dec.close()

    # a fresh context serving the same request without reuse
    fresh = ads.Decoder(to_binding_dims(d), dw, 64)
    fresh.prefill(system)
    a3, st3 = request(fresh, suf_a, 4)
    kf, vf = fresh.get_kv(0, end)
    assert np.array_equal(a1, a3) and st1 == st3
    assert np.array_equal(ka1, kf) and np.array_equal(va1, vf)
    fresh.close()


def test_prefix_errors(ads, model):
    d, w = model
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, 32)
    with pytest.raises(ads.TtsError):
        dec.prefix_restore()  # nothing saved
    with pytest.raises(ads.TtsError):
        dec.prefix_save()     # position 0: nothing to save
    dec.prefill(synth.delayed_prompt_codes(5))
    dec.prefix_save()
    dec.decode_steps(2)
    dec.prefix_restore()
    assert dec.state() == (5, 0, -1)
    dec.close()


def test_one_call_and_split_prefill_agree(ads, model):
    """prefill(prefix + suffix) in one call against prefill(prefix) then
    prefill(suffix): the rows are the same computation (the GEMMs reduce each
    row alone in a fixed k order, attention is per row), so the caches agree
    bit for bit."""
    d, w = model
    dw = ads.DeviceWeights(w, precision=0)
    system = synth.delayed_prompt_codes(13)
    suf = synth.random_codes(7, seed=2, stream=33)
    one = ads.Decoder(to_binding_dims(d), dw, 64)
    one.prefill(np.concatenate([system, suf]))
    two = ads.Decoder(to_binding_dims(d), dw, 64)
    two.prefill(system)
    two.prefill(suf)
    k1, v1 = one.get_kv(0, 20)
    k2, v2 = two.get_kv(0, 20)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    assert np.array_equal(one.decode_steps(3), two.decode_steps(3))
    one.close()
    two.close()


@pytest.mark.parametrize("precision", [0, 1])
def test_repeated_prefill_replays_identically(ads, model, precision):
    """A batched prefill chunk runs directly the first time its shape is seen,
    is captured as a graph the second time and replayed after that: the three
    runs of one request must leave the same cache rows and codes, bit for bit,
    and a chunk of another shape in between must not disturb the replay."""
    d, w = model
    dw = ads.DeviceWeights(w, precision=precision)
    prompt = synth.delayed_prompt_codes(21)
    other = synth.random_codes(9, seed=2, stream=34)
    dec = ads.Decoder(to_binding_dims(d), dw, 64)
    runs = []
    for rep in range(4):
        dec.reset()
        if rep == 2:
            dec.prefill(other)
            dec.reset()
        dec.prefill(prompt)
        k, v = dec.get_kv(0, 21)
        runs.append((k, v, dec.decode_steps(3), dec.state()))
    for k, v, codes, st in runs[1:]:
        assert np.array_equal(k, runs[0][0]) and np.array_equal(v, runs[0][1])
        assert np.array_equal(codes, runs[0][2]) and st == runs[0][3]
    dec.close()


@pytest.mark.parametrize("precision", [0, 1])
def test_request_after_restore_matches_the_oracle(ads, model, precision):
    """A request served after a restore (the prefix rows overwritten in
    between) against the CPU oracle: the prefix + suffix K/V rows meet the
    prefill bar against the oracle's prefill of the whole prompt, and the
    request's decode frames, teacher-forced from the same cache, meet the
    frame bar."""
    d, w = model
    dw = ads.DeviceWeights(w, precision=precision)
    system = synth.delayed_prompt_codes(13)
    suf = synth.random_codes(7, seed=2, stream=35)
    dec = ads.Decoder(to_binding_dims(d), dw, 64)
    dec.prefill(system)
    dec.prefix_save()
    dec.prefill(synth.random_codes(6, seed=2, stream=36))  # another request
    dec.rewind(0)
    dec.prefill(synth.random_codes(9, seed=2, stream=37))  # overwrites the prefix rows
    dec.prefix_restore()
    dec.prefill(suf)
    orc = oracle.Oracle(w, 64, precision=precision)
    orc.prefill(np.concatenate([system, suf]), a16=True)
    gk, gv = dec.get_kv(0, 20)
    if precision == 0:
        check_kv_rows(gk, orc.k[:, :, :20], "K after restore")
        check_kv_rows(gv, orc.v[:, :, :20], "V after restore")
    else:
        from helpers import bf16_f64, cosine
        for l in range(d.n_layers):
            assert cosine(bf16_f64(gk[l]), bf16_f64(orc.k[l, :, :20])) >= 0.999
            assert cosine(bf16_f64(gv[l]), bf16_f64(orc.v[l, :, :20])) >= 0.999
    adopt_gpu_cache(dec, orc, 20)
    cin = np.full(d.n_cb, d.cb_vocab - 2, np.int32)
    for f in range(4):
        t, e = orc.st.t, orc.st.eoc
        g = dec.decode_step(cin)
        o, ol, og = orc.decode_step(cin)
        check_frame(g, dec.get_logits(), o, ol, og, precision == 1, t, e, f"request frame {f}")
        cin = g
    dec.close()
