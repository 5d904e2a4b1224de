"""GPU parity of the configurations besides the default one, through the C ABI.

The default model has 4 query heads per kv head and runs the persistent step
kernel with the batched prefill.  The library also accepts 1, 2 and 8 query
heads per kv head (multi-head attention and other GQA groupings: the step
kernel, the prefill attention and the stand-alone attention are built for
each), and two `tts_config.options` bits: the step as a graph of separate
kernels, and prompts prefilled position by position through the decode
step.  Each is compared with the oracle on reduced-width models (two layers,
hidden 512), teacher-forced frame by frame, with the K/V rows each side
writes compared as well.  Decode frames run at a short context (one
attention unit per query head where the grid has room) and at a long one
(one unit per kv head and split)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (FP8_COS, adopt_gpu_cache, bf16_f64, check_frame, check_kv_rows, cosine, reduced_dims,
                     to_binding_dims, upload_kv)

pytestmark = pytest.mark.gpu

MAX_POS = 1300
# (prefix length, codes stream): 41 attended positions fit one split; 1251
# take 20 splits of 64, which leaves no room for a unit per query head
SEGMENTS = ((40, 51), (1250, 52))
FRAMES = 3


@pytest.fixture(scope="module")
def ads():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import ar_decode_step_gb300.build as b
    b.build()
    import ar_decode_step_gb300 as m
    m.load()
    return m


def check_kv(gpu_bits, oracle_bits, fp8: bool, where: str):
    """BF16: the decode step's bar on K/V rows (helpers.check_kv_rows).  FP8:
    per layer cosine >= 0.999 (the FP8 bar; an E4M3 code of an activation may
    round the other way on either side)."""
    if not fp8:
        return check_kv_rows(gpu_bits, oracle_bits, where)
    for l in range(gpu_bits.shape[0]):
        c = cosine(bf16_f64(gpu_bits[l]), bf16_f64(oracle_bits[l]))
        assert c >= FP8_COS, f"{where}: layer {l}: cos {c}"


def decode_segments(dec, orc, k, v, fp8: bool, where: str, n_cb: int = 8):
    """Teacher-forced frames from each SEGMENTS prefix; the new K/V rows are
    checked after each segment."""
    for prefix, stream in SEGMENTS:
        kd, vd = upload_kv(k, v, prefix)
        dec.set_kv(kd, vd, prefix)
        orc.set_kv(k, v, prefix)
        codes = synth.random_codes(FRAMES, n_cb=n_cb, seed=2, stream=stream)
        dec.set_frame(8)
        orc.set_frame(8)
        stats = []
        for f, cin in enumerate(codes):
            t, eoc = orc.st.t, orc.st.eoc
            g = dec.decode_step(cin)
            o, ol, og = orc.decode_step(cin)
            stats.append(check_frame(g, dec.get_logits(), o, ol, og, fp8, t, eoc,
                                     f"{where}, context {prefix + 1 + f}"))
        print(f"{where}, contexts {prefix + 1}..{prefix + FRAMES}:", stats)
        gk, gv = dec.get_kv(prefix, prefix + FRAMES)
        check_kv(gk, orc.k[:, :, prefix:prefix + FRAMES], fp8, f"{where} K rows from {prefix}")
        check_kv(gv, orc.v[:, :, prefix:prefix + FRAMES], fp8, f"{where} V rows from {prefix}")


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
@pytest.mark.parametrize("n_q,n_kv", [(4, 4), (8, 4), (16, 2)], ids=["G1", "G2", "G8"])
def test_query_group_sizes(ads, n_q, n_kv, precision):
    """A batched prefill of 24 rows from an empty cache (K/V rows against the
    oracle's prefill), then decode frames at both contexts."""
    fp8 = precision == 1
    d = synth.Dims(n_layers=2, hidden=512, n_q=n_q, n_kv=n_kv, head_dim=128, inter=1024)
    w = synth.make_weights(d, gamma_variant=True)
    dw = ads.DeviceWeights(w, precision=precision)
    dec = ads.Decoder(to_binding_dims(d), dw, MAX_POS)
    orc = oracle.Oracle(w, MAX_POS, precision=precision)
    where = f"n_q {n_q}, n_kv {n_kv}, {'fp8' if fp8 else 'bf16'}"
    prompt = synth.delayed_prompt_codes(24, stream=5)
    dec.prefill(prompt)
    orc.prefill(prompt, a16=True)  # the batched prefill rounds its projection inputs to bf16
    assert dec.state()[0] == orc.pos == 24
    gk, gv = dec.get_kv(0, 24)
    check_kv(gk, orc.k[:, :, :24], fp8, f"{where}: prefill K")
    check_kv(gv, orc.v[:, :, :24], fp8, f"{where}: prefill V")
    k, v = synth.make_kv_prefix(d, SEGMENTS[-1][0], MAX_POS)
    decode_segments(dec, orc, k, v, fp8, where)
    dec.close()


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_codebook_count_and_vocabulary(ads, precision):
    """4 codebooks of 2050 entries (BOS-pad 2048, EOC 2049) instead of 8 of
    1026: the embedding gather, the head's rows, the per-codebook argmax and
    the delay mask follow the configuration."""
    fp8 = precision == 1
    d = synth.Dims(n_layers=2, hidden=512, n_q=8, n_kv=2, head_dim=128, inter=1024, n_cb=4, cb_vocab=2050)
    w = synth.make_weights(d, gamma_variant=True)
    dw = ads.DeviceWeights(w, precision=precision)
    dec = ads.Decoder(to_binding_dims(d), dw, MAX_POS)
    orc = oracle.Oracle(w, MAX_POS, precision=precision)
    k, v = synth.make_kv_prefix(d, SEGMENTS[-1][0], MAX_POS)
    decode_segments(dec, orc, k, v, fp8, f"4 x 2050 codebooks, {'fp8' if fp8 else 'bf16'}", n_cb=4)
    # frame 0 from the all-BOS input: codebooks 1..3 are forced to BOS-pad
    dec.set_kv(*upload_kv(k, v, 40), 40)
    orc.set_kv(k, v, 40)
    dec.set_frame(0)
    orc.set_frame(0)
    bos = np.full(4, 2048, np.int32)
    g = dec.decode_step(bos)
    o, ol, og = orc.decode_step(bos)
    check_frame(g, dec.get_logits(), o, ol, og, fp8, 0, -1, "4 x 2050, frame 0")
    assert (g[1:] == 2048).all()
    dec.close()


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_longest_context(ads, precision):
    """The largest cache the library accepts (65536 positions): the last
    three positions decoded against the oracle (64 splits of 1024 positions
    per kv head), then the cache is full."""
    fp8 = precision == 1
    d = reduced_dims(2)
    max_pos = 65536
    w = synth.make_weights(d, gamma_variant=True)
    dw = ads.DeviceWeights(w, precision=precision)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=precision)
    prefix = max_pos - FRAMES
    k, v = synth.make_kv_prefix(d, prefix, max_pos)
    kd, vd = upload_kv(k, v, prefix)
    dec.set_kv(kd, vd, prefix)
    orc.set_kv(k, v, prefix)
    codes = synth.random_codes(FRAMES, seed=2, stream=53)
    dec.set_frame(8)
    orc.set_frame(8)
    for f, cin in enumerate(codes):
        g = dec.decode_step(cin)
        o, ol, og = orc.decode_step(cin)
        check_frame(g, dec.get_logits(), o, ol, og, fp8, 8 + f, -1, f"context {prefix + 1 + f}")
    gk, gv = dec.get_kv(prefix, max_pos)
    check_kv(gk, orc.k[:, :, prefix:], fp8, "K rows at the end of the cache")
    check_kv(gv, orc.v[:, :, prefix:], fp8, "V rows at the end of the cache")
    assert dec.state()[0] == max_pos
    with pytest.raises(ads.TtsError) as e:
        dec.decode_step(codes[-1])
    assert e.value.status == -3
    dec.close()


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_separate_kernel_graph(ads, precision):
    """The step as a graph of one kernel per projection and one attention
    kernel per layer (TTS_OPT_SEPARATE_KERNELS)."""
    fp8 = precision == 1
    d = reduced_dims(2)
    w = synth.make_weights(d, gamma_variant=True)
    dw = ads.DeviceWeights(w, precision=precision)
    dec = ads.Decoder(to_binding_dims(d), dw, MAX_POS, options=ads.OPT_SEPARATE_KERNELS)
    orc = oracle.Oracle(w, MAX_POS, precision=precision)
    k, v = synth.make_kv_prefix(d, SEGMENTS[-1][0], MAX_POS)
    decode_segments(dec, orc, k, v, fp8, f"separate kernels, {'fp8' if fp8 else 'bf16'}")
    dec.close()


@pytest.mark.parametrize("separate", [False, True], ids=["persistent", "separate"])
@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_position_by_position_prefill(ads, precision, separate):
    """TTS_OPT_PREFILL_STEPS: each prompt row runs through the decode step's
    layers (the decode arithmetic, no bf16 rounding of activations in BF16),
    in two calls; the oracle's prefill without that rounding is the
    reference.  Then the all-BOS frame from the GPU's cache."""
    fp8 = precision == 1
    d = reduced_dims(2)
    w = synth.make_weights(d, gamma_variant=True)
    dw = ads.DeviceWeights(w, precision=precision)
    opts = ads.OPT_PREFILL_STEPS | (ads.OPT_SEPARATE_KERNELS if separate else 0)
    dec = ads.Decoder(to_binding_dims(d), dw, 40, options=opts)
    orc = oracle.Oracle(w, 40, precision=precision)
    prompt = synth.delayed_prompt_codes(9, stream=6)
    dec.prefill(prompt[:4])
    dec.prefill(prompt[4:])
    orc.prefill(prompt, a16=False)
    assert dec.state()[0] == orc.pos == 9
    gk, gv = dec.get_kv(0, 9)
    check_kv(gk, orc.k[:, :, :9], fp8, "prefill K")
    check_kv(gv, orc.v[:, :, :9], fp8, "prefill V")
    adopt_gpu_cache(dec, orc, 9)
    g = dec.decode_step()
    o, ol, og = orc.decode_step(np.full(8, 1024, np.int32))
    check_frame(g, dec.get_logits(), o, ol, og, fp8, 0, -1, "after the prefill")
    dec.close()
