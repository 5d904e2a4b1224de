"""GPU parity of the decode step against the CPU oracle, through the C ABI.

Reduced-width backbones (two layers, same head structure) exercise several
attention splits, the ragged last split, the delay mask and the FP8 path in
seconds; the single-layer full-width case is the one-layer workload (hidden
2560, 32q/8kv, 9728, 8 x 1026 head, 64 cached positions).  Inputs are seeded
synthetic draws (synth); the oracle sees exactly the same inputs."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (BF16_COS, FP8_COS, adopt_gpu_cache, check_frame, check_kv_rows, cosine, reduced_dims,
                     to_binding_dims, upload_kv)

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


def make_pair(ads, dims, max_pos, precision, gamma_variant=False, std=0.02):
    w = synth.make_weights(dims, std=std, gamma_variant=gamma_variant)
    dw = ads.DeviceWeights(w, precision=precision)
    dec = ads.Decoder(to_binding_dims(dims), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=precision)
    return w, dec, orc


def run_teacher_forced(dec, orc, codes, t0, fp8, where):
    dec.set_frame(t0)
    orc.set_frame(t0)
    stats = []
    for f, cin in enumerate(codes):
        t = t0 + f
        eoc = orc.st.eoc
        g_codes = dec.decode_step(cin)
        g_logits = dec.get_logits()
        o_codes, o_logits, o_gaps = orc.decode_step(cin)
        stats.append(check_frame(g_codes, g_logits, o_codes, o_logits, o_gaps, fp8, t, eoc,
                                 f"{where} frame {f}"))
    return stats


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_reduced_teacher_forced_with_kv_prefix(ads, precision):
    d = reduced_dims(2)
    max_pos = 64
    w, dec, orc = make_pair(ads, d, max_pos, precision, gamma_variant=True)
    k, v = synth.make_kv_prefix(d, 40, max_pos)
    kd, vd = upload_kv(k, v, 40)
    dec.set_kv(kd, vd, 40)
    orc.set_kv(k, v, 40)
    codes = synth.random_codes(6, seed=2, stream=1)
    stats = run_teacher_forced(dec, orc, codes, 3, precision == 1, "reduced")
    assert sum(s[2] for s in stats) >= 24
    assert dec.state()[0] == orc.pos == 46
    # the K/V rows the GPU wrote match the oracle's to within one bf16 rounding
    gk, gv = dec.get_kv(40, 46)
    ok, ov = orc.k[:, :, 40:46], orc.v[:, :, 40:46]
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(f(gk), f(ok), rtol=2 ** -6, atol=1e-3)
    assert np.allclose(f(gv), f(ov), rtol=2 ** -6, atol=1e-3)
    # the untouched prefix is byte-identical
    gk0, _ = dec.get_kv(0, 40)
    assert np.array_equal(gk0, k[:, :, :40])
    dec.close()


def test_reduced_from_empty_cache_and_eoc(ads):
    """Positions 0.. (single split, the new row only) and a forced EOC."""
    d = reduced_dims(2)
    w, dec, orc = make_pair(ads, d, 32, 0)
    codes = synth.random_codes(5, seed=2, stream=2)
    run_teacher_forced(dec, orc, codes[:2], 0, False, "empty")
    # pretend codebook 0 emitted EOC at frame 1: the mask forces 1025 from t >= 1 + k
    dec.set_frame(4, 1)
    orc.set_frame(4, 1)
    for f in range(3):
        g = dec.decode_step(codes[2 + f])
        o, ol, og = orc.decode_step(codes[2 + f])
        check_frame(g, dec.get_logits(), o, ol, og, False, 4 + f, 1, f"eoc frame {f}")
        assert (g[: 4 + f - 1 + 1] == 1025).all()
    dec.close()


def test_free_run_equals_stepwise(ads):
    d = reduced_dims(2)
    w = synth.make_weights(d)
    dw = ads.DeviceWeights(w)
    a = ads.Decoder(to_binding_dims(d), dw, 48)
    b = ads.Decoder(to_binding_dims(d), dw, 48)
    prompt = synth.delayed_prompt_codes(5)
    a.prefill(prompt)
    b.prefill(prompt)
    run = a.decode_steps(12)
    steps = np.stack([b.decode_step() for _ in range(12)])
    assert np.array_equal(run, steps)
    assert a.state() == b.state() == (17, 12, a.state()[2])
    # delay pattern on the free run: codebook k is BOS-pad for t < k
    for t in range(8):
        assert (run[t, t + 1:] == 1024).all()
    assert np.array_equal(a.get_logits(), b.get_logits())
    a.close()
    b.close()


def test_prefill_matches_oracle(ads):
    d = reduced_dims(2)
    w, dec, orc = make_pair(ads, d, 40, 0, gamma_variant=True)
    prompt = synth.delayed_prompt_codes(9, stream=1)
    dec.prefill(prompt[:4])
    dec.prefill(prompt[4:])
    orc.prefill(prompt, a16=True)  # the batched prefill is W16A16
    assert dec.state()[0] == orc.pos == 9
    gk, gv = dec.get_kv(0, 9)
    check_kv_rows(gk, orc.k[:, :, :9], "prefill K")
    check_kv_rows(gv, orc.v[:, :, :9], "prefill V")
    # the frame after a prefill is the all-BOS frame at t = 0 (from the GPU's cache)
    adopt_gpu_cache(dec, orc, 9)
    g = dec.decode_step()
    o, ol, og = orc.decode_step(np.full(8, 1024, np.int32))
    check_frame(g, dec.get_logits(), o, ol, og, False, 0, -1, "after prefill")
    dec.close()


@pytest.mark.parametrize("t0", [0, 8])
def test_one_layer_full_width(ads, t0):
    """One full-width layer, 64 cached N(0,1) positions, one step from random codes."""
    d = synth.Dims(n_layers=1)
    w, dec, orc = make_pair(ads, d, 128, 0)
    k, v = synth.make_kv_prefix(d, 64, 128)
    kd, vd = upload_kv(k, v, 64)
    dec.set_kv(kd, vd, 64)
    orc.set_kv(k, v, 64)
    codes = synth.random_codes(2, seed=2)
    stats = run_teacher_forced(dec, orc, codes, t0, False, f"one-layer t0={t0}")
    print("one-layer", stats)
    dec.close()


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_one_layer_full_width_attention_schedule_edges(ads, precision):
    """One full-width layer decoding across the edges of the step kernel's
    attention schedule (152 CTAs, 8 kv heads, splits of at least 64
    positions over at most 19 splits per kv head), teacher-forced against the
    oracle frame by frame, with the new K/V rows compared as well:
    - 255 to 258 attended positions: at 256 the four q heads of a kv head
      still get a unit each (4 splits of 64); at 257 a fifth split appears,
      holding one position, and the units become one per (kv head, split);
    - 1215 to 1220: the split length goes from 64 to 65 positions (19
      splits, the last one ragged and not a multiple of the 8 positions a
      warp scores at a time), and the last frame runs at the last cache
      position, after which the cache is full."""
    d = synth.Dims(n_layers=1)
    max_pos = 1220
    fp8 = precision == 1
    w, dec, orc = make_pair(ads, d, max_pos, precision)
    k, v = synth.make_kv_prefix(d, max_pos - 6, max_pos)
    for prefix, frames, stream in ((254, 4, 31), (max_pos - 6, 6, 32)):
        kd, vd = upload_kv(k, v, prefix)
        dec.set_kv(kd, vd, prefix)
        orc.set_kv(k, v, prefix)
        codes = synth.random_codes(frames, seed=2, stream=stream)
        stats = run_teacher_forced(dec, orc, codes, 8, fp8, f"context {prefix + 1}")
        print(f"contexts {prefix + 1}..{prefix + frames}:", stats)
        gk, gv = dec.get_kv(prefix, prefix + frames)
        check_kv_rows(gk, orc.k[:, :, prefix:prefix + frames], f"K rows from {prefix}")
        check_kv_rows(gv, orc.v[:, :, prefix:prefix + frames], f"V rows from {prefix}")
    assert dec.state()[0] == max_pos
    with pytest.raises(ads.TtsError) as e:
        dec.decode_step(codes[-1])
    assert e.value.status == -3
    assert dec.state()[0] == max_pos
    dec.close()


@pytest.mark.parametrize("precision", [0, 1], ids=["bf16", "fp8"])
def test_device_loop_input_hidden_trace_and_gemv_timing(ads, precision):
    """The calls around the device loop, each checked against the oracle:
    - tts_set_input then one device-loop frame (tts_decode_steps) is the
      teacher-forced frame for those codes;
    - tts_get_hidden returns that frame's residual stream after the last
      layer (the oracle's embedding and layers composed at the same position);
    - a traced frame (tts_trace_step: the phase-stamping variant of the step
      kernel) computes the same frame: its logits meet the frame bar and
      every CTA stamped its start;
    - timing each projection as separate launches (tts_time_gemv) leaves the
      decode state usable: the next frame still meets the bar."""
    fp8 = precision == 1
    d = reduced_dims(2)
    max_pos = 64
    w, dec, orc = make_pair(ads, d, max_pos, precision, gamma_variant=True)
    k, v = synth.make_kv_prefix(d, 30, max_pos)
    kd, vd = upload_kv(k, v, 30)
    dec.set_kv(kd, vd, 30)
    orc.set_kv(k, v, 30)
    dec.set_frame(8)
    orc.set_frame(8)
    codes = synth.random_codes(4, seed=2, stream=61)
    # set_input + one device-loop frame; the oracle's final residual stream
    pos = orc.pos
    h = orc.embed(codes[0])
    for l in range(d.n_layers):
        h = orc.layer(l, pos, h)
    dec.set_input(codes[0])
    g = dec.decode_steps(1)[0]
    o, ol, og = orc.decode_step(codes[0])
    check_frame(g, dec.get_logits(), o, ol, og, fp8, 8, -1, "set_input + decode_steps")
    hc = cosine(dec.get_hidden(), h)
    assert hc >= (FP8_COS if fp8 else BF16_COS), f"hidden cos {hc}"
    # a traced frame
    dec.set_input(codes[1])
    tr = dec.trace_step()
    o, ol, og = orc.decode_step(codes[1])
    lc = cosine(dec.get_logits(), ol)
    assert lc >= (FP8_COS if fp8 else BF16_COS), f"traced frame cos {lc}"
    assert tr.shape[1] == 8 + 31 * d.n_layers and (tr[:, 0] > 0).all()
    assert dec.state() == (orc.pos, orc.st.t, orc.st.eoc)
    # projection timings, then a frame
    for kind in range(5):
        assert dec.time_gemv(kind, 2) > 0.0
    g = dec.decode_step(codes[2])
    o, ol, og = orc.decode_step(codes[2])
    check_frame(g, dec.get_logits(), o, ol, og, fp8, 10, -1, "after the projection timings")
    dec.close()


def test_errors_leave_state_unchanged(ads):
    d = reduced_dims(1)
    w = synth.make_weights(d)
    dw = ads.DeviceWeights(w)
    dec = ads.Decoder(to_binding_dims(d), dw, 4)
    bad = np.zeros(8, np.int32)
    bad[3] = 1026
    with pytest.raises(ads.TtsError) as e:
        dec.decode_step(bad)
    assert e.value.status == -2
    with pytest.raises(ads.TtsError) as e:
        dec.prefill(np.zeros((5, 8), np.int32))
    assert e.value.status == -3
    assert dec.state()[0] == 0
    dec.decode_steps(4)
    with pytest.raises(ads.TtsError) as e:
        dec.decode_step()
    assert e.value.status == -3
    assert dec.state()[0] == 4
    dec.reset()
    assert dec.state() == (0, 0, -1)
    dec.close()


def test_prefill_edge_sizes(ads):
    """An empty prompt is a no-op; a prompt that fills the cache exactly is
    accepted, after which the next frame has no position left."""
    d = reduced_dims(1)
    w = synth.make_weights(d)
    dw = ads.DeviceWeights(w)
    a = ads.Decoder(to_binding_dims(d), dw, 16)
    b = ads.Decoder(to_binding_dims(d), dw, 16)
    prompt = synth.delayed_prompt_codes(6)
    a.prefill(np.zeros((0, 8), np.int32))
    assert a.state() == (0, 0, -1)
    a.prefill(prompt)
    b.prefill(prompt)
    assert np.array_equal(a.decode_steps(3), b.decode_steps(3))
    a.close()
    b.close()
    full = ads.Decoder(to_binding_dims(d), dw, 16)
    full.prefill(synth.delayed_prompt_codes(16))
    assert full.state()[0] == 16
    with pytest.raises(ads.TtsError) as e:
        full.decode_step()
    assert e.value.status == -3
    assert full.state()[0] == 16
    full.close()
