"""GPU parity at the full 36-layer sizes of the benchmark workloads, through the
C ABI and in the launch configuration the benchmark times (the persistent step
kernel, one graph per frame).

Each case checks every output of a few sampled frames (all 8 x 1026 logits and
the 8 codes) against the CPU oracle run on the same seeded inputs:
  - BF16, 13-position prompt under the delay pattern, then the first frames;
  - FP8 E4M3 W8A8 (weights quantised from the same draws), 1024 cached
    positions of N(0, 1) K/V;
  - BF16 with 8192 cached positions (split-K attention over many splits).
The oracle runs these full-size frames in fp64 on the host cores (tens of
seconds).

FP8 at full depth is checked layer by layer: the oracle's layer l starts from
the GPU's own input to layer l (the traced step kernel records the residual
stream after every layer) and the layer's contribution h_{l+1} - h_l must
agree within the FP8 bar; the head is checked on the GPU's final stream.  A
frame-level comparison is not meaningful at 36 FP8 layers: fp32 accumulation
in any order flips some bf16-rounded projection outputs against the oracle's
exact sums, and the per-token FP8 re-quantisation of every layer amplifies
those flips (the oracle with only its FP8 sums taken sequentially in fp32
already differs from itself by logits cos 0.992 at 36 layers)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import adopt_gpu_cache, check_frame, check_kv_rows, cosine, to_binding_dims, upload_kv

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
def full_weights():
    d = synth.Dims(n_layers=36)
    return d, synth.make_weights(d)


def teacher_forced(dec, orc, inputs, fp8, where):
    out = []
    for f, cin in enumerate(inputs):
        t, eoc = orc.st.t, orc.st.eoc
        g = dec.decode_step(cin)
        o, ol, og = orc.decode_step(cin)
        out.append(check_frame(g, dec.get_logits(), o, ol, og, fp8, t, eoc, f"{where} frame {f}"))
    return out


def test_full36_bf16_prompt13(ads, full_weights):
    d, w = full_weights
    max_pos = 32
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=0)
    prompt = synth.delayed_prompt_codes(13)
    dec.prefill(prompt)
    orc.prefill(prompt, a16=True)  # the batched prefill is W16A16
    assert dec.state()[0] == orc.pos == 13
    gk, gv = dec.get_kv(0, 13)
    check_kv_rows(gk, orc.k[:, :, :13], "prefill K")
    check_kv_rows(gv, orc.v[:, :, :13], "prefill V")
    adopt_gpu_cache(dec, orc, 13)  # decode frames compared from the same cache
    bos = np.full(8, 1024, np.int32)
    stats = teacher_forced(dec, orc, [bos, synth.random_codes(1, seed=2, stream=7)[0]], False, "bf16-36L")
    print("bf16 36L", stats)
    assert sum(s[2] for s in stats) >= 12
    dec.close()
    del dw


def test_full36_bf16_kv8192(ads, full_weights):
    d, w = full_weights
    L = 8192
    max_pos = L + 4
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=0)
    k, v = synth.make_kv_prefix(d, L, max_pos)
    kd, vd = upload_kv(k, v, L)
    dec.set_kv(kd, vd, L)
    orc.set_kv(k, v, L)
    del kd, vd
    codes = synth.random_codes(1, seed=2, stream=8)
    dec.set_frame(9)
    orc.set_frame(9)
    stats = teacher_forced(dec, orc, codes, False, "bf16-36L-kv8192")
    print("bf16 36L kv8192", stats)
    assert stats[0][2] >= 6
    dec.close()


def layerwise(orc, hs, pos, bar, where):
    """Each layer of the oracle from the GPU's input to it; returns per-layer cosines
    of the layer's contribution to the residual stream."""
    coss = []
    for l in range(hs.shape[0] - 1):
        hin = hs[l].astype(np.float64)
        ho = orc.layer(l, pos, hin)
        c = cosine(hs[l + 1].astype(np.float64) - hin, ho - hin)
        coss.append(c)
        assert c >= bar, f"{where}: layer {l} contribution cos {c}"
    return coss


def test_full36_fp8_kv1024(ads, full_weights):
    d, w = full_weights
    L = 1024
    max_pos = L + 4
    dw = ads.DeviceWeights(w, precision=1)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=1)
    k, v = synth.make_kv_prefix(d, L, max_pos)
    kd, vd = upload_kv(k, v, L)
    dec.set_kv(kd, vd, L)
    orc.set_kv(k, v, L)
    del kd, vd
    for f, cin in enumerate([np.full(8, 1024, np.int32), synth.random_codes(1, seed=2, stream=9)[0]]):
        pos, t = L + f, f
        g_codes, hs = dec.layer_states(cin)
        g_logits = dec.get_logits()
        h0 = orc.embed(cin)
        assert np.allclose(hs[0], h0, rtol=1e-6, atol=1e-6)
        coss = layerwise(orc, hs, pos, 0.999, f"fp8-36L-kv1024 frame {f}")
        orc.set_frame(t)
        o_codes, o_logits, o_gaps = orc.head(hs[-1].astype(np.float64))
        # the head is bf16 in both precisions: the bf16 bar applies
        stat = check_frame(g_codes, g_logits, o_codes, o_logits, o_gaps, False, t, -1, f"fp8 head frame {f}")
        print(f"fp8 36L kv1024 frame {f}: min layer cos {min(coss):.6f}, head {stat}")
        assert stat[2] >= 6
        orc.st.pos = pos + 1
    dec.close()


def test_full36_bf16_layerwise(ads, full_weights):
    """The BF16 36-layer step, layer by layer from the GPU's own inputs."""
    d, w = full_weights
    L = 64
    max_pos = L + 4
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=0)
    k, v = synth.make_kv_prefix(d, L, max_pos)
    kd, vd = upload_kv(k, v, L)
    dec.set_kv(kd, vd, L)
    orc.set_kv(k, v, L)
    del kd, vd
    cin = synth.random_codes(1, seed=2, stream=10)[0]
    dec.set_frame(10)
    g_codes, hs = dec.layer_states(cin)
    coss = layerwise(orc, hs, L, 0.9999, "bf16-36L layerwise")
    orc.set_frame(10)
    o_codes, o_logits, o_gaps = orc.head(hs[-1].astype(np.float64))
    stat = check_frame(g_codes, dec.get_logits(), o_codes, o_logits, o_gaps, False, 10, -1, "bf16 head")
    print(f"bf16 36L layerwise: min layer cos {min(coss):.7f}, head {stat}")
    dec.close()
