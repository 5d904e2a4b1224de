"""The batched prompt prefill (tensor-core GEMMs, causal attention over the
prompt) against the CPU oracle's W16A16 prefill: the K/V rows it writes for
every layer and position (helpers.check_kv_rows), and the first decode frame
after it, run by both sides from the GPU's cache.

Cases: a reduced-width backbone over two chunks (600 positions: 512 + 88,
the second chunk attending the first through the cache, after a cached
prefix); 512 positions at full width (2 layers: the batched-prefill workload's
shapes, 512 x 2560 x {6144, 2560, 19456, 2560}); and the full 36-layer model
over a 64-position prompt."""
import numpy as np
import pytest

import oracle
import synth
from fp8_restatement import Fp8Fp32Step, layerwise_spread
from helpers import adopt_gpu_cache, bf16_f64, check_frame, check_kv_rows, cosine, reduced_dims, to_binding_dims, upload_kv

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


def run_case(ads, d, P, prefix, seed_stream, gamma_variant=False):
    max_pos = prefix + P + 4
    w = synth.make_weights(d, gamma_variant=gamma_variant)
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=0)
    if prefix:
        k, v = synth.make_kv_prefix(d, prefix, max_pos)
        kd, vd = upload_kv(k, v, prefix)
        dec.set_kv(kd, vd, prefix)
        orc.set_kv(k, v, prefix)
    prompt = synth.delayed_prompt_codes(P, stream=seed_stream)
    dec.prefill(prompt)
    orc.prefill(prompt, a16=True)
    assert dec.state()[0] == orc.pos == prefix + P
    gk, gv = dec.get_kv(prefix, prefix + P)
    kv_stat = (check_kv_rows(gk, orc.k[:, :, prefix:prefix + P], f"P={P} K"),
               check_kv_rows(gv, orc.v[:, :, prefix:prefix + P], f"P={P} V"))
    if prefix:
        gk, _ = dec.get_kv(0, prefix)
        assert np.array_equal(gk, orc.k[:, :, :prefix])
    adopt_gpu_cache(dec, orc, prefix + P)
    g = dec.decode_step()
    o, ol, og = orc.decode_step(np.full(8, 1024, np.int32))
    stat = check_frame(g, dec.get_logits(), o, ol, og, False, 0, -1, f"frame after prefill P={P}")
    dec.close()
    return kv_stat, stat


def restatement_prefill_spread(w, d, P, prefix, prompt, max_pos):
    """The float32 restatement of the FP8 step (exact projection sums) run
    over the prompt rows and checked by the same layer-by-layer protocol as
    the GPU: the spread of per-row layer-contribution cosines that fp32
    arithmetic alone leaves against the oracle.  [n_layers][P]."""
    r = Fp8Fp32Step(w, max_pos, "exact")
    orc = oracle.Oracle(w, max_pos, precision=1)
    if prefix:
        k, v = synth.make_kv_prefix(d, prefix, max_pos)
        r.set_kv(k, v, prefix)
        orc.set_kv(k, v, prefix)
    else:
        r.pos = 0
    rows = []
    for p in range(P):
        rows.append([h.numpy() for h in r.layer_states(prompt[p])])
        r.pos += 1
    return layerwise_spread(orc, rows, prefix, d.n_layers)


def run_case_fp8(ads, d, P, prefix, seed_stream):
    """The batched FP8 W8A8 prefill (tcgen05 kind::f8f6f4 GEMMs, per-token
    activation scales) against the oracle's FP8 layers, layer by layer from
    the GPU's own residual stream (as the FP8 decode step is checked: every
    layer re-quantises per token).  The attention of FP8 prefills carries Q
    and P as two bf16 terms each on the tensor cores (about 2^-16 of the
    oracle's exact attention).  The layer's K/V rows reach the FP8 bar (cos
    >= 0.999).  Each row's layer contribution is held to the spread that
    fp32 arithmetic alone leaves under this protocol, measured on the same
    rows by the float32 restatement with exact projection sums
    (fp8_restatement.py; the cache each side attends is its own, so rare
    E4M3 flips of the quantised inputs move single rows by ~1e-3 at this
    width): no row below the restatement's worst by more than 5e-4, at most
    3 more rows below 0.999, and a mean no lower by more than 1e-4.  The
    first frame after the prefill, run from the GPU's cache, meets the FP8
    frame bar."""
    max_pos = prefix + P + 4
    w = synth.make_weights(d, gamma_variant=True)
    dw = ads.DeviceWeights(w, precision=1)
    dec = ads.Decoder(to_binding_dims(d), dw, max_pos)
    orc = oracle.Oracle(w, max_pos, precision=1)
    if prefix:
        k, v = synth.make_kv_prefix(d, prefix, max_pos)
        kd, vd = upload_kv(k, v, prefix)
        dec.set_kv(kd, vd, prefix)
        orc.set_kv(k, v, prefix)
    prompt = synth.delayed_prompt_codes(P, stream=seed_stream)
    hs = dec.prefill_states(prompt).astype(np.float64)
    assert dec.state()[0] == prefix + P
    gk, gv = dec.get_kv(prefix, prefix + P)
    G = layerwise_spread(orc, [hs[:, p] for p in range(P)], prefix, d.n_layers)
    for l in range(d.n_layers):
        for name, g_, o_ in (("K", gk[l], orc.k[l, :, prefix:prefix + P]), ("V", gv[l], orc.v[l, :, prefix:prefix + P])):
            c = cosine(bf16_f64(g_).ravel(), bf16_f64(o_).ravel())
            assert c >= 0.999, f"FP8 prefill P={P} {name} layer {l}: cos {c}"
    R = restatement_prefill_spread(w, d, P, prefix, prompt, max_pos)
    stats = dict(gpu_min=float(G.min()), gpu_mean=float(G.mean()), gpu_below=int((G < 0.999).sum()),
                 fp32_min=float(R.min()), fp32_mean=float(R.mean()), fp32_below=int((R < 0.999).sum()))
    print(f"FP8 prefill P={P} layer contributions:", stats)
    assert G.min() >= min(0.999, R.min() - 5e-4), stats
    assert stats["gpu_below"] <= stats["fp32_below"] + 3, stats
    assert G.mean() >= R.mean() - 1e-4, stats
    adopt_gpu_cache(dec, orc, prefix + P)
    orc.st.pos = prefix + P
    g = dec.decode_step()
    o, ol, og = orc.decode_step(np.full(8, 1024, np.int32))
    stat = check_frame(g, dec.get_logits(), o, ol, og, True, 0, -1, f"FP8 frame after prefill P={P}")
    dec.close()
    return stats, stat


def test_prefill_fp8_batched(ads):
    print(run_case_fp8(ads, reduced_dims(2), 40, 0, 6))


def test_prefill_fp8_after_prefix(ads):
    # one chunk (the states hook records up to 512 rows); the chunk loop is
    # the same for both precisions and runs two chunks in the BF16 case below
    print(run_case_fp8(ads, reduced_dims(2), 480, 24, 7))


def test_prefill_two_chunks_after_prefix(ads):
    print(run_case(ads, reduced_dims(2), 600, 24, 3, gamma_variant=True))


def test_prefill_512_full_width(ads):
    print(run_case(ads, synth.Dims(n_layers=2), 512, 0, 4))


def test_prefill_full_depth(ads):
    print(run_case(ads, synth.Dims(n_layers=36), 64, 0, 5))


def test_prefill_layerwise_full_depth(ads):
    """36 layers, 48 prompt rows: the oracle's layer l (W16A16) runs every row
    from the GPU's own input to layer l; each row's layer contribution and the
    K/V rows of the layer must agree within the BF16 bar."""
    d = synth.Dims(n_layers=36)
    P = 48
    w = synth.make_weights(d)
    dw = ads.DeviceWeights(w, precision=0)
    dec = ads.Decoder(to_binding_dims(d), dw, P + 4)
    orc = oracle.Oracle(w, P + 4, precision=0)
    prompt = synth.delayed_prompt_codes(P, stream=6)
    hs = dec.prefill_states(prompt).astype(np.float64)
    for p in range(P):
        assert np.allclose(hs[0, p], orc.embed(prompt[p]), rtol=1e-6, atol=1e-6)
    gk, gv = dec.get_kv(0, P)
    worst = 1.0
    for l in range(d.n_layers):
        for p in range(P):
            out = orc.layer(l, p, hs[l, p], a16=True)
            c = cosine(hs[l + 1, p] - hs[l, p], out - hs[l, p])
            worst = min(worst, c)
            assert c >= 0.9999, f"layer {l} row {p}: contribution cos {c}"
        for name, g, o in (("K", gk[l], orc.k[l, :, :P]), ("V", gv[l], orc.v[l, :, :P])):
            a, b = bf16_f64(g), bf16_f64(o)
            err = float((np.abs(a - b) / np.maximum(1.0, np.abs(b))).max())
            assert err <= 2e-2, f"layer {l} {name}: scaled max error {err}"
    print("prefill layerwise: worst contribution cos", worst)
    dec.close()
