"""The shared input generator: Philox4x32-10 known-answer vectors (published
with the Random123 library for the SC'11 paper), determinism, layout and
distribution of the model-shaped inputs.  No GPU."""
import numpy as np

import synth


def test_philox_known_answers():
    # counter = (idx lo, idx hi, stream lo, stream hi), key = (seed lo, seed hi)
    assert [hex(x) for x in synth.raw_u32(0, 0, 0)] == \
        ["0x6627e8d5", "0xe169c58d", "0xbc57ac4c", "0x9b00dbd8"]
    assert [hex(x) for x in synth.raw_u32(0xffffffffffffffff, 0xffffffffffffffff, 0xffffffffffffffff)] == \
        ["0x408f276d", "0x41c83b0e", "0xa20bc7c6", "0x6d5451fd"]
    assert [hex(x) for x in synth.raw_u32(0x299f31d0a4093822, 0x0370734413198a2e, 0x85a308d3243f6a88)] == \
        ["0xd16cfe09", "0x94fdcceb", "0x5001e420", "0x24126ea1"]


def test_normals_deterministic_and_distributed():
    a = synth.normal_f32(0, 11, (1_000_001,), std=0.02)
    b = synth.normal_f32(0, 11, (1_000_001,), std=0.02)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 1e-4 and abs(a.std() - 0.02) < 1e-4
    c = synth.normal_f32(0, 12, (1000,), std=0.02)
    assert not np.array_equal(a[:1000], c)
    # a prefix of a longer draw equals the shorter draw (pure function of index)
    assert np.array_equal(synth.normal_f32(0, 11, (10,), std=0.02), a[:10])
    bits = synth.normal_bf16(0, 11, (1000,), std=0.02)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.allclose(f, a[:1000], rtol=2 ** -8, atol=0)


def test_strided_rows_match_flat_draw():
    out = np.zeros((10, 64), np.uint16)
    synth.normal_bf16_rows(1, 5, 6, 48, out[:, :])
    flat = synth.normal_bf16(1, 5, (6 * 48,))
    assert np.array_equal(out[:6, :48].reshape(-1), flat)
    assert not out[6:].any() and not out[:, 48:].any()


def test_codes_and_delayed_prompt():
    c = synth.random_codes(1000)
    assert c.shape == (1000, 8) and c.min() >= 0 and c.max() < 1024
    assert len(np.unique(c)) > 900
    p = synth.delayed_prompt_codes(13)
    for k in range(8):
        assert (p[:k, k] == 1024).all()
        assert (p[k:, k] < 1024).all()


def test_model_weights_layout():
    d = synth.Dims(n_layers=2, hidden=64, n_q=4, n_kv=2, head_dim=16, inter=96)
    w = synth.make_weights(d)
    assert w.embed.shape == (8, 1026, 64) and w.head.shape == (8208, 64)
    assert w.wqkv[0].shape == (128, 64) and w.wo[1].shape == (64, 64)
    assert w.wgu[0].shape == (192, 64) and w.wd[0].shape == (64, 96)
    assert (w.ln_in[0] == 0x3F80).all()
    assert not np.array_equal(w.wqkv[0], w.wqkv[1])
    wg = synth.make_weights(d, gamma_variant=True)
    assert not (wg.ln_in[0] == 0x3F80).all()
    assert np.array_equal(wg.wqkv[0], w.wqkv[0])
    k, v = synth.make_kv_prefix(d, 5, 9)
    assert k.shape == (2, 2, 9, 16) and k[:, :, :5].any() and not k[:, :, 5:].any()
    assert not np.array_equal(k, v)
