"""The oracle's temperature-sampling head ("Higgs Audio v3 TTS-4B on FlashRT",
section 4 sampling policy), pinned without the GPU: its Philox4x32-10 against
the known-answer vectors published with the Random123 library (SC'11 paper),
the inverse-CDF draw against closed forms, and the draw frequencies against
the softmax probabilities."""
import math

import numpy as np

import oracle


def test_philox_known_answers():
    assert [hex(x) for x in oracle.philox4x32_10([0, 0, 0, 0], [0, 0])] == \
        ["0x6627e8d5", "0xe169c58d", "0xbc57ac4c", "0x9b00dbd8"]
    assert [hex(x) for x in oracle.philox4x32_10([0xffffffff] * 4, [0xffffffff] * 2)] == \
        ["0x408f276d", "0x41c83b0e", "0xa20bc7c6", "0x6d5451fd"]
    assert [hex(x) for x in oracle.philox4x32_10([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344],
                                                 [0xa4093822, 0x299f31d0])] == \
        ["0xd16cfe09", "0x94fdcceb", "0x5001e420", "0x24126ea1"]


def uniform(seed, t, k):
    r = oracle.philox4x32_10([t, k, 0, 0], [seed & 0xffffffff, seed >> 32])
    return (r[0] >> 8) / 2.0 ** 24


def test_two_way_draw_closed_form():
    # weights 1 : 3 (logits 0, ln 3): code 0 exactly when u < 1/4
    logits = np.array([0.0, math.log(3.0)])
    seed = 0x0123456789abcdef
    for t in range(200):
        for k in range(8):
            code, _ = oracle.sample_code(logits, 1.0, seed, t, k)
            assert code == (0 if uniform(seed, t, k) < 0.25 else 1)


def test_temperature_scales_logits():
    # logits (0, 2) at T = 2 are logits (0, 1) at T = 1: the same draws
    seed = 77
    for t in range(300):
        a, _ = oracle.sample_code(np.array([0.0, 2.0]), 2.0, seed, t, 3)
        b, _ = oracle.sample_code(np.array([0.0, 1.0]), 1.0, seed, t, 3)
        assert a == b


def test_low_temperature_is_argmax():
    rng = np.random.default_rng(5)
    for trial in range(20):
        logits = rng.permutation(np.arange(1026) * 0.1)
        for t in range(5):
            code, _ = oracle.sample_code(logits, 1e-3, 1000 + trial, t, trial % 8)
            assert code == int(np.argmax(logits))


def test_draw_frequencies_follow_softmax():
    logits = np.array([0.0, 1.0, 2.0, 3.0, -1.0])
    T = 1.5
    p = np.exp(logits / T)
    p /= p.sum()
    n = 20000
    counts = np.zeros(len(logits))
    for t in range(n):
        code, _ = oracle.sample_code(logits, T, 2024, t, t % 8)
        counts[code] += 1
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 25.0, (counts, n * p, chi2)  # 4 degrees of freedom: far beyond the 99.99 % point is ~23.5


def test_seed_and_counter_change_the_draws():
    logits = np.zeros(1026)
    a = [oracle.sample_code(logits, 1.0, 1, t, 0)[0] for t in range(64)]
    b = [oracle.sample_code(logits, 1.0, 2, t, 0)[0] for t in range(64)]
    c = [oracle.sample_code(logits, 1.0, 1, t, 1)[0] for t in range(64)]
    assert a != b and a != c
    assert a == [oracle.sample_code(logits, 1.0, 1, t, 0)[0] for t in range(64)]
    # uniform logits: the code is floor(u * V) up to the running-sum rounding
    for t in range(64):
        assert abs(a[t] - int(uniform(1, t, 0) * 1026)) <= 1
