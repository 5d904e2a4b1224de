"""Whole-step pins for the CPU oracle at tiny dimensions.

The oracle's decode step is compared with an independent float64 restatement
written here with torch library routines (F.rms_norm, matmul,
scaled_dot_product_attention, F.silu, torch's own bf16/e4m3 casts).  The two
share no code; a mis-wired residual, a norm gain on the wrong vector, a
transposed head or a wrong KV write position fails these tests.  No GPU."""
import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

TINY = synth.Dims(n_layers=2, hidden=64, n_q=4, n_kv=2, head_dim=16, inter=96, n_cb=8,
                  cb_vocab=1026)
MAXPOS = 32


def dec_bf16(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64)


def to_bf16_f64(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).to(torch.float64)


def fp8_quant(x64: torch.Tensor):
    x32 = x64.to(torch.float32)
    s = torch.clamp(x32.abs().amax(), min=1e-12) / 448.0
    q = (x32 / s).to(torch.float8_e4m3fn)
    return q.to(torch.float64), s


def fp8_weight(W64: torch.Tensor):
    W32 = W64.to(torch.float32)
    amax = W32.abs().amax(dim=1)
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (W32 / s[:, None]).to(torch.float8_e4m3fn)
    return q.to(torch.float64), s


class TorchRestatement:
    """The decode step as written from the model description, in torch float64."""

    def __init__(self, w: synth.Weights, max_pos: int, fp8: bool = False, a16: bool = False):
        self.d = w.dims
        self.fp8 = fp8
        self.a16 = a16  # W16A16: every projection input rounded to bf16 (the batched prefill)
        d = self.d
        self.E = dec_bf16(w.embed)
        self.head = dec_bf16(w.head)
        self.fn = dec_bf16(w.final_norm)
        self.L = []
        for l in range(d.n_layers):
            layer = dict(qkv=dec_bf16(w.wqkv[l]), o=dec_bf16(w.wo[l]), gu=dec_bf16(w.wgu[l]),
                         d=dec_bf16(w.wd[l]), ln_in=dec_bf16(w.ln_in[l]), ln_post=dec_bf16(w.ln_post[l]),
                         qn=dec_bf16(w.q_norm[l]), kn=dec_bf16(w.k_norm[l]))
            if fp8:
                for key in ("qkv", "o", "gu", "d"):
                    layer[key + "_q"] = fp8_weight(layer[key])
            self.L.append(layer)
        self.K = torch.zeros(d.n_layers, d.n_kv, max_pos, d.head_dim, dtype=torch.float64)
        self.V = torch.zeros_like(self.K)
        self.pos, self.t, self.eoc = 0, 0, -1

    def rope(self, x, pos):
        D = x.shape[-1]
        i = torch.arange(D // 2, dtype=torch.float64)
        ang = pos * self.d.rope_theta ** (-2.0 * i / D)
        c, s = torch.cos(ang), torch.sin(ang)
        x1, x2 = x[..., : D // 2], x[..., D // 2:]
        return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)

    def proj(self, layer, key, a):
        if not self.fp8:
            return layer[key] @ (to_bf16_f64(a) if self.a16 else a)
        qa, sa = fp8_quant(a)
        qw, sw = layer[key + "_q"]
        acc = (qw @ qa).to(torch.float32)
        return to_bf16_f64(acc * (sa * sw))

    def layers(self, codes):
        """The embedding and every layer at self.pos; returns the residual
        stream after the embedding and after each layer."""
        d = self.d
        D, NQ, NKV, I = d.head_dim, d.n_q, d.n_kv, d.inter
        eps = d.rms_eps
        h = sum(self.E[k, int(codes[k])] for k in range(d.n_cb))
        hs = [h]
        for l, P in enumerate(self.L):
            a = F.rms_norm(h, (d.hidden,), P["ln_in"], eps)
            qkv = self.proj(P, "qkv", a)
            q = qkv[: NQ * D].view(NQ, D)
            k = qkv[NQ * D:(NQ + NKV) * D].view(NKV, D)
            v = qkv[(NQ + NKV) * D:].view(NKV, D)
            q = self.rope(F.rms_norm(q, (D,), P["qn"], eps), self.pos)
            k = self.rope(F.rms_norm(k, (D,), P["kn"], eps), self.pos)
            self.K[l, :, self.pos] = to_bf16_f64(k)
            self.V[l, :, self.pos] = to_bf16_f64(v)
            Kc = self.K[l, :, : self.pos + 1].repeat_interleave(NQ // NKV, 0)
            Vc = self.V[l, :, : self.pos + 1].repeat_interleave(NQ // NKV, 0)
            attn = F.scaled_dot_product_attention(q[:, None, :], Kc, Vc)[:, 0, :].reshape(-1)
            h = h + self.proj(P, "o", attn)
            a2 = F.rms_norm(h, (d.hidden,), P["ln_post"], eps)
            gu = self.proj(P, "gu", a2)
            m = F.silu(gu[:I]) * gu[I:]
            if self.fp8:
                m = to_bf16_f64(m)
            h = h + self.proj(P, "d", m)
            hs.append(h)
        return hs

    def step(self, codes):
        d = self.d
        h = self.layers(codes)[-1]
        f = F.rms_norm(h, (d.hidden,), self.fn, d.rms_eps)
        logits = (self.head @ f).view(d.n_cb, d.cb_vocab)
        out = []
        bos, eoc_code = d.cb_vocab - 2, d.cb_vocab - 1  # 1024 and 1025 for the 1026-entry codebooks
        for k in range(d.n_cb):
            am = int(torch.argmax(logits[k]))
            if self.t < k:
                c = bos
            elif self.eoc >= 0 and self.t >= self.eoc + k:
                c = eoc_code
            else:
                c = am
            out.append(c)
        if self.eoc < 0 and out[0] == eoc_code:
            self.eoc = self.t
        self.pos += 1
        self.t += 1
        return np.array(out, np.int32), logits.numpy()


def _weights(gamma_variant=True):
    return synth.make_weights(TINY, std=0.1, gamma_variant=gamma_variant)


@pytest.mark.parametrize("fp8", [False, True])
def test_tiny_step_matches_torch_restatement(fp8):
    w = _weights()
    orc = oracle.Oracle(w, MAXPOS, precision=1 if fp8 else 0)
    ref = TorchRestatement(w, MAXPOS, fp8=fp8)
    codes = synth.random_codes(12, seed=2)
    orc.set_frame(5)
    ref.t = 5
    cin = codes[0]
    for f in range(12):
        out, logits, gaps = orc.decode_step(cin)
        rout, rlogits = ref.step(cin)
        tol = 1e-9 if not fp8 else 1e-6
        assert np.allclose(logits, rlogits, rtol=tol, atol=tol), f
        live = gaps > 1e-6
        assert np.array_equal(out[live], rout[live]), f
        cin = out
    assert orc.pos == 12


def test_other_vocabulary_bos_eoc_and_forced_eoc():
    """4 codebooks of 40 entries: BOS-pad and EOC are the last two entries
    (38, 39), as 1024 and 1025 are of the pages' 1026.  Codebook 0's head rows
    are zero except its EOC row, set to the sign pattern of frame 0's
    normalised final stream, so codebook 0 emits EOC at frame 0; the delay
    mask then fixes every code of frames 0..4, which both the oracle and the
    torch restatement must produce."""
    d = synth.Dims(n_layers=2, hidden=64, n_q=4, n_kv=2, head_dim=16, inter=96, n_cb=4, cb_vocab=40)
    w = synth.make_weights(d, std=0.1, gamma_variant=True)
    V = d.cb_vocab
    codes = np.random.default_rng(4).integers(0, V - 2, (5, d.n_cb)).astype(np.int32)
    probe = TorchRestatement(w, MAXPOS)
    h0 = probe.layers(codes[0])[-1]
    f0 = F.rms_norm(h0, (d.hidden,), probe.fn, d.rms_eps)
    head = w.head.copy()
    head[:V] = 0
    head[V - 1] = np.where(f0.numpy() >= 0, 0x3F80, 0xBF80).astype(np.uint16)  # bf16 +1 / -1
    w = dataclasses.replace(w, head=head)
    orc = oracle.Oracle(w, MAXPOS)
    ref = TorchRestatement(w, MAXPOS)
    want = [[V - 1] + [V - 1 if t >= k else V - 2 for k in range(1, d.n_cb)] for t in range(5)]
    for t in range(5):
        out, logits, _ = orc.decode_step(codes[t])
        rout, rlogits = ref.step(codes[t])
        assert np.allclose(logits, rlogits, rtol=1e-9, atol=1e-9), t
        assert out.tolist() == want[t] == rout.tolist(), (t, out, rout)
    assert orc.st.eoc == ref.eoc == 0
    # the un-forced path: without the EOC row, codes are the argmax, in [0, V)
    assert all(oracle.delay_code(k, 9, -1, 7, V) == 7 for k in range(d.n_cb))
    assert oracle.delay_code(3, 2, -1, 7, V) == V - 2 and oracle.delay_code(3, 5, 2, 7, V) == V - 1


def test_tiny_step_with_kv_prefix_and_kv_contents():
    w = _weights(gamma_variant=False)
    orc = oracle.Oracle(w, MAXPOS)
    ref = TorchRestatement(w, MAXPOS)
    k, v = synth.make_kv_prefix(TINY, 9, MAXPOS)
    orc.set_kv(k, v, 9)
    ref.K[:, :, :9] = dec_bf16(k[:, :, :9])
    ref.V[:, :, :9] = dec_bf16(v[:, :, :9])
    ref.pos = 9
    cin = synth.random_codes(1, seed=2)[0]
    out, logits, _ = orc.decode_step(cin)
    rout, rlogits = ref.step(cin)
    assert np.allclose(logits, rlogits, rtol=1e-9, atol=1e-9)
    # the new K/V row went to position 9 in bf16
    assert np.allclose(dec_bf16(orc.k[:, :, 9]).numpy(), ref.K[:, :, 9].numpy(), rtol=2 ** -7, atol=1e-12)
    assert np.allclose(dec_bf16(orc.v[:, :, 9]).numpy(), ref.V[:, :, 9].numpy(), rtol=2 ** -7, atol=1e-12)
    assert not np.array_equal(orc.k[:, :, 9], np.zeros_like(orc.k[:, :, 9]))
    assert np.array_equal(orc.k[:, :, 10:], np.zeros_like(orc.k[:, :, 10:]))


def test_prefill_equals_repeated_steps():
    w = _weights()
    codes = synth.delayed_prompt_codes(7)
    a = oracle.Oracle(w, MAXPOS)
    a.prefill(codes)
    b = oracle.Oracle(w, MAXPOS)
    for p in range(7):
        b.decode_step(codes[p])
    b.set_frame(0)
    assert a.pos == b.pos == 7
    assert np.array_equal(a.k, b.k) and np.array_equal(a.v, b.v)
    k_after_prefill, v_after_prefill = a.k.copy(), a.v.copy()
    nxt = synth.random_codes(1, seed=2, stream=3)[0]
    oa, la, _ = a.decode_step(nxt)
    ob, lb, _ = b.decode_step(nxt)
    assert np.array_equal(la, lb) and np.array_equal(oa, ob)
    # prefill split in two calls equals one call
    c = oracle.Oracle(w, MAXPOS)
    c.prefill(codes[:3])
    c.prefill(codes[3:])
    assert np.array_equal(c.k, k_after_prefill) and np.array_equal(c.v, v_after_prefill)


def test_prefill_a16_matches_torch_restatement():
    """The W16A16 prefill (every projection input rounded to bf16 with torch's
    own cast): the K/V rows it writes are bit-identical to the oracle's
    or_prefill(a16), and the residual stream after every layer of every row
    (the oracle's or_layer with a16, which also covers the last layer's O and
    down inputs that no K/V row sees) agrees to fp64 rounding."""
    w = _weights()
    P = 6
    codes = synth.delayed_prompt_codes(P)
    orc = oracle.Oracle(w, MAXPOS)
    orc.prefill(codes, a16=True)
    ref = TorchRestatement(w, MAXPOS, a16=True)
    per_row = []
    for p in range(P):
        per_row.append(ref.layers(codes[p]))
        ref.pos += 1
    to_bits = lambda x: x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.k[:, :, :P], to_bits(ref.K[:, :, :P]))
    assert np.array_equal(orc.v[:, :, :P], to_bits(ref.V[:, :, :P]))
    lay = oracle.Oracle(w, MAXPOS)
    for p in range(P):
        h = lay.embed(codes[p])
        for l in range(TINY.n_layers):
            h = lay.layer(l, p, h, a16=True)
            assert np.allclose(h, per_row[p][l + 1].numpy(), rtol=1e-12, atol=1e-12), (p, l)
    # the rounding matters: without it the restatement's rows differ
    plain = TorchRestatement(w, MAXPOS, a16=False)
    for p in range(P):
        plain.layers(codes[p])
        plain.pos += 1
    assert not np.array_equal(orc.k[:, :, :P], to_bits(plain.K[:, :, :P]))


def test_prefill_a16_rounds_projection_inputs():
    """a16 changes the result by bf16-rounding-sized amounts only."""
    w = _weights()
    codes = synth.delayed_prompt_codes(5)
    a = oracle.Oracle(w, MAXPOS)
    a.prefill(codes, a16=True)
    b = oracle.Oracle(w, MAXPOS)
    b.prefill(codes, a16=False)
    ka, kb = dec_bf16(a.k[:, :, :5]).numpy(), dec_bf16(b.k[:, :, :5]).numpy()
    assert not np.array_equal(ka, kb)
    assert np.abs(ka - kb).max() < 0.1


def test_oracle_rejects_bad_input():
    w = _weights()
    orc = oracle.Oracle(w, MAXPOS)
    with pytest.raises(ValueError):
        orc.decode_step(np.array([0, 0, 0, 1026, 0, 0, 0, 0], np.int32))
    with pytest.raises(ValueError):
        orc.prefill(np.zeros((MAXPOS + 1, 8), np.int32))


@pytest.mark.parametrize("precision", [0, 1])
def test_step_equals_embed_layers_head(precision):
    """The layer-level entry points compose to the step exactly (same logits,
    codes, gaps and KV rows): what the full-depth GPU checks build on."""
    w = synth.make_weights(TINY, gamma_variant=True)
    a = oracle.Oracle(w, MAXPOS, precision=precision)
    b = oracle.Oracle(w, MAXPOS, precision=precision)
    k, v = synth.make_kv_prefix(TINY, 5, MAXPOS)
    a.set_kv(k, v, 5)
    b.set_kv(k, v, 5)
    a.set_frame(3)
    b.set_frame(3)
    codes = synth.random_codes(1, seed=2, stream=5)[0]
    ca, la, ga = a.decode_step(codes)
    h = b.embed(codes)
    for l in range(TINY.n_layers):
        h = b.layer(l, 5, h)
    cb, lb, gb = b.head(h)
    assert np.array_equal(ca, cb)
    assert np.array_equal(la, lb)
    assert np.array_equal(ga, gb)
    assert np.array_equal(a.k[:, :, :6], b.k[:, :, :6]) and np.array_equal(a.v[:, :, :6], b.v[:, :, :6])
    # the layer call leaves the position alone; the step advanced it
    assert b.pos == 5 and a.pos == 6
