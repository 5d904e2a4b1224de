"""The FP8 W8A8 decode step restated in float32, for measuring how much the
order of fp32 summation alone moves the 36-layer result away from the oracle.

Written here from the model description with torch and numpy routines (no
code shared with the oracle or the CUDA library).  It computes what the FP8
step computes ("Higgs Audio v3 TTS-4B on FlashRT", Performance "FP8 W8A8" and
section 5; readings c5-c8 and c18 of the design notes): per-output-row E4M3
weights, per-token E4M3 activations with scale max(amax, 1e-12)/448, products
summed in fp32, each projection output bf16(acc * (s_a * s_w[n])), the SwiGLU
of the bf16 gate/up rounded to bf16, everything else in fp32, and a BF16 head.
The variants differ only in how each projection's sum of products is taken,
chosen by `order`:

  "exact"    in fp64, which is exact for E4M3 products (as the oracle sums);
             everything else still fp32;
  "blas"     torch.mv in float32 (the BLAS library's blocked order);
  "chunked"  fp32 sums over 64-element chunks of the row, then the chunk sums
             added in fp32 from the last chunk to the first (a GPU-like
             split of the row).

Every e4m3 x e4m3 product is exact in fp32, so the orders differ only in how
the sums round; "exact" removes that difference and keeps only the fp32
rounding of the rest of the step (norms, attention, SwiGLU, residual adds).
Through the bf16 rounding of the outputs and the E4M3 re-quantisation of the
next activation, any such difference can flip codes."""
from __future__ import annotations

import numpy as np
import torch

import synth

ORDERS = ("exact", "blas", "chunked")


def _bf16(bits) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def _round_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).to(torch.float32)


def quant_rows(W_bits) -> tuple[torch.Tensor, torch.Tensor]:
    """Per-row E4M3 weights: s[n] = max|W[n]| / 448 (1 for a zero row), codes
    e4m3(W / s) with torch's float8_e4m3fn cast (round to nearest even, the
    finite range saturating), in fp32."""
    W = _bf16(W_bits).to(torch.float32)
    amax = W.abs().amax(dim=1)
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = torch.clamp(W / s[:, None], -448.0, 448.0).to(torch.float8_e4m3fn)
    return q, s


def quant_act(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    s = torch.clamp(x.abs().amax(), min=1e-12) / 448.0
    return torch.clamp(x / s, -448.0, 448.0).to(torch.float8_e4m3fn).to(torch.float32), s


def rms_norm(x: torch.Tensor, g: torch.Tensor, eps: float) -> torch.Tensor:
    r = torch.rsqrt((x * x).sum() / x.shape[-1] + eps) if x.dim() == 1 else \
        torch.rsqrt((x * x).sum(dim=-1, keepdim=True) / x.shape[-1] + eps)
    return x * r * g


class Fp8Fp32Step:
    """One model copy (E4M3 weights quantised here), a bf16 KV cache and the
    decode state; step() runs one teacher-forced frame."""

    def __init__(self, w: synth.Weights, max_pos: int, order: str = "blas", share: "Fp8Fp32Step" = None):
        """share: another instance built from the same weights whose quantised
        model this one uses (it keeps its own order, cache and state)."""
        assert order in ORDERS
        self.order = order
        d = w.dims
        self.d = d
        if share is not None:
            self.E, self.head, self.fn, self.L = share.E, share.head, share.fn, share.L
        else:
            self.E = _bf16(w.embed).to(torch.float32)
            self.head = _bf16(w.head).to(torch.float32)
            self.fn = _bf16(w.final_norm).to(torch.float32)
            self.L = []
            for l in range(d.n_layers):
                lay = {k: quant_rows(getattr(w, k)[l]) for k in ("wqkv", "wo", "wgu", "wd")}
                for k in ("ln_in", "ln_post", "q_norm", "k_norm"):
                    lay[k] = _bf16(getattr(w, k)[l]).to(torch.float32)
                self.L.append(lay)
        shape = (d.n_layers, d.n_kv, max_pos, d.head_dim)
        self.K = torch.zeros(shape, dtype=torch.bfloat16)
        self.V = torch.zeros(shape, dtype=torch.bfloat16)
        i = np.arange(d.head_dim // 2, dtype=np.float64)
        self.inv_f = d.rope_theta ** (-2.0 * i / d.head_dim)
        self.pos, self.t, self.eoc = 0, 0, -1

    def set_kv(self, k_bits, v_bits, length: int) -> None:
        self.K[:, :, :length] = _bf16(k_bits[:, :, :length])
        self.V[:, :, :length] = _bf16(v_bits[:, :, :length])
        self.pos = length

    def _dot(self, q8: torch.Tensor, a8: torch.Tensor) -> torch.Tensor:
        if self.order == "exact":
            return torch.mv(q8.to(torch.float64), a8.to(torch.float64)).to(torch.float32)
        Wf = q8.to(torch.float32)
        if self.order == "blas":
            return torch.mv(Wf, a8)
        N, K = Wf.shape
        part = (Wf.view(N, K // 64, 64) * a8.view(K // 64, 64)).sum(dim=-1)  # exact products, fp32 sums
        acc = part[:, -1].clone()
        for c in range(K // 64 - 2, -1, -1):
            acc = acc + part[:, c]
        return acc

    def _proj(self, qs, x: torch.Tensor) -> torch.Tensor:
        q8, sw = qs
        a8, sa = quant_act(x)
        acc = self._dot(q8, a8)
        return _round_bf16(acc * (sa * sw))

    def _rope(self, x: torch.Tensor, pos: int) -> torch.Tensor:
        ang = pos * self.inv_f
        c = torch.from_numpy(np.cos(ang).astype(np.float32))
        s = torch.from_numpy(np.sin(ang).astype(np.float32))
        h = x.shape[-1] // 2
        x1, x2 = x[..., :h], x[..., h:]
        return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)

    def layer_states(self, codes):
        """The embedding and every layer at self.pos for input `codes` (K/V
        rows written at self.pos; the position is not advanced).  Returns the
        residual stream after the embedding and after each layer."""
        d = self.d
        D, NQ, NKV, I, eps = d.head_dim, d.n_q, d.n_kv, d.inter, d.rms_eps
        pos = self.pos
        h = torch.zeros(d.hidden, dtype=torch.float32)
        for k in range(d.n_cb):
            h = h + self.E[k, int(codes[k])]
        hs = [h]
        for l, P in enumerate(self.L):
            qkv = self._proj(P["wqkv"], rms_norm(h, P["ln_in"], eps))
            q = self._rope(rms_norm(qkv[:NQ * D].view(NQ, D), P["q_norm"], eps), pos)
            k = self._rope(rms_norm(qkv[NQ * D:(NQ + NKV) * D].view(NKV, D), P["k_norm"], eps), pos)
            v = qkv[(NQ + NKV) * D:].view(NKV, D)
            self.K[l, :, pos] = k.to(torch.bfloat16)
            self.V[l, :, pos] = v.to(torch.bfloat16)
            Kc = self.K[l, :, :pos + 1].to(torch.float32).repeat_interleave(NQ // NKV, 0)
            Vc = self.V[l, :, :pos + 1].to(torch.float32).repeat_interleave(NQ // NKV, 0)
            s = torch.einsum("hd,htd->ht", q, Kc) / np.float32(np.sqrt(D))
            p = torch.softmax(s, dim=-1)
            attn = torch.einsum("ht,htd->hd", p, Vc).reshape(-1)
            h = h + self._proj(P["wo"], attn)
            gu = self._proj(P["wgu"], rms_norm(h, P["ln_post"], eps))
            g, u = gu[:I], gu[I:]
            m = _round_bf16(g / (1.0 + torch.exp(-g)) * u)
            h = h + self._proj(P["wd"], m)
            hs.append(h)
        return hs

    def step(self, codes):
        """One frame at self.pos with input `codes`; returns (codes, logits
        float64 [n_cb][cb_vocab])."""
        d = self.d
        h = self.layer_states(codes)[-1]
        f = rms_norm(h, self.fn, d.rms_eps)
        logits = torch.mv(self.head, f).view(d.n_cb, d.cb_vocab).to(torch.float64).numpy()
        out = []
        for k in range(d.n_cb):
            am = int(np.argmax(logits[k]))
            if self.t < k:
                out.append(d.cb_vocab - 2)
            elif self.eoc >= 0 and self.t >= self.eoc + k:
                out.append(d.cb_vocab - 1)
            else:
                out.append(am)
        if self.eoc < 0 and out[0] == d.cb_vocab - 1:
            self.eoc = self.t
        self.pos += 1
        self.t += 1
        return np.array(out, np.int32), logits


def frame_stats(logits, or_logits, codes, or_codes, or_gaps, gap: float = 1e-2):
    """(logits cosine against the oracle, codes compared where the oracle's
    top-2 gap exceeds `gap`, how many of those differ)."""
    a = np.asarray(logits, np.float64).ravel()
    b = np.asarray(or_logits, np.float64).ravel()
    cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
    live = np.asarray(or_gaps) > gap
    return cos, int(live.sum()), int((np.asarray(codes)[live] != np.asarray(or_codes)[live]).sum())


def layerwise_spread(orc, hs_of_row, pos0: int, n_layers: int):
    """Per-row, per-layer contribution cosines of a run against the oracle's
    layer applied to the run's own input to that layer: hs_of_row(p) gives
    the run's residual stream [n_layers + 1] of prompt row p (position pos0 +
    p).  Layers outer, rows inner, so the oracle's cache for layer l holds the
    rows before p when row p is computed.  Returns the cosines, [n_layers][P]."""
    out = []
    P = len(hs_of_row)
    for l in range(n_layers):
        row = []
        for p in range(P):
            hin = np.asarray(hs_of_row[p][l], np.float64)
            ho = orc.layer(l, pos0 + p, hin)
            a, b = np.asarray(hs_of_row[p][l + 1], np.float64) - hin, ho - hin
            row.append(float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b))))
        out.append(row)
    return np.array(out)
