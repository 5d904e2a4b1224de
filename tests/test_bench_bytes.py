"""The roofline's algorithmic bytes (bench.step_bytes) against an independent
count: the byte sizes of the arrays the seeded generator actually builds for
a model (every weight, scale and gain once, the embedding rows of one frame,
the cached K/V rows read and the new one written).  No GPU."""
import numpy as np

import bench
import synth


def _arrays_bytes(w, precision: int) -> int:
    layers = 0
    for l in range(w.dims.n_layers):
        for m in (w.wqkv[l], w.wo[l], w.wgu[l], w.wd[l]):
            # bf16: two bytes a weight; E4M3: one byte a weight and an fp32 scale per row
            layers += m.nbytes if precision == 0 else m.size + 4 * m.shape[0]
        layers += sum(g.nbytes for g in (w.ln_in[l], w.ln_post[l], w.q_norm[l], w.k_norm[l]))
    return layers + w.head.nbytes + w.final_norm.nbytes


def test_step_bytes_counts_every_array_once():
    d = synth.Dims(n_layers=2, hidden=512, n_q=8, n_kv=2, head_dim=128, inter=1024, n_cb=8, cb_vocab=1026)
    w = synth.make_weights(d)
    embed_rows = d.n_cb * w.embed[0][0].nbytes          # one row of each codebook table
    for ctx in (1, 37, 300):
        kv = d.n_layers * 2 * d.n_kv * d.head_dim * 2 * ctx  # ctx - 1 cached rows read, one row written
        for precision in (0, 1):
            assert bench.step_bytes(d, precision, ctx) == _arrays_bytes(w, precision) + embed_rows + kv



def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    """bench.read_traffic scales a capture to n layers (fixed + n x per layer)
    and refuses a record whose source digest is not the kernel's."""
    import json
    (tmp_path / "profiles").mkdir()
    rec = {"source_digest": "abc", "method": "m",
           "workloads": {"w": {"fixed": 1000.0, "per_layer": 10.0}}}
    (tmp_path / "profiles" / "step_kernel_traffic.txt").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "abc")
    assert bench.read_traffic("w", 36)[0] == 1000.0 + 36 * 10.0
    assert bench.read_traffic("other", 36)[0] is None
    monkeypatch.setattr(bench, "source_digest", lambda: "changed")
    assert bench.read_traffic("w", 36)[0] is None
