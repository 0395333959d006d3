"""The bench's roofline accounting (CPU): the algorithmic bytes and flops of one forward counted
independently from the config, and the rule that a stored ncu traffic figure is only used while
the measured kernel's sources are unchanged."""
import json

import numpy as np

import bench
from synth import CONFIGS, make_workload


def _count(cfg, ctx_lens, logits=True):
    """Bytes and flops of one gamma-block forward, counted tensor by tensor."""
    es = 2 if cfg.dtype == "bf16" else 4
    H, F, V, hd = cfg.hidden, cfg.n_ff, cfg.vocab, cfg.head_dim
    nh, nkv, L, g = cfg.n_q_heads, cfg.n_kv_heads, cfg.n_layers, cfg.gamma
    M = len(ctx_lens) * g
    per_layer = {
        "wq": nh * hd * H, "wk": nkv * hd * H, "wv": nkv * hd * H, "wo": H * nh * hd,
        "w_gate": F * H, "w_up": F * H, "w_down": H * F,
        "ln_in": H, "ln_post": H, "q_norm": hd, "k_norm": hd,
    }
    weights = L * sum(per_layer.values()) * es + V * H * es
    visible = 0
    for c in ctx_lens:
        for l in range(L):
            sliding = cfg.sliding(l) and cfg.sliding_window > 0
            visible += min(c + g, cfg.sliding_window + g - 1) if sliding else c + g
    kv_read = visible * 2 * nkv * hd * es          # K and V of every visible key, once per layer
    kv_write = L * M * 2 * nkv * hd * es           # the block's K/V rows
    embed = M * H * es                             # embedding rows gathered
    out = M * V * es if logits else 0
    matmul = sum(v for k, v in per_layer.items() if k.startswith("w")) * L + V * H
    flops = 2 * M * matmul + sum(4 * g * nh * hd * (min(c + g, cfg.sliding_window + g - 1)
                                                   if (cfg.sliding(l) and cfg.sliding_window > 0) else c + g)
                                 for c in ctx_lens for l in range(L))
    return weights + kv_read + kv_write + embed + out, flops


def test_work_model_matches_an_independent_count():
    for name, ctxs in (("qwen3_8l_bf16", [4096]), ("qwen3_8l_bf16", [512, 8192, 3000]),
                       ("wide_5l_yarn_bf16", [16384]), ("wide_5l_yarn_bf16", [100])):
        cfg = CONFIGS[name]
        wl = make_workload(cfg, 1, ctxs)
        for logits in (True, False):
            nbytes, flops, per_kernel = bench.work_model(cfg, wl, logits)
            b, f = _count(cfg, ctxs, logits)
            assert nbytes == b, (name, ctxs, logits, nbytes, b)
            assert flops == f, (name, ctxs, logits, flops, f)
            assert per_kernel["persistent_forward"] == (nbytes, flops)


def test_headline_bytes():
    # 8-layer drafter, one sequence, context 4096, logits written: the figure the bench's
    # roofline divides by (235 us at the measured 6.8 TB/s)
    cfg = CONFIGS["qwen3_8l_bf16"]
    nbytes, _, _ = bench.work_model(cfg, make_workload(cfg, 2, [4096]), True)
    assert nbytes == 1_600_929_792


def test_stored_traffic_only_for_unchanged_sources(tmp_path, monkeypatch):
    sha = bench.kernel_sources_sha("persistent_forward")
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"persistent_forward@w": {"dram_bytes_per_launch": 123, "sources_sha": sha}}
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench.os.path, "abspath", lambda p: str(tmp_path / "bench.py")
                        if p == bench.__file__ else p)
    # the record is looked up next to bench.py; the kernel sources stay where they are
    real_sha = bench.kernel_sources_sha
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda k="persistent_forward", read=None: real_sha(k, read)
                        if read else sha)
    assert bench.measured_traffic("persistent_forward", "w") == 123
    assert bench.measured_traffic("persistent_forward", "other") is None
    assert bench.measured_traffic("attention", "w") is None
    rec["persistent_forward@w"]["sources_sha"] = "0" * 16
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.measured_traffic("persistent_forward", "w") is None


def test_sources_hash_follows_the_kernel_files():
    files = {f: f.encode() * 3 for f in bench.KERNEL_SOURCES["persistent_forward"]}
    a = bench.kernel_sources_sha("persistent_forward", lambda f: files[f])
    files["persist_tc.cu"] += b"// changed"
    b = bench.kernel_sources_sha("persistent_forward", lambda f: files[f])
    assert a != b and len(a) == 16
    assert np.all([f.endswith((".cu", ".cuh")) for f in files])
