"""Host logic of the benchmark on CPU: the algorithmic byte/flop model the
roofline line divides by, and the choice of bound and peak.

The per-launch bytes at the batch-1 Qwen shape are the weights each fused
launch must stream plus its activations; they are checked against the sizes
computed here from the weight shapes (a launch streams every weight matrix
of its GEMMs once) and the figures the design notes quote.
"""
from types import SimpleNamespace

import numpy as np
import pytest

import bench
from synth import WORKLOADS

QWEN = WORKLOADS["qwen8b-b1"].cfg


def _weights(cfg):
    H, D = cfg.hidden, cfg.head_dim
    qd, kvd = cfg.n_heads * D, cfg.n_kv_heads * D
    return {
        "o": H * qd, "gate_up": 2 * cfg.intermediate * H, "down": H * cfg.intermediate,
        "qkv": (qd + 2 * kvd) * H, "lm_head": cfg.vocab * H,
        "fc": H * cfg.n_sel * cfg.target_hidden, "kv": cfg.n_layers * 2 * kvd * H,
    }


def test_program_bytes_are_the_streamed_weights_plus_activations():
    fam = bench.algorithmic(QWEN, 1, 1024.0, 6.4)
    w = {k: 2 * v for k, v in _weights(QWEN).items()}      # bf16
    layer = w["o"] + w["gate_up"] + w["down"] + w["qkv"]
    last = w["o"] + w["gate_up"] + w["down"] + w["lm_head"]
    norm = (4 + 2) * 16 * QWEN.hidden + 4 * 16 * (QWEN.hidden // 128)   # the final norm phase
    inject = w["fc"] + w["kv"]
    # activations and outputs of 16 rows add well under 1% to the weights
    assert layer <= fam["gemm_layer_program"][0] <= layer * 1.01
    assert last + norm <= fam["gemm_last_program"][0] <= last * 1.01
    assert inject <= fam["gemm_inject_program"][0] <= inject * 1.01
    # the figures of the design notes (MB per launch)
    assert fam["gemm_layer_program"][0] / 1e6 == pytest.approx(388.3, abs=0.1)
    assert fam["gemm_last_program"][0] / 1e6 == pytest.approx(1582.8, abs=0.1)
    # (the injection projects the committed rows only: 6.4 of the block's 16)
    assert fam["gemm_inject_program"][0] / 1e6 == pytest.approx(252.2, abs=0.1)
    # a program is the sum of its GEMMs
    parts = [fam[n] for n in ("gemm_o", "gemm_gate_up", "gemm_down", "gemm_qkv")]
    assert fam["gemm_layer_program"] == tuple(sum(p[i] for p in parts) for i in range(2))


def _fake(cfg, B, ctx):
    return SimpleNamespace(cfg=cfg, B=B, T=np.full(B, ctx))


def test_roofline_bound_peak_and_fraction():
    hbm, tf, tf_sus, src = bench.peaks()
    # batch 1: the layer program is HBM-bound; 4 launches of 98.75 us per cycle
    r = bench.dominant_roofline(_fake(QWEN, 1, 1024), {"gemm_layer_program": (4.0, 0.395),
                                                       "attention": (5.0, 0.082)}, 6.4, "qwen8b-b1")
    fam = bench.algorithmic(QWEN, 1, 1024.0, 6.4)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == hbm
    assert r["kernel"] == "gemm_layer_program"
    assert r["achieved"] == pytest.approx(fam["gemm_layer_program"][0] / (0.395e-3 / 4) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / hbm)
    assert r["share"] == pytest.approx(0.395 / 0.477)
    assert r["peak_source"] == src
    # 512 rows: the same launch is a contraction, judged against the sustained bf16 peak
    r32 = bench.dominant_roofline(_fake(QWEN, 32, 2048), {"gemm_layer_program": (4.0, 1.66)},
                                  6.4, "qwen8b-b32")
    assert r32["bound"] == "tensor" and r32["unit"] == "TFLOP/s" and r32["peak"] == tf_sus
    fam32 = bench.algorithmic(QWEN, 32, 2048.0, 6.4)
    assert r32["achieved"] == pytest.approx(fam32["gemm_layer_program"][1] / (1.66e-3 / 4) / 1e12)


def test_attention_bytes_follow_the_cache_type_and_the_windows():
    """Context K/V bytes: one byte per element with the FP8 cache (half of
    bf16), and only the keys a layer can see under its sliding window and the
    draft window."""
    T = np.array([100.0, 5000.0, 30000.0])
    bf = bench.algorithmic(QWEN, 3, T, 6.4)["attention"][0]
    f8 = bench.algorithmic(QWEN, 3, T, 6.4, kv_fp8=True)["attention"][0]
    kvd, S = QWEN.n_kv_heads * QWEN.head_dim, QWEN.block_size
    ctx_bf = 2 * 2 * T.sum() * kvd
    assert bf - f8 == pytest.approx(ctx_bf / 2)
    win = bench.algorithmic(QWEN, 3, T, 6.4, draft_window=4096)["attention"][0]
    assert bf - win == pytest.approx(2 * 2 * kvd * (T - np.minimum(T, 4096)).sum())
    kimi = WORKLOADS["kimi-b8"].cfg            # five layers of window 2048, one full
    keys = bench.visible_keys(kimi, np.full(8, 8192.0))
    assert keys == pytest.approx(8 * (5 * 2048 + 8192) / 6)
    assert S == 16


def test_traffic_entries_follow_their_kernel_sources():
    """The DRAM bytes of a committed capture stay valid only while the sources
    of that kernel family are unchanged: every listed file exists, the GEMM
    and attention families differ, and a launch name outside them hashes all
    sources."""
    import os
    csrc = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)),
                        "block_diffusion_speculative_fc_gb300", "csrc")
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), f
    assert "gemm_tc.cu" in bench.KERNEL_SOURCES["gemm"]
    assert "attention_tc.cu" in bench.KERNEL_SOURCES["attention"]
    g, a = bench.source_hash("gemm_layer_program"), bench.source_hash("attention")
    assert g != a and bench.source_hash("gemm_inject_program") == g
    assert bench.source_hash() not in (g, a)
