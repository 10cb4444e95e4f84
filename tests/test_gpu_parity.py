"""GPU parity of the full draft-verify cycle against the CPU oracle.

Workloads at sizes the oracle finishes in seconds, spanning several tiles and
ragged tails (context lengths that are not page multiples, vocabularies that
are not tile multiples), plus the shapes of the five named workloads.
"""
import numpy as np
import pytest

from synth import WORKLOADS
from synth.configs import shrink

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from tests.harness import CycleRun  # noqa: E402

TINY = WORKLOADS["tiny"].cfg
QWEN = WORKLOADS["qwen8b-b1"].cfg
KIMI = WORKLOADS["kimi-b8"].cfg

QWEN_MINI = shrink(QWEN, name="qwen-mini", target_hidden=256, hidden=512, n_layers=2, n_heads=8,
                   n_kv_heads=2, intermediate=1024, vocab=4096, mask_token_id=4095)
KIMI_MINI = shrink(KIMI, name="kimi-mini", target_hidden=256, target_layer_ids=(1, 12, 24),
                   hidden=512, n_layers=3, n_heads=8, n_kv_heads=1, intermediate=768,
                   vocab=3000, mask_token_id=2998, sliding_window=(64, 64, 0))


def _report(stats):
    print({k: (max(v) if isinstance(v, list) and v else v)
           for k, v in stats.items() if k not in ("accept", "e2e_flips")},
          "e2e flips", len(stats["e2e_flips"]),
          "mean accept", float(np.mean(stats["accept"])) if stats["accept"] else None)


def test_tiny_f32_eight_cycles():
    run = CycleRun(TINY, 1, [32], cycles=8, match=("bernoulli", 0.8))
    _report(run.run())


def test_tiny_f32_random_gains_batch3():
    run = CycleRun(TINY, 3, [32, 5, 70], cycles=4, gains="random", permuted=True,
                   match=("bernoulli", 0.8))
    _report(run.run())


def test_qwen_mini_bf16_b1_ragged_context():
    run = CycleRun(QWEN_MINI, 1, [100], cycles=4, gains="random")
    _report(run.run())


def test_qwen_mini_bf16_paged_batch():
    run = CycleRun(QWEN_MINI, 5, [30, 300, 64, 1, 129], cycles=3, permuted=True,
                   match=("bernoulli_per_req", 0.6, 0.95))
    _report(run.run())


def test_kimi_mini_sliding_window():
    run = CycleRun(KIMI_MINI, 3, [150, 40, 64], cycles=4, gains="random", permuted=True)
    _report(run.run())


def test_stress_mini_geometric_commits():
    cfg = shrink(QWEN_MINI, name="stress-mini", block_size=8)
    run = CycleRun(cfg, 16, np.random.default_rng(3).integers(8, 200, 16), cycles=3,
                   permuted=True, match=("geometric", 6.4), check=[0, 7, 15])
    _report(run.run())


def test_prefill_chunked_equals_single_chunk():
    """max_rows smaller than the prefill: the chunked injection must match."""
    run = CycleRun(QWEN_MINI, 2, [150, 90], cycles=1, max_rows=64, permuted=True)
    _report(run.run())


def test_qwen_mini_long_contexts_multi_page_splits():
    """Contexts of thousands of rows: attention splits span several pages and
    are merged across splits."""
    run = CycleRun(QWEN_MINI, 4, [1500, 2100, 700, 3000], cycles=2, permuted=True,
                   check=[0, 3], max_rows=2048)
    _report(run.run())


def test_kimi_mini_long_context_window_edge():
    """Window 64 against contexts far longer than the window."""
    run = CycleRun(KIMI_MINI, 2, [1000, 130], cycles=3, permuted=True)
    _report(run.run())


def test_many_request_heads_use_the_split_attention():
    """80 (request, KV head) pairs: more than the cluster path takes, so the
    persistent split kernel with ticketed merges runs (windowed layer too)."""
    cfg = shrink(QWEN_MINI, name="many-pairs", sliding_window=(100, 0))
    lens = np.random.default_rng(5).integers(20, 700, 40)
    run = CycleRun(cfg, 40, lens, cycles=2, permuted=True, check=[0, 17, 39])
    _report(run.run())


@pytest.mark.parametrize("fused", [False, True])
def test_qwen_mini_fused_and_split_launches(fused):
    """The per-layer GEMM chain and the injection as one fused launch each, or
    as one launch per GEMM: both must match the oracle."""
    run = CycleRun(QWEN_MINI, 3, [100, 37, 260], cycles=3, gains="random", permuted=True,
                   fused=fused)
    _report(run.run())


def test_kimi_mini_fused_launches():
    run = CycleRun(KIMI_MINI, 2, [150, 64], cycles=3, gains="random", permuted=True, fused=True)
    _report(run.run())
