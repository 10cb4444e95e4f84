"""Injection of a dense verify block: the features of every request's block
sit at rows b*S of one buffer and only the first n_rows[b] of them are
committed.  With more than 128 feature rows the fused path gathers the
committed rows first and runs fc and the K/V projections on them alone (the
row count read from the device); the one-launch-per-GEMM path projects the
whole block and writes the committed rows.  Both are compared with the
oracle's context K/V, with empty, one-row and full commits and a request
whose rows lie outside the buffer (flagged, nothing written, length kept).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from synth import WORKLOADS, make_features  # noqa: E402
from synth.configs import shrink  # noqa: E402
from tests.harness import CycleRun, i32  # noqa: E402

QWEN_MINI = shrink(WORKLOADS["qwen8b-b1"].cfg, name="qwen-mini", target_hidden=256, hidden=512,
                   n_layers=2, n_heads=8, n_kv_heads=2, intermediate=1024, vocab=4096,
                   mask_token_id=4095)
ROW_RANGE = 0x40


@pytest.mark.parametrize("fused", [True, False], ids=["gathered", "whole-block"])
def test_dense_block_injection(fused):
    cfg = QWEN_MINI
    B, S = 12, cfg.block_size                       # 192 feature rows: more than one tile
    ctx = np.random.default_rng(31).integers(10, 200, B)
    run = CycleRun(cfg, B, ctx, cycles=0, seed=31, gains="random", permuted=True, fused=fused)
    run.prefill()
    assert run.sess.error() == 0
    n = np.array([0, S, 1, 5, S - 1, 7, 3, S, 0, 2, 9, 4])
    offs = np.arange(B) * S
    offs[-1] = B * S - 2                            # rows B*S-2 .. B*S+1: past the buffer
    feats = make_features(cfg, B * S, 31, "dense-block", device="cuda")
    run.sess.inject(run.kv, feats, i32(offs), i32(n))
    assert run.sess.error() & ROW_RANGE
    expect = ctx.copy()
    for b in range(B - 1):
        if n[b] > 0:
            run.ctx[b].inject(run._feat_rows(feats, slice(int(offs[b]), int(offs[b] + n[b]))), run.Wn)
            expect[b] += n[b]
    assert np.array_equal(run.kv.kv_len.cpu().numpy(), expect)
    run.compare_kv()
    assert run.sess.error() == 0


def test_gathered_rows_never_exceed_the_feature_rows():
    """Requests may share feature rows, but the gathered rows stop at the
    buffer's row count: here the commits sum to 208 of 192 rows, so the last
    request keeps its first 16 rows (flagged); every written row is checked."""
    cfg = QWEN_MINI
    B, S = 12, cfg.block_size
    ctx = np.random.default_rng(37).integers(10, 200, B)
    run = CycleRun(cfg, B, ctx, cycles=0, seed=37, gains="random", permuted=True, fused=True)
    run.prefill()
    assert run.sess.error() == 0
    offs = np.arange(B) * S
    n = np.full(B, S)
    offs[-1], n[-1] = 0, 2 * S                      # rows 0 .. 31, shared with request 0
    feats = make_features(cfg, B * S, 37, "shared-rows", device="cuda")
    run.sess.inject(run.kv, feats, i32(offs), i32(n))
    assert run.sess.error() & ROW_RANGE
    kept = n.copy()
    kept[-1] = B * S - int(n[:-1].sum())            # 16
    for b in range(B):
        run.ctx[b].inject(run._feat_rows(feats, slice(int(offs[b]), int(offs[b] + kept[b]))), run.Wn)
    assert np.array_equal(run.kv.kv_len.cpu().numpy(), ctx + kept)
    run.compare_kv()
    assert run.sess.error() == 0
