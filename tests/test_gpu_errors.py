"""Device-side error detection of injection and drafting (no fault is ever
provoked: the kernels check and skip, then the host reads the error word)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import block_diffusion_speculative_fc_gb300 as pkg  # noqa: E402
from synth import WORKLOADS, make_features, make_weights  # noqa: E402
from tests.harness import i32  # noqa: E402

CFG = WORKLOADS["tiny"].cfg


@pytest.fixture(scope="module")
def env():
    W = make_weights(CFG, device="cuda")
    s = pkg.DraftSession(CFG, W, max_batch=2, max_rows=256, max_position=512)
    yield s
    s.close()


def test_inject_past_capacity_is_flagged_and_clamped(env):
    kv = env.new_kv(2, 2, np.array([[0, 1], [2, 3]], dtype=np.int32))   # 128 rows each
    feats = make_features(CFG, 200, 0, "cap", device="cuda")
    env.inject(kv, feats, i32([0, 130]), i32([130, 10]))
    word = env.error()
    assert word & 0x1
    assert list(kv.kv_len.cpu().numpy()) == [128, 10]


def test_inject_rows_outside_buffer_are_flagged(env):
    kv = env.new_kv(1, 2, np.array([[0, 1]], dtype=np.int32))
    feats = make_features(CFG, 16, 0, "rows", device="cuda")
    env.inject(kv, feats, i32([10]), i32([20]), batch=1)
    assert env.error() & 0x40
    assert int(kv.kv_len[0].item()) == 0


def test_bad_page_id_and_bad_anchor_are_flagged(env):
    kv = env.new_kv(1, 2, np.array([[0, 1]], dtype=np.int32))
    kv.page_table[0, 1] = 99                         # outside the pool
    feats = make_features(CFG, 100, 0, "pages", device="cuda")
    env.inject(kv, feats, i32([0]), i32([100]), batch=1)
    assert env.error() & 0x2
    draft = torch.zeros((1, CFG.block_size), dtype=torch.int32, device="cuda")
    env.draft(kv, i32([CFG.vocab + 1]), draft, batch=1)
    assert env.error() & 0x4


def test_negative_sizes_are_refused_on_host(env):
    kv = env.new_kv(1, 1, np.array([[0]], dtype=np.int32))
    feats = make_features(CFG, 4, 0, "neg", device="cuda")
    with pytest.raises(pkg.DFlashError):
        pkg.dflash_inject_context(env.h, kv.struct, -1, 4, [feats[j] for j in range(3)],
                                  i32([0]), i32([4]), None)
    with pytest.raises(pkg.DFlashError) as ei:
        env.draft(kv, i32([1, 2, 3]), torch.zeros((3, 4), dtype=torch.int32, device="cuda"),
                  batch=3)
    assert ei.value.status == -3
