"""Acceptance / commit kernel: bit-exact against the oracle on every match
pattern, plus the device error paths."""
import itertools

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import block_diffusion_speculative_fc_gb300 as pkg  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402
from synth import WORKLOADS, make_weights  # noqa: E402
from synth.configs import shrink  # noqa: E402
from tests.harness import i32  # noqa: E402

CFG = shrink(WORKLOADS["tiny"].cfg, name="acc", block_size=16)


@pytest.fixture(scope="module")
def sess():
    W = make_weights(CFG, device="cuda")
    s = pkg.DraftSession(CFG, W, max_batch=1 << 15, max_rows=16, max_position=4096)
    yield s
    s.close()


@pytest.mark.parametrize("S", [2, 4, 8, 16])
def test_accept_all_match_patterns(sess, S):
    cfg = shrink(CFG, block_size=S)
    W = make_weights(cfg, device="cuda")
    s = pkg.DraftSession(cfg, W, max_batch=1 << (S - 1), max_rows=16, max_position=4096)
    rng = np.random.default_rng(S)
    pats = np.array(list(itertools.product([0, 1], repeat=S - 1)), dtype=bool)
    B = len(pats)
    draft = rng.integers(0, 500, (B, S))
    post = rng.integers(500, 1000, (B, S))
    post[:, :-1] = np.where(pats, draft[:, 1:], post[:, :-1])
    start = rng.integers(0, 40, B)
    stride = 64
    out_ids = np.full((B, stride), 7, dtype=np.int64)
    d_out = i32(out_ids)
    seq = i32(start)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    com, bon = torch.zeros_like(acc), torch.zeros_like(acc)
    tok = torch.zeros((B, S), dtype=torch.int32, device="cuda")
    s.accept(B, i32(draft), i32(post), seq, acc, com, bon, tok, d_out)
    acc_g, com_g, bon_g = acc.cpu().numpy(), com.cpu().numpy(), bon.cpu().numpy()
    tok_g, seq_g, ids_g = tok.cpu().numpy(), seq.cpu().numpy(), d_out.cpu().numpy()
    for b in range(B):
        a, bonus, commit, out = O.accept_block(draft[b], post[b])
        ref_ids, ref_start = O.commit_output(out_ids[b], int(start[b]), draft[b], a, bonus)
        assert (acc_g[b], com_g[b], bon_g[b], seq_g[b]) == (a, commit, bonus, ref_start)
        assert np.array_equal(tok_g[b], out)
        assert np.array_equal(ids_g[b], ref_ids)
    assert s.error() == 0
    s.close()


def test_accept_flags_bad_ids_and_output_overflow(sess):
    S = CFG.block_size
    draft = np.tile(np.arange(S), (3, 1))
    post = np.roll(draft, -1, axis=1)                      # everything matches
    draft[1, 0] = CFG.vocab + 5                            # row 1: anchor id out of range
    seq = i32([0, 0, 60])                                  # row 2: overflows stride 64
    out = torch.zeros((3, 64), dtype=torch.int32, device="cuda")
    acc = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    com, bon = acc.clone(), acc.clone()
    tok = torch.zeros((3, S), dtype=torch.int32, device="cuda")
    sess.accept(3, i32(draft), i32(post), seq, acc, com, bon, tok, out)
    word = sess.error()
    assert word & 0x4 and word & 0x10
    a = acc.cpu().numpy()
    assert a[0] == S - 1 and a[1] == -1 and a[2] == -1     # flagged rows are not written
    assert list(seq.cpu().numpy()) == [S, 0, 60]
    assert sess.error() == 0                               # the word was cleared


def test_host_validation_refuses_oversized_batch(sess):
    S = CFG.block_size
    z = torch.zeros((1, S), dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DFlashError) as ei:
        sess.accept((1 << 15) + 1, z, z, z, z, z, z, z)
    assert ei.value.status == -3
