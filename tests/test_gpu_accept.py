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


# ------------------------------------------------ sampled (lossless) verification
def _sampled_case(rng, B, S, V, favour=0.7):
    """Drafts, target rows (softmax of random logits, the next draft boosted
    in some rows so that acceptance runs vary), uniforms, Exp(1) noise."""
    draft = rng.integers(0, V, (B, S))
    logits = rng.standard_normal((B, S, V)).astype(np.float32) * 2.0
    boost = rng.random((B, S - 1)) < favour
    for b in range(B):
        for i in range(S - 1):
            if boost[b, i]:
                logits[b, i, draft[b, i + 1]] += rng.uniform(2.0, 12.0)
    p = np.exp(logits - logits.max(-1, keepdims=True))
    p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
    u = rng.random((B, S - 1)).astype(np.float32)
    e = rng.exponential(size=(B, V)).astype(np.float32)
    return draft, p, u, e


def _run_sampled(s, draft, p, u, e, start, stride=64):
    B, S = draft.shape
    out_ids = np.full((B, stride), 7, dtype=np.int64)
    d_out = i32(out_ids)
    seq = i32(start)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    com, bon = torch.zeros_like(acc), torch.zeros_like(acc)
    tok = torch.zeros((B, S), dtype=torch.int32, device="cuda")
    f32 = lambda a: torch.as_tensor(a, dtype=torch.float32, device="cuda")  # noqa: E731
    s.accept_sampled(B, i32(draft), f32(p), f32(u), f32(e), seq, acc, com, bon, tok, d_out)
    return (out_ids, acc.cpu().numpy(), com.cpu().numpy(), bon.cpu().numpy(), tok.cpu().numpy(),
            seq.cpu().numpy(), d_out.cpu().numpy())


@pytest.mark.parametrize("B,S,V", [(1, 16, 1000), (37, 8, 3001), (5, 16, 151936)])
def test_sampled_accept_bit_exact(B, S, V):
    """Every decision (acceptance compare, race quotient, argmax) is a float32
    operation both sides take identically: outputs must match exactly."""
    cfg = shrink(CFG, block_size=S, vocab=V, mask_token_id=V - 1)
    W = make_weights(cfg, device="cuda")
    s = pkg.DraftSession(cfg, W, max_batch=B, max_rows=16, max_position=4096)
    rng = np.random.default_rng(B * 1000 + S)
    for rep in range(3):
        draft, p, u, e = _sampled_case(rng, B, S, V)
        start = rng.integers(0, 40, B)
        out_ids, acc_g, com_g, bon_g, tok_g, seq_g, ids_g = _run_sampled(s, draft, p, u, e, start)
        for b in range(B):
            a, bonus, commit, out = O.accept_block_sampled(draft[b], p[b], u[b], e[b])
            ref_ids, ref_start = O.commit_output(out_ids[b], int(start[b]), draft[b], a, bonus)
            assert (acc_g[b], com_g[b], bon_g[b], seq_g[b]) == (a, commit, bonus, ref_start), (rep, b)
            assert np.array_equal(tok_g[b], out)
            assert np.array_equal(ids_g[b], ref_ids)
    assert s.error() == 0
    s.close()


def test_sampled_accept_edge_cases():
    """Certain acceptance (target one-hot at the drafts), certain rejection
    (p(y) = 0: the correction never repeats y), equal race keys (lowest id),
    and an out-of-vocabulary draft (flagged, request not committed)."""
    B, S, V = 4, 8, 64
    cfg = shrink(CFG, block_size=S, vocab=V, mask_token_id=V - 1)
    W = make_weights(cfg, device="cuda")
    s = pkg.DraftSession(cfg, W, max_batch=B, max_rows=16, max_position=4096)
    rng = np.random.default_rng(3)
    draft = rng.integers(0, V, (B, S))
    p = np.full((B, S, V), 1.0 / V, np.float32)
    p[0] = 0.0
    p[0, np.arange(S - 1), draft[0, 1:]] = 1.0          # request 0: every draft certain
    p[0, S - 1, 9] = 1.0
    p[1, 0, draft[1, 1]] = 0.0                          # request 1: first draft impossible
    u = rng.random((B, S - 1)).astype(np.float32)
    e = rng.exponential(size=(B, V)).astype(np.float32)
    e[2] = 1.0                                          # request 2: all keys equal where p equal
    u[2] = 0.999
    start = np.zeros(B, dtype=np.int64)
    out_ids, acc_g, com_g, bon_g, tok_g, seq_g, ids_g = _run_sampled(s, draft, p, u, e, start)
    assert (acc_g[0], bon_g[0]) == (S - 1, 9)
    assert acc_g[1] == 0 and bon_g[1] != draft[1, 1]
    a2, b2, _, _ = O.accept_block_sampled(draft[2], p[2], u[2], e[2])
    assert (acc_g[2], bon_g[2]) == (a2, b2) and a2 == 0
    assert b2 == (0 if draft[2, 1] != 0 else 1)         # lowest id among equal keys
    assert s.error() == 0
    bad = draft.copy()
    bad[3, 1] = V + 5
    seq = i32(np.full(B, 11))
    acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    com, bon = torch.zeros_like(acc), torch.zeros_like(acc)
    tok = torch.zeros((B, S), dtype=torch.int32, device="cuda")
    f32 = lambda a: torch.as_tensor(a, dtype=torch.float32, device="cuda")  # noqa: E731
    s.accept_sampled(B, i32(bad), f32(p), f32(u), f32(e), seq, acc, com, bon, tok)
    word = s.error()
    assert "TOKEN_RANGE" in pkg.decode_error(word)
    assert seq.cpu().numpy()[3] == 11 and acc.cpu().numpy()[3] == -1
    s.close()


# ------------------------------------- sampled verification with a real proposal
def _q_case(rng, B, S, V, K):
    """K distinct candidates per position (the draft token among them in most
    positions, absent in some), proposal probabilities q over them, target
    rows p, uniforms and noise."""
    draft, p, u, e = _sampled_case(rng, B, S, V)
    cand = np.empty((B, S - 1, K), np.int64)
    q = np.empty((B, S - 1, K), np.float32)
    for b in range(B):
        for i in range(S - 1):
            c = rng.choice(V, size=K, replace=False)
            if rng.random() < 0.85 and draft[b, i + 1] not in c:
                c[rng.integers(K)] = draft[b, i + 1]
            cand[b, i] = c
            q[b, i] = rng.dirichlet(np.full(K, 0.7)).astype(np.float32)
    return draft, p, cand, q, u, e


@pytest.mark.parametrize("B,S,V,K", [(1, 16, 1000, 8), (29, 8, 3001, 3), (4, 16, 151936, 8),
                                     (6, 4, 64, 1)])
def test_sampled_q_accept_bit_exact(B, S, V, K):
    """Acceptance u < p(y)/q(y), residual [p - q]+ and the race are float32
    operations both sides take identically: outputs must match exactly."""
    cfg = shrink(CFG, block_size=S, vocab=V, mask_token_id=V - 1)
    W = make_weights(cfg, device="cuda")
    s = pkg.DraftSession(cfg, W, max_batch=B, max_rows=16, max_position=4096)
    rng = np.random.default_rng(B * 7 + K)
    f32 = lambda a: torch.as_tensor(a, dtype=torch.float32, device="cuda")  # noqa: E731
    for rep in range(3):
        draft, p, cand, q, u, e = _q_case(rng, B, S, V, K)
        start = rng.integers(0, 40, B)
        out_ids = np.full((B, 64), 7, dtype=np.int64)
        d_out = i32(out_ids)
        seq = i32(start)
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        com, bon = torch.zeros_like(acc), torch.zeros_like(acc)
        tok = torch.zeros((B, S), dtype=torch.int32, device="cuda")
        s.accept_sampled_q(B, i32(draft), f32(p), i32(cand), f32(q), f32(u), f32(e), seq, acc, com,
                           bon, tok, d_out)
        acc_g, com_g, bon_g = acc.cpu().numpy(), com.cpu().numpy(), bon.cpu().numpy()
        tok_g, seq_g, ids_g = tok.cpu().numpy(), seq.cpu().numpy(), d_out.cpu().numpy()
        for b in range(B):
            a, bonus, commit, out = O.accept_block_sampled_q(draft[b], p[b], cand[b], q[b], u[b], e[b])
            ref_ids, ref_start = O.commit_output(out_ids[b], int(start[b]), draft[b], a, bonus)
            assert (acc_g[b], com_g[b], bon_g[b], seq_g[b]) == (a, commit, bonus, ref_start), (rep, b)
            assert np.array_equal(tok_g[b], out) and np.array_equal(ids_g[b], ref_ids)
    assert s.error() == 0
    s.close()
