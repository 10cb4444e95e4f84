"""Pins of the CPU oracle against what the pages and the mathematics fix.

No check here re-types an oracle formula: each one uses a worked example
printed on the pages (tests/golden/), a closed form, an invariant, a special
case with a known answer, or brute force over tiny inputs.
"""
import itertools
import json
import math
import os
from types import SimpleNamespace

import numpy as np
import pytest

from oracle import dflash_oracle as O
from tests.loop_restatement import draft_forward_loops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def tiny_cfg(**over):
    base = dict(hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=48, vocab=40,
                mask_token_id=39, block_size=4, n_layers=2, sliding_window=(0, 0),
                rms_eps=1e-6, rope_theta=10000.0, target_hidden=16, target_layer_ids=(0, 2, 4))
    base.update(over)
    c = SimpleNamespace(**base)
    c.n_sel = len(c.target_layer_ids)
    return c


def tiny_weights(cfg, rng, gains=True):
    H, D = cfg.hidden, cfg.head_dim
    g = (lambda n: rng.uniform(0.5, 1.5, n)) if gains else (lambda n: np.ones(n))
    W = {"fc": rng.normal(0, 0.2, (H, cfg.n_sel * cfg.target_hidden)),
         "hidden_norm": g(H), "final_norm": g(H),
         "embed": rng.normal(0, 1.0, (cfg.vocab, H)),
         "lm_head": rng.normal(0, 0.3, (cfg.vocab, H)), "layers": []}
    for _ in range(cfg.n_layers):
        W["layers"].append({
            "qkv": rng.normal(0, 0.3, ((cfg.n_heads + 2 * cfg.n_kv_heads) * D, H)),
            "o": rng.normal(0, 0.2, (H, cfg.n_heads * D)),
            "gate_up": rng.normal(0, 0.2, (2 * cfg.intermediate, H)),
            "down": rng.normal(0, 0.2, (H, cfg.intermediate)),
            "in_norm": g(H), "post_norm": g(H), "q_norm": g(D), "k_norm": g(D)})
    return W


# ----------------------------------------------------------------- acceptance
def test_accept_worked_example_p1():
    gd = _golden("accept_worked_example_p1.json")
    voc, ex = gd["vocab"], gd["expected"]
    draft = [voc[t] for t in gd["block"]]
    post = [voc[t] for t in gd["target_choices"]]
    acc, bonus, commit, out = O.accept_block(draft, post)
    assert acc == ex["accept_len"] and commit == ex["commit_len"]
    assert bonus == voc[ex["bonus"]]
    assert list(out[:commit]) == [voc[t] for t in ex["out_tokens_valid"]]
    L = gd["prefix_len"]
    assert list(L + np.arange(len(draft))) == ex["block_positions"]
    output_ids = np.full(32, -1)
    output_ids[L] = voc["of"]
    new_ids, new_start = O.commit_output(output_ids, L, draft, acc, bonus)
    assert new_start == ex["new_seq_len"] == ex["next_anchor_position"]
    # inputs whose target state became valid, and the emitted tokens, at their positions
    assert [new_ids[p] for p in ex["computed_positions"]] == [voc[t] for t in ex["computed_inputs"]]
    assert [new_ids[p] for p in ex["emitted_positions"]] == [voc[t] for t in ex["out_tokens_valid"]]
    assert new_ids[new_start] == voc[ex["next_anchor"]]


def test_accept_block5_example_p3():
    gd = _golden("accept_block5_example_p3.json")
    voc, ex = gd["vocab"], gd["expected"]
    acc, bonus, commit, out = O.accept_block([voc[t] for t in gd["candidates"]],
                                             [voc[t] for t in gd["target"]])
    assert commit == ex["accept_lens"]
    assert bonus == voc[ex["verified_id"]]
    assert list(out) == [voc[t] if isinstance(t, str) else t for t in ex["out_tokens"]]


def test_accept_zero_and_full():
    # zero survivors: one correction is emitted, the old anchor's state commits
    acc, bonus, commit, out = O.accept_block([7, 1, 2, 3], [9, 1, 2, 3])
    assert (acc, bonus, commit) == (0, 9, 1) and list(out) == [9, 0, 0, 0]
    # all survive: S-1 drafts plus a bonus from the last target row
    acc, bonus, commit, out = O.accept_block([7, 1, 2, 3], [1, 2, 3, 5])
    assert (acc, bonus, commit) == (3, 5, 4) and list(out) == [1, 2, 3, 5]


@pytest.mark.parametrize("S", [2, 3, 4, 8, 16])
def test_accept_bruteforce_all_patterns(S):
    rng = np.random.default_rng(S)
    for bits in itertools.product([0, 1], repeat=S - 1):
        draft = rng.integers(0, 100, S)
        post = rng.integers(100, 200, S)           # never equal to a draft
        for i, b in enumerate(bits):
            if b:
                post[i] = draft[i + 1]
        n = 0                                       # explicit first-mismatch loop
        while n < S - 1 and bits[n]:
            n += 1
        acc, bonus, commit, out = O.accept_block(draft, post)
        assert acc == n and commit == n + 1 and bonus == post[n]
        assert list(out[:n]) == list(draft[1:n + 1]) and out[n] == post[n]
        assert all(v == 0 for v in out[n + 1:])


def test_commit_crop_accumulates():
    # the z-lab loop advances start by acceptance_length + 1 every cycle
    ids = np.zeros(64, dtype=np.int64)
    start = 5
    for acc in [0, 3, 1, 3]:
        draft = np.arange(100, 104)
        ids, new_start = O.commit_output(ids, start, draft, acc, 999)
        assert new_start == start + acc + 1
        assert ids[new_start] == 999
        assert list(ids[start:start + acc + 1]) == list(draft[:acc + 1])
        start = new_start


# ------------------------------------------------------- context feature concat
def test_extract_context_feature_offset_and_order():
    # hidden_states[k] is the constant k: the embedding output is index 0
    hs = [np.full((3, 4), float(k)) for k in range(8)]
    f = O.extract_context_feature(hs, [0, 2, 4])
    assert f.shape == (3, 12)
    for j, lid in enumerate([0, 2, 4]):
        assert np.all(f[:, 4 * j:4 * (j + 1)] == lid + 1)


def test_concat_column_blocks_reach_fc_in_list_order():
    rows, Ht, n_sel, H = 3, 5, 3, 15
    feats = [np.full((rows, Ht), j + 1.0) + np.arange(Ht) * 0.01 for j in range(n_sel)]
    # fc rows are one-hot selectors: output r reads concat column r
    fc = np.eye(H, n_sel * Ht)
    y = O.linear(np.concatenate(feats, -1), fc)
    for j in range(n_sel):
        assert np.allclose(y[:, j * Ht:(j + 1) * Ht], feats[j])
    # with a unit gain the norm of the projection only rescales rows
    yh = O.project_target_hidden(feats, fc, np.ones(H), 0.0)
    assert np.allclose(yh / yh[:, :1], y / y[:, :1])


def _check_projection_closed_form(project):
    """fc + hidden_norm ("Inside SGLang", Step 1: project_target_hidden() is fc
    then hidden_norm; CSDN article, "draft model predict": hidden_norm(fc(x))).
    Inputs are built so that fc(X) has rows c_r * s with s a +-1 pattern: an
    RMSNorm applied after fc sees a row of RMS |c_r|, so the output row is
    exactly sign(c_r) * s * g (times |c_r| / sqrt(c_r^2 + eps)).  fc is dense
    and the gain is not uniform."""
    rng = np.random.default_rng(7)
    rows, Ht, n_sel, H = 4, 24, 3, 16
    fc = rng.normal(0, 0.3, (H, n_sel * Ht))
    s = rng.choice([-1.0, 1.0], H)
    c = np.array([0.7, -2.5, 11.0, 0.05])
    Y = c[:, None] * s[None, :]
    # X with X fc^T = Y: fc^T has full column rank, so pinv(fc^T) fc^T = I
    X = Y @ np.linalg.pinv(fc.T)
    assert np.allclose(X @ fc.T, Y, atol=1e-12)
    feats = [X[:, j * Ht:(j + 1) * Ht] for j in range(n_sel)]
    g = rng.uniform(0.5, 1.5, H)
    for eps in (0.0, 1e-6, 0.3):
        y = project(feats, fc, g, eps)
        want = (c / np.sqrt(c * c + eps))[:, None] * s[None, :] * g[None, :]
        assert np.allclose(y, want, rtol=1e-9, atol=1e-12), eps


def test_project_target_hidden_is_fc_then_gained_rmsnorm():
    _check_projection_closed_form(O.project_target_hidden)


def test_projection_pin_catches_planted_mistakes():
    def norm_before_fc(feats, fc, g, eps):
        x = np.concatenate(feats, -1)
        return O.linear(O.rms_norm(x, np.ones(x.shape[1]), eps), fc) * g

    def gain_dropped(feats, fc, g, eps):
        return O.rms_norm(O.linear(np.concatenate(feats, -1), fc), np.ones_like(g), eps)

    def reversed_concat(feats, fc, g, eps):
        return O.rms_norm(O.linear(np.concatenate(feats[::-1], -1), fc), g, eps)

    for wrong in (norm_before_fc, gain_dropped, reversed_concat):
        with pytest.raises(AssertionError):
            _check_projection_closed_form(wrong)


# ----------------------------------------------------------------- RMSNorm
def test_rms_norm_hand_vector_and_invariants():
    y = O.rms_norm(np.array([[3.0, 4.0]]), np.ones(2), 0.0)
    assert np.allclose(y, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]])
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, 64))
    eps = 1e-6
    y = O.rms_norm(x, np.ones(64), eps)
    ms = np.mean(x * x, axis=1)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + eps)))
    assert np.allclose(O.rms_norm(7.0 * x, np.ones(64), 0.0), O.rms_norm(x, np.ones(64), 0.0))
    g = rng.uniform(0.5, 1.5, 64)
    assert np.allclose(O.rms_norm(x, g, eps), O.rms_norm(x, np.ones(64), eps) * g)


def test_head_rms_norm_is_per_head():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(3, 4, 8))
    x[:, 2] *= 100.0                     # one loud head must not affect the others
    y = O.head_rms_norm(x, np.ones(8), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0)


# --------------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(2).normal(size=(3, 2, 16))
    assert np.allclose(O.rope_neox(x, [0, 0, 0], 1e6), x)


def test_rope_planes_are_i_and_i_plus_half():
    D, theta = 16, 10000.0
    for i in (0, 1, 5):
        e = np.zeros((1, 1, D))
        e[0, 0, i] = 1.0
        p = 7
        y = O.rope_neox(e, [p], theta)[0, 0]
        ang = p * theta ** (-2.0 * i / D)            # frequency of plane i
        expect = np.zeros(D)
        expect[i], expect[i + D // 2] = math.cos(ang), math.sin(ang)
        assert np.allclose(y, expect)


def test_rope_norm_relative_and_composition():
    rng = np.random.default_rng(3)
    D, theta = 32, 1e6
    q = rng.normal(size=(1, 1, D))
    k = rng.normal(size=(1, 1, D))
    qr = O.rope_neox(q, [11], theta)
    assert np.allclose(np.linalg.norm(qr), np.linalg.norm(q))
    dots = [float(np.sum(O.rope_neox(q, [m], theta) * O.rope_neox(k, [m - 4], theta)))
            for m in (4, 9, 1000, 32000)]
    assert np.allclose(dots, dots[0], atol=1e-9)
    two = O.rope_neox(O.rope_neox(q, [5], theta), [9], theta)
    assert np.allclose(two, O.rope_neox(q, [14], theta))


# ---------------------------------------------------------------- projections
def test_linear_matches_triple_loop():
    rng = np.random.default_rng(4)
    x, w = rng.normal(size=(3, 5)), rng.normal(size=(4, 5))
    y = O.linear(x, w)
    for i in range(3):
        for o in range(4):
            assert math.isclose(y[i, o], sum(x[i, k] * w[o, k] for k in range(5)), rel_tol=1e-12)


def test_split_qkv_row_order():
    cfg = tiny_cfg()
    D = cfg.head_dim
    w = np.arange((cfg.n_heads + 2 * cfg.n_kv_heads) * D)[:, None] * np.ones((1, 3))
    q, k, v = O.split_qkv(w, cfg)
    assert q[0, 0] == 0 and k[0, 0] == cfg.n_heads * D
    assert v[0, 0] == (cfg.n_heads + cfg.n_kv_heads) * D and v.shape[0] == cfg.n_kv_heads * D


def test_silu_closed_form():
    assert O.silu(np.array(0.0)) == 0.0
    assert math.isclose(float(O.silu(np.array(1.0))), 1 / (1 + math.exp(-1)))
    assert math.isclose(float(O.silu(np.array(40.0))), 40.0, rel_tol=1e-12)


# ---------------------------------------------------------------- attention
def _attn_loops(q, kc, vc, kb, vb, q_pos, ctx_pos, window):
    S, nh, D = q.shape
    grp = nh // kb.shape[1]
    out = np.zeros_like(q)
    for j in range(S):
        for h in range(nh):
            g = h // grp
            keys, vals = [], []
            for t in range(kc.shape[0]):
                if window == 0 or q_pos[j] - ctx_pos[t] < window:
                    keys.append(kc[t, g]); vals.append(vc[t, g])
            for t in range(S):
                keys.append(kb[t, g]); vals.append(vb[t, g])
            sc = [float(np.dot(q[j, h], kk)) / math.sqrt(D) for kk in keys]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            out[j, h] = sum(ei * vv for ei, vv in zip(e, vals)) / sum(e)
    return out


@pytest.mark.parametrize("window", [0, 1, 3, 6])
def test_attention_bruteforce(window):
    rng = np.random.default_rng(5 + window)
    S, nh, kvh, D, T = 4, 4, 2, 8, 7
    q = rng.normal(size=(S, nh, D))
    kc, vc = rng.normal(size=(T, kvh, D)), rng.normal(size=(T, kvh, D))
    kb, vb = rng.normal(size=(S, kvh, D)), rng.normal(size=(S, kvh, D))
    q_pos, ctx_pos = T + np.arange(S), np.arange(T)
    got = O.block_attention(q, kc, vc, kb, vb, q_pos, ctx_pos, window)
    assert np.allclose(got, _attn_loops(q, kc, vc, kb, vb, q_pos, ctx_pos, window), atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    S, nh, kvh, D, T = 3, 2, 1, 4, 5
    q = rng.normal(size=(S, nh, D))
    # identical keys: uniform weights, so the output is the mean of the values
    k = np.tile(rng.normal(size=(1, kvh, D)), (T, 1, 1))
    kb = np.tile(k[:1], (S, 1, 1))
    vc, vb = rng.normal(size=(T, kvh, D)), rng.normal(size=(S, kvh, D))
    out = O.block_attention(q, k, vc, kb, vb, T + np.arange(S), np.arange(T), 0)
    mean_v = np.concatenate([vc, vb])[:, 0].mean(axis=0)
    assert np.allclose(out, mean_v[None, None, :])
    # one block row, window 1: no context key is visible, the output is that row's value
    out = O.block_attention(q[:1], rng.normal(size=(T, kvh, D)), vc, kb[:1], vb[:1],
                            [T], np.arange(T), 1)
    assert np.allclose(out[0], vb[0, 0])


def test_attention_window_edges():
    # a context key at distance W-1 is visible, at distance W it is not
    D = 4
    W = 3
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 50.0          # strongly prefers key direction e0
    kc = np.zeros((4, 1, D)); vc = np.zeros((4, 1, D))
    q_pos = [10]
    ctx_pos = np.array([7, 8, 2, 3])                    # distances 3, 2, 8, 7
    kc[1, 0, 0] = 1.0; vc[1, 0, 1] = 1.0                # distance 2 = W-1: visible, wins
    kc[0, 0, 0] = 2.0; vc[0, 0, 2] = 1.0                # distance 3 = W: hidden although larger
    kb = np.zeros((1, 1, D)); vb = np.zeros((1, 1, D))
    out = O.block_attention(q, kc, vc, kb, vb, q_pos, ctx_pos, W)
    assert out[0, 0, 1] > 0.99 and out[0, 0, 2] == 0.0


def test_attention_is_non_causal_and_gqa_grouped():
    rng = np.random.default_rng(7)
    S, nh, kvh, D, T = 4, 4, 2, 8, 3
    q = rng.normal(size=(S, nh, D))
    kc, vc = rng.normal(size=(T, kvh, D)), rng.normal(size=(T, kvh, D))
    kb, vb = rng.normal(size=(S, kvh, D)), rng.normal(size=(S, kvh, D))
    args = (T + np.arange(S), np.arange(T), 0)
    base = O.block_attention(q, kc, vc, kb, vb, *args)
    vb2 = vb.copy(); vb2[S - 1] += 1.0                  # last block row changes row 0
    assert not np.allclose(O.block_attention(q, kc, vc, kb, vb2, *args)[0], base[0])
    vc2 = vc.copy(); vc2[:, 1] += 1.0                   # KV head 1 feeds query heads 2,3 only
    alt = O.block_attention(q, kc, vc2, kb, vb, *args)
    assert np.allclose(alt[:, :2], base[:, :2]) and not np.allclose(alt[:, 2:], base[:, 2:])


# ----------------------------------------------------------------- lm head
def test_lm_head_argmax_planted_and_ties():
    H, V = 6, 9
    w = np.zeros((V, H))
    for v in range(V):
        w[v, v % H] = 1.0                               # logit v = x[v % H]
    x = np.array([[0, 0, 5.0, 0, 0, 0], [0, 1.0, 0, 0, 0, 0.5]])
    ids, margin = O.lm_head_argmax(x, w)
    assert list(ids) == [2, 1]                          # 2 ties with 8 and 1 with 7: lowest index
    assert margin[0] == 0.0 and margin[1] == 0.0
    x = np.array([[0, 0, 0, 3.0, 1.0, 0]])
    ids, margin = O.lm_head_argmax(x, w[:6])
    assert ids[0] == 3 and margin[0] == 2.0


# ------------------------------------------------------ injection and context
def test_inject_positions_continue_across_calls():
    cfg = tiny_cfg()
    rng = np.random.default_rng(8)
    W = tiny_weights(cfg, rng)
    feats = [rng.normal(size=(6, cfg.target_hidden)) for _ in range(cfg.n_sel)]
    a = O.DraftContext(cfg)
    a.inject(feats, W)
    b = O.DraftContext(cfg)
    b.inject([f[:2] for f in feats], W)
    b.inject([f[2:] for f in feats], W)
    assert a.kv_len == b.kv_len == 6
    for l in range(cfg.n_layers):
        assert np.allclose(a.k[l], b.k[l]) and np.allclose(a.v[l], b.v[l])
    # un-rotating row i by its position gives back a unit-RMS head
    k0 = O.rope_neox(a.k[0], -np.arange(6), cfg.rope_theta)
    gk = W["layers"][0]["k_norm"]
    assert np.allclose(np.sqrt(np.mean((k0 / gk) ** 2, axis=-1)), 1.0, atol=1e-5)


def test_context_rows_are_rotated_by_their_positions():
    cfg = tiny_cfg()
    rng = np.random.default_rng(9)
    W = tiny_weights(cfg, rng)
    y = rng.normal(size=(3, cfg.hidden))
    k0, v0 = O.context_kv(y, W["layers"][0], np.array([0, 0, 0]), cfg)
    k5, v5 = O.context_kv(y, W["layers"][0], np.array([5, 6, 7]), cfg)
    assert np.allclose(v0, v5)
    assert np.allclose(O.rope_neox(k0, [5, 6, 7], cfg.rope_theta), k5)


# --------------------------------------------------- composition (loop level)
def _to_lists(W):
    out = {k: np.asarray(v).tolist() for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: np.asarray(v).tolist() for k, v in L.items()} for L in W["layers"]]
    return out


@pytest.mark.parametrize("window", [(0, 0), (3, 0)])
def test_draft_forward_matches_loop_restatement(window):
    cfg = tiny_cfg(sliding_window=window)
    rng = np.random.default_rng(10)
    W = tiny_weights(cfg, rng)
    ctx = O.DraftContext(cfg)
    feats = [rng.normal(size=(6, cfg.target_hidden)) for _ in range(cfg.n_sel)]
    ctx.inject(feats, W)
    got = O.draft_forward(cfg, W, 5, ctx.layers(), ctx.kv_len)
    ref = draft_forward_loops(cfg, _to_lists(W), 5, [k.tolist() for k in ctx.k],
                              [v.tolist() for v in ctx.v], ctx.kv_len)
    assert np.allclose(got, np.array(ref), rtol=1e-10, atol=1e-10)


def test_draft_block_ids_layout():
    cfg = tiny_cfg()
    rng = np.random.default_rng(11)
    W = tiny_weights(cfg, rng)
    ctx = O.DraftContext(cfg)
    ctx.inject([rng.normal(size=(4, cfg.target_hidden)) for _ in range(cfg.n_sel)], W)
    ids, hid, margin = O.draft_block(cfg, W, 17, ctx.layers(), ctx.kv_len)
    assert ids[0] == 17 and len(ids) == cfg.block_size and len(margin) == cfg.block_size - 1
    logits = hid[1:] @ W["lm_head"].T
    assert list(ids[1:]) == [int(np.argmax(r)) for r in logits]


def test_draft_block_does_not_depend_on_cache_rows_past_kv_len():
    cfg = tiny_cfg()
    rng = np.random.default_rng(12)
    W = tiny_weights(cfg, rng)
    ctx = O.DraftContext(cfg)
    ctx.inject([rng.normal(size=(5, cfg.target_hidden)) for _ in range(cfg.n_sel)], W)
    a = O.draft_forward(cfg, W, 3, ctx.layers(), 3)
    junk = [(np.concatenate([k[:3], 9 + k[3:]]), v) for k, v in ctx.layers()]
    assert np.allclose(a, O.draft_forward(cfg, W, 3, junk, 3))


# ------------------------------------- planted mistakes must trip these pins
def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (CPU only) and check a pin fails."""
    # 1. interleaved (GPT-J) RoPE pairs instead of rotate-half
    def rope_interleaved(x, positions, theta):
        x = np.asarray(x, float)
        d = x.shape[-1]
        ang = np.asarray(positions, float)[:, None] * O.rope_frequencies(d, theta)[None]
        c, s = np.cos(ang)[:, None], np.sin(ang)[:, None]
        ev, od = x[..., 0::2], x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2], out[..., 1::2] = ev * c - od * s, od * c + ev * s
        return out
    monkeypatch.setattr(O, "rope_neox", rope_interleaved)
    with pytest.raises(AssertionError):
        test_rope_planes_are_i_and_i_plus_half()
    monkeypatch.undo()
    # 2. causal mask inside the block
    orig = O.block_attention

    def causal(q, kc, vc, kb, vb, q_pos, ctx_pos, window):
        out = np.empty_like(np.asarray(q, float))
        for j in range(q.shape[0]):
            out[j:j + 1] = orig(q[j:j + 1], kc, vc, kb[:j + 1], vb[:j + 1], q_pos[j:j + 1],
                                ctx_pos, window)
        return out
    monkeypatch.setattr(O, "block_attention", causal)
    with pytest.raises(AssertionError):
        test_attention_is_non_causal_and_gqa_grouped()
    monkeypatch.undo()
    # 3. off-by-one acceptance (count the first mismatch as accepted)
    orig_acc = O.accept_block

    def acc_plus_one(d, p):
        a, b, c, o = orig_acc(d, p)
        a = min(a + 1, len(d) - 1)
        return a, int(np.asarray(p)[a]), a + 1, o
    monkeypatch.setattr(O, "accept_block", acc_plus_one)
    with pytest.raises(AssertionError):
        test_accept_worked_example_p1()
    monkeypatch.undo()
    # 4. hidden-state offset forgotten
    monkeypatch.setattr(O, "extract_context_feature",
                        lambda hs, ids: np.concatenate([hs[j] for j in ids], -1))
    with pytest.raises(AssertionError):
        test_extract_context_feature_offset_and_order()
    monkeypatch.undo()
    # 5. RMSNorm gain dropped
    monkeypatch.setattr(O, "rms_norm", lambda x, g, eps: np.asarray(x, float) / np.sqrt(
        np.mean(np.asarray(x, float) ** 2, -1, keepdims=True) + eps))
    with pytest.raises(AssertionError):
        test_rms_norm_hand_vector_and_invariants()
    monkeypatch.undo()


# ------------------------------------------------ sampled (lossless) verification
# [P1] "Sampling: preserve the proposal distribution the walk actually used":
# accept y with probability min(1, p(y)/q(y)); at the first rejection draw from
# the normalised residual [p - q]+; after full acceptance the target supplies a
# bonus token.  The plain drafter proposes argmax tokens (q = point mass).
def _chi2_pvalue(counts, probs):
    from scipy.stats import chisquare
    probs = np.asarray(probs, float)
    keep = probs > 0
    exp = probs[keep] / probs[keep].sum() * counts.sum()
    assert counts[~keep].sum() == 0
    return chisquare(counts[keep], exp).pvalue


def test_sampled_reduces_to_greedy_for_a_deterministic_target():
    """A one-hot target at the posterior tokens turns the sampled rule into the
    greedy cumprod rule, for every uniform and every noise: the worked
    examples of the pages carry over."""
    rng = np.random.default_rng(5)
    V, S = 11, 6
    for _ in range(200):
        draft = rng.integers(0, V, S)
        post = np.where(rng.random(S) < 0.6, np.r_[draft[1:], 0], rng.integers(0, V, S))
        probs = np.zeros((S, V), np.float32)
        probs[np.arange(S), post] = 1.0
        u = rng.random(S - 1).astype(np.float32)
        e = rng.exponential(size=V).astype(np.float32)
        assert O.accept_block_sampled(draft, probs, u, e)[:3] == O.accept_block(draft, post)[:3]
    gd = _golden("accept_worked_example_p1.json")
    voc, ex = gd["vocab"], gd["expected"]
    d = [voc[t] for t in gd["block"]]
    p = [voc[t] for t in gd["target_choices"]]
    V = max(voc.values()) + 1
    probs = np.zeros((len(d), V), np.float32)
    probs[np.arange(len(d)), p] = 1.0
    acc, bonus, commit, out = O.accept_block_sampled(d, probs, np.full(len(d) - 1, 0.99, np.float32),
                                                     np.ones(V, np.float32))
    assert (acc, bonus, commit) == (ex["accept_len"], voc[ex["bonus"]], ex["commit_len"])
    assert list(out[:commit]) == [voc[t] for t in ex["out_tokens_valid"]]


def test_sampled_zero_probability_rejects_and_is_excluded():
    rng = np.random.default_rng(6)
    V = 7
    probs = np.full((3, V), 1.0 / (V - 1), np.float32)
    probs[0, 4] = 0.0                       # the first proposed token is impossible
    for _ in range(300):
        acc, bonus, _, out = O.accept_block_sampled([1, 4, 2], probs, rng.random(2).astype(np.float32),
                                                    rng.exponential(size=V).astype(np.float32))
        assert acc == 0 and bonus != 4 and out[0] == bonus


def test_exponential_race_samples_the_weights():
    rng = np.random.default_rng(7)
    w = np.array([0.05, 0.0, 0.4, 0.15, 0.3, 0.1], np.float32)
    n = 30000
    counts = np.zeros(len(w), np.int64)
    for _ in range(n):
        counts[O.exponential_race(w, rng.exponential(size=len(w)).astype(np.float32))] += 1
    assert _chi2_pvalue(counts, w) > 1e-3
    # unnormalised weights give the same distribution
    counts2 = np.zeros(len(w), np.int64)
    for _ in range(n):
        counts2[O.exponential_race(7.0 * w, rng.exponential(size=len(w)).astype(np.float32))] += 1
    assert _chi2_pvalue(counts2, w) > 1e-3


@pytest.mark.parametrize("p_y", [0.0, 0.3, 0.9])
def test_sampled_verification_is_lossless(p_y):
    """The first emitted token (accepted draft or correction) follows the
    target distribution p exactly, whatever the drafter proposed."""
    rng = np.random.default_rng(int(p_y * 100) + 8)
    V = 5
    p0 = np.array([0.2, 0.15, 0.0, 0.25, 0.4], np.float64)
    y = 2
    p0 = p0 * (1 - p_y) / p0.sum()
    p0[y] = p_y
    probs = np.tile(p0.astype(np.float32), (3, 1))
    n = 30000
    counts = np.zeros(V, np.int64)
    for _ in range(n):
        _, _, _, out = O.accept_block_sampled([0, y, 1], probs, rng.random(2).astype(np.float32),
                                              rng.exponential(size=V).astype(np.float32))
        counts[out[0]] += 1
    assert _chi2_pvalue(counts, probs[0]) > 1e-3


def test_sampled_pins_catch_planted_mistakes(monkeypatch):
    """Plausible mistakes in the sampled rule must trip a pin (CPU only)."""
    orig = O.accept_block_sampled

    # 1. the rejected token is not removed from the correction distribution
    def no_residual(draft, probs, u, e):
        draft = np.asarray(draft); probs = np.asarray(probs, np.float32); u = np.asarray(u, np.float32)
        acc = 0
        while acc < len(draft) - 1 and u[acc] < probs[acc, draft[acc + 1]]:
            acc += 1
        bonus = O.exponential_race(probs[acc], e)
        out = np.zeros(len(draft), np.int64); out[:acc] = draft[1:acc + 1]; out[acc] = bonus
        return acc, bonus, acc + 1, out
    monkeypatch.setattr(O, "accept_block_sampled", no_residual)
    with pytest.raises(AssertionError):
        test_sampled_verification_is_lossless(0.3)
    monkeypatch.undo()
    # 2. acceptance with the complementary probability (accept iff u >= p)
    def flipped(draft, probs, u, e):
        draft = np.asarray(draft); probs = np.asarray(probs, np.float32); u = np.asarray(u, np.float32)
        acc = 0
        while acc < len(draft) - 1 and u[acc] >= probs[acc, draft[acc + 1]]:
            acc += 1
        w = probs[acc].copy()
        if acc < len(draft) - 1:
            w[draft[acc + 1]] = 0.0
        bonus = O.exponential_race(w, e)
        out = np.zeros(len(draft), np.int64); out[:acc] = draft[1:acc + 1]; out[acc] = bonus
        return acc, bonus, acc + 1, out
    monkeypatch.setattr(O, "accept_block_sampled", flipped)
    with pytest.raises(AssertionError):
        test_sampled_verification_is_lossless(0.9)
    monkeypatch.undo()
    # 3. the race taken as argmin instead of argmax of w / e
    monkeypatch.setattr(O, "exponential_race",
                        lambda w, e: int(np.argmin(np.where(np.asarray(w) > 0, np.asarray(w, np.float32) /
                                                            np.asarray(e, np.float32), np.inf))))
    with pytest.raises(AssertionError):
        test_exponential_race_samples_the_weights()
    monkeypatch.undo()


# ------------------------------------------------ DFlash 2 candidate selector
# [P1] "DFlash 2: replace selection, retain the serving loop": per position the
# K best lm_head logits are candidates; score(p, c; h) = U(c) + <A[p] * W_h h,
# B[c]>; the predecessor is the anchor, then the candidate chosen before; the
# walk is greedy or sampled, never a search for the best full path; q_rows is
# the softmax of the chosen predecessor's row.
def _lm_rows(logit_rows):
    """hidden rows = identity, lm_head = the logits transposed: logits come out as given."""
    L = np.asarray(logit_rows, float)
    return np.eye(L.shape[0]), L.T.copy()


def test_candidates_order_ties_and_k1():
    h, lm = _lm_rows([[1.0, 3.0, 3.0, 2.0, -1.0], [0.5, 0.5, 0.5, 0.5, 0.5]])
    ids, u = O.compute_candidates(h, lm, 3)
    assert ids.tolist() == [[1, 2, 3], [0, 1, 2]]
    assert u.tolist() == [[3.0, 3.0, 2.0], [0.5, 0.5, 0.5]]
    rng = np.random.default_rng(20)
    hid, lmh = rng.normal(size=(6, 8)), rng.normal(size=(40, 8))
    ids1, _ = O.compute_candidates(hid, lmh, 1)
    assert ids1[:, 0].tolist() == O.lm_head_argmax(hid, lmh)[0].tolist()
    idsV, _ = O.compute_candidates(hid, lmh, 40)     # K = V: a permutation of the vocabulary
    assert all(sorted(r) == list(range(40)) for r in idsV.tolist())
    with pytest.raises(ValueError):
        O.compute_candidates(hid, lmh, 41)


def _walk_example():
    """Hand-built lattice, V = 4, r = 1, K = 2 (numbers chosen for the test).
    position 1: candidates [0, 1], U = [0, 0], wh = 1; anchor 2 with A[2] = 1;
                B[0] = 1, B[1] = -1: scores [1, -1] -> token 0.
    position 2: candidates [1, 3], U = [0, 0.5], wh = 2; predecessor 0 with
                A[0] = -1: scores [2, -1.5] -> token 1.
    Using the anchor (A = 1) at position 2 would give [-2, 2.5] -> token 3;
    the best full path is [1, 3] (-1 + 6.5 via A[1] = 3) -- the greedy walk
    does not take it."""
    A = np.array([[-1.0], [3.0], [1.0], [0.0]])
    B = np.array([[1.0], [-1.0], [0.0], [1.0]])
    cand = np.array([[0, 1], [1, 3]])
    unary = np.array([[0.0, 0.0], [0.0, 0.5]])
    wh = np.array([[1.0], [2.0]])
    return A, B, cand, unary, wh


def test_selector_walk_hand_lattice():
    A, B, cand, unary, wh = _walk_example()
    ids, slots, q = O.selector_walk(2, cand, unary, wh, A, B)
    assert ids.tolist() == [0, 1] and slots.tolist() == [0, 0]
    # a two-way softmax is the logistic of the score difference
    assert q[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-2.0)), rel=1e-12)
    assert q[1, 0] == pytest.approx(1.0 / (1.0 + math.exp(-3.5)), rel=1e-12)
    assert np.allclose(q.sum(axis=1), 1.0)


def test_selector_without_compatibility_is_plain_dflash():
    """A = 0 (or W_h = 0) leaves only the unary logits: the greedy walk picks
    every position's top candidate, i.e. the plain argmax draft."""
    cfg = tiny_cfg()
    rng = np.random.default_rng(21)
    W = tiny_weights(cfg, rng)
    ctx = O.DraftContext(cfg)
    ctx.inject([rng.normal(size=(5, cfg.target_hidden)) for _ in range(cfg.n_sel)], W)
    r = 3
    for sel in ({"A": np.zeros((cfg.vocab, r)), "B": rng.normal(size=(cfg.vocab, r)),
                 "W_h": rng.normal(size=(r, cfg.hidden))},
                {"A": rng.normal(size=(cfg.vocab, r)), "B": rng.normal(size=(cfg.vocab, r)),
                 "W_h": np.zeros((r, cfg.hidden))}):
        ids, cand, unary, q, wh, _ = O.draft_block_selector(cfg, W, sel, 7, ctx.layers(), ctx.kv_len, 4)
        plain, _, _ = O.draft_block(cfg, W, 7, ctx.layers(), ctx.kv_len)
        assert ids.tolist() == plain.tolist()
        assert np.allclose(q, np.exp(unary - unary.max(1, keepdims=True)) /
                           np.exp(unary - unary.max(1, keepdims=True)).sum(1, keepdims=True))


def test_selector_sampled_walk_follows_q_rows():
    """Sampling at one position draws the candidates with the softmax of the
    chosen predecessor's scores; a shift of all unary logits changes nothing."""
    A, B, cand, unary, wh = _walk_example()
    rng = np.random.default_rng(22)
    n = 20000
    counts = np.zeros(2, np.int64)
    for _ in range(n):
        _, slots, q = O.selector_walk(2, cand[:1], unary[:1] + 5.0, wh[:1], A, B,
                                      rng.exponential(size=(1, 2)).astype(np.float32))
        counts[slots[0]] += 1
    assert _chi2_pvalue(counts, [1.0 / (1.0 + math.exp(-2.0)), 1.0 / (1.0 + math.exp(2.0))]) > 1e-3


def test_selector_sampled_walk_conditions_on_the_drawn_predecessor():
    """Two sampled positions: P(y1, y2) = q1(y1) q2(y2 | y1), position 2's
    softmax taken for the token actually drawn at position 1 (predecessor 0:
    A = -1, predecessor 1: A = 3 in the hand lattice)."""
    A, B, cand, unary, wh = _walk_example()
    # position-2 scores for predecessor p: U + A[p] * 2 * B[c], c in [1, 3]
    def q2(pred):
        s = np.array([0.0 + A[pred, 0] * 2.0 * B[1, 0], 0.5 + A[pred, 0] * 2.0 * B[3, 0]])
        e = np.exp(s - s.max())
        return e / e.sum()
    q1 = np.array([1.0 / (1.0 + math.exp(-2.0)), 1.0 / (1.0 + math.exp(2.0))])
    expect = np.array([q1[0] * q2(0)[0], q1[0] * q2(0)[1], q1[1] * q2(1)[0], q1[1] * q2(1)[1]])
    rng = np.random.default_rng(25)
    counts = np.zeros(4, np.int64)
    for _ in range(20000):
        _, slots, _ = O.selector_walk(2, cand, unary, wh, A, B,
                                      rng.exponential(size=(2, 2)).astype(np.float32))
        counts[2 * slots[0] + slots[1]] += 1
    assert _chi2_pvalue(counts, expect) > 1e-3


def test_selector_walk_with_sampled_verification_is_lossless():
    """The sampled walk's q_rows, fed to the real-q verification: given the
    first draft accepted, the second emitted token follows the target row of
    position 1 -- which holds only if q_rows[1] is the distribution the walk
    drew position 2 from, i.e. conditioned on the predecessor it chose."""
    A, B, cand, unary, wh = _walk_example()
    V = 4
    p = np.array([[0.1, 0.6, 0.2, 0.1], [0.3, 0.2, 0.15, 0.35], [0.25, 0.25, 0.25, 0.25]],
                 np.float32)
    rng = np.random.default_rng(26)
    counts = np.zeros(V, np.int64)
    for _ in range(40000):
        ids, _, q = O.selector_walk(2, cand, unary, wh, A, B,
                                    rng.exponential(size=(2, 2)).astype(np.float32))
        draft = np.array([2, ids[0], ids[1]])
        acc, _, _, out = O.accept_block_sampled_q(draft, p, cand, q.astype(np.float32),
                                                  rng.random(2).astype(np.float32),
                                                  rng.exponential(size=V).astype(np.float32))
        if acc >= 1:
            counts[out[1]] += 1
    assert _chi2_pvalue(counts, p[1]) > 1e-3


def test_sampled_q_point_mass_is_the_plain_rule():
    """q = 1 on the proposed token (K = 1 candidate list of the draft) is the
    argmax drafter's rule."""
    rng = np.random.default_rng(23)
    V, S = 9, 5
    for _ in range(300):
        draft = rng.integers(0, V, S)
        probs = rng.dirichlet(np.ones(V), S).astype(np.float32)
        u = rng.random(S - 1).astype(np.float32)
        e = rng.exponential(size=V).astype(np.float32)
        a = O.accept_block_sampled_q(draft, probs, draft[1:, None], np.ones((S - 1, 1)), u, e)
        b = O.accept_block_sampled(draft, probs, u, e)
        assert a[:3] == b[:3] and a[3].tolist() == b[3].tolist()


def test_sampled_q_accepts_whenever_q_is_at_most_p():
    probs = np.full((3, 4), 0.25, np.float32)
    cand = np.array([[1, 2], [3, 0]])
    q = np.array([[0.2, 0.8], [0.25, 0.75]], np.float32)      # q(1) = 0.2 <= p, q(3) = 0.25 <= p
    for u in (0.0, 0.5, 0.999):
        acc, _, _, out = O.accept_block_sampled_q([0, 1, 3], probs, cand, q, np.full(2, u, np.float32),
                                                  np.ones(4, np.float32))
        assert acc == 2 and out[:2].tolist() == [1, 3]
    # a token outside the candidate list (q = 0) is rejected
    acc, bonus, _, _ = O.accept_block_sampled_q([0, 2, 3], probs, np.array([[1, 3], [3, 0]]), q,
                                                np.zeros(2, np.float32), np.ones(4, np.float32))
    assert acc == 0


def test_sampled_q_is_lossless():
    """y drawn from q over K candidates, accepted with min(1, p/q), else the
    correction from [p - q]+: the emitted token follows p exactly."""
    rng = np.random.default_rng(24)
    V = 6
    p0 = np.array([0.3, 0.05, 0.25, 0.0, 0.15, 0.25])
    cand = np.array([2, 4, 3, 1])
    q0 = np.array([0.1, 0.5, 0.3, 0.1])          # over-proposes 4 and the impossible 3
    probs = np.tile(p0.astype(np.float32), (2, 1))
    n = 30000
    counts = np.zeros(V, np.int64)
    for _ in range(n):
        k = O.exponential_race(q0, rng.exponential(size=4).astype(np.float32))
        _, _, _, out = O.accept_block_sampled_q([0, cand[k]], probs, cand[None, :], q0[None, :],
                                                rng.random(1).astype(np.float32),
                                                rng.exponential(size=V).astype(np.float32))
        counts[out[0]] += 1
    assert _chi2_pvalue(counts, p0) > 1e-3


def test_selector_pins_catch_planted_mistakes(monkeypatch):
    """Plausible mistakes in the selector must trip a pin (CPU only)."""
    # 1. the predecessor stays the anchor for every position
    orig_scores = O.selector_scores

    def anchor_always(unary_row, cand_row, pred, wh_row, A, B):
        return orig_scores(unary_row, cand_row, 2, wh_row, A, B)
    monkeypatch.setattr(O, "selector_scores", anchor_always)
    with pytest.raises(AssertionError):
        test_selector_walk_hand_lattice()
    with pytest.raises(AssertionError):
        test_selector_sampled_walk_conditions_on_the_drawn_predecessor()
    monkeypatch.undo()
    # q_rows reported for the anchor's row while the draw used the true predecessor
    orig_walk = O.selector_walk

    def wrong_rows(anchor, cand, unary, wh, A, B, exp_noise=None):
        ids, slots, q = orig_walk(anchor, cand, unary, wh, A, B, exp_noise)
        for j in range(1, len(ids)):
            q[j] = O.softmax(orig_scores(unary[j], cand[j], anchor, wh[j], A, B))
        return ids, slots, q
    monkeypatch.setattr(O, "selector_walk", wrong_rows)
    with pytest.raises(AssertionError):
        test_selector_walk_with_sampled_verification_is_lossless()
    monkeypatch.undo()
    # 2. the compatibility term with A and B swapped (successor factor on the predecessor)
    monkeypatch.setattr(O, "selector_scores", lambda u, c, p, w, A, B: orig_scores(u, c, p, w, B, A))
    with pytest.raises(AssertionError):
        test_selector_walk_hand_lattice()
    monkeypatch.undo()
    # 3. candidates in ascending logit order
    orig_cand = O.compute_candidates
    monkeypatch.setattr(O, "compute_candidates",
                        lambda h, lm, K: tuple(x[:, ::-1] for x in orig_cand(h, lm, K)))
    with pytest.raises(AssertionError):
        test_candidates_order_ties_and_k1()
    monkeypatch.undo()
    # 4. residual without subtracting q (the plain rule's [p - 1{y}]+ applied to a real q)
    orig_acc = O.accept_block_sampled_q

    def residual_point_mass(draft, probs, cand, q_rows, u, e):
        draft = np.asarray(draft); probs = np.asarray(probs, np.float32)
        acc, bonus, commit, out = orig_acc(draft, probs, cand, q_rows, u, e)
        if acc < len(draft) - 1:
            w = probs[acc].copy(); w[draft[acc + 1]] = 0.0
            bonus = O.exponential_race(w, e); out[acc] = bonus
        return acc, bonus, commit, out
    monkeypatch.setattr(O, "accept_block_sampled_q", residual_point_mass)
    with pytest.raises(AssertionError):
        test_sampled_q_is_lossless()
    monkeypatch.undo()


# ------------------------------------------------------------ FP8 draft KV cache
# [P3] Kimi-K2.6 draft card: "12 KiB / token (FP8)".  Reading: OCP FP8 E4M3
# (bias 7, 3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN, max
# 448), nearest code with ties to the even mantissa, saturation, one scale per
# layer and tensor.
def test_fp8_footprint_is_one_byte_per_element():
    """The card's shape (6 layers, 8 KV heads, head_dim 128) and its 12 KiB per
    token leave exactly one byte per K or V element: no per-token scales."""
    layers, kv_heads, head_dim = 6, 8, 128
    assert layers * 2 * kv_heads * head_dim * 1 == 12 * 1024


def test_e4m3_decode_format_values():
    v = O.e4m3_decode(np.arange(256))
    # values fixed by the format: zero, smallest subnormal, largest subnormal,
    # smallest normal, one, largest finite, NaN, negative zero, negative max
    assert v[0x00] == 0.0 and v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9
    assert v[0x08] == 2.0 ** -6 and v[0x38] == 1.0 and v[0x7E] == 448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x80] == 0.0 and np.signbit(v[0x80]) and v[0xFE] == -448.0
    # exponent field e >= 1: (1 + m/8) 2^(e-7); each binade holds 8 codes
    assert v[0x40] == 2.0 and v[0x48] == 4.0 and v[0x30] == 0.5 and v[0x3C] == 1.5
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # codes order like their values
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign bit mirrors


def test_e4m3_encode_round_trip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)
    pos = O.e4m3_decode(np.arange(0x7F))
    mid = (pos[:-1] + pos[1:]) / 2
    got = O.e4m3_encode(mid)
    even = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F))
    assert np.array_equal(got, even)                      # ties go to the even mantissa
    assert O.e4m3_encode(mid[10] * (1 + 1e-9)) == 11      # just above a midpoint: up
    assert O.e4m3_encode(mid[10] * (1 - 1e-9)) == 10      # just below: down
    assert list(O.e4m3_encode([1e6, -1e6, 464.0, 470.0])) == [0x7E, 0xFE, 0x7E, 0x7E]
    assert O.e4m3_encode(np.nan) == 0x7F
    rng = np.random.default_rng(30)
    x = rng.uniform(2.0 ** -6, 448.0, 20000) * rng.choice([-1, 1], 20000)
    err = np.abs(O.e4m3_decode(O.e4m3_encode(x)) - x) / np.abs(x)
    assert err.max() <= 2.0 ** -4 + 1e-12                 # half a unit in the last place


def test_fp8_cache_is_exact_for_representable_values_and_feeds_attention():
    """Values that are codes times the scale survive the cache unchanged, so
    attention over the FP8 cache equals attention over the originals; other
    values move by at most half a code step."""
    rng = np.random.default_rng(31)
    codes = rng.integers(0, 0x7F, (20, 2, 8)) | (rng.integers(0, 2, (20, 2, 8)) << 7)
    codes = np.where(codes == 0xFF, 0xFE, codes)
    k = O.e4m3_decode(codes) * 0.25
    v = O.e4m3_decode(np.flip(codes, 0)) * 2.0
    kq, vq = O.fp8_kv(k, v, 0.25, 2.0)
    assert np.array_equal(kq, k) and np.array_equal(vq, v)
    q = rng.normal(size=(3, 4, 8))
    a = O.block_attention(q, k, v, k[:3], v[:3], np.arange(20, 23), np.arange(20), 0)
    b = O.block_attention(q, kq, vq, k[:3], v[:3], np.arange(20, 23), np.arange(20), 0)
    assert np.array_equal(a, b)
    x = rng.normal(size=(50, 2, 8))
    xq, _ = O.fp8_kv(x, x, 0.01, 0.01)
    assert np.all(np.abs(xq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 0.01 * 2.0 ** -10) + 1e-15)


def test_fp8_pins_catch_planted_mistakes(monkeypatch):
    orig = O.e4m3_decode
    # exponent bias 8 instead of 7
    monkeypatch.setattr(O, "e4m3_decode", lambda c: orig(c) / 2.0)
    with pytest.raises(AssertionError):
        test_e4m3_decode_format_values()
    monkeypatch.undo()
    # ties away from zero instead of to even
    enc = O.e4m3_encode

    def away(x):
        x = np.asarray(x, float)
        c = enc(x)
        up = enc(x * (1 + 1e-12))
        return np.where(c != up, up, c)
    monkeypatch.setattr(O, "e4m3_encode", away)
    with pytest.raises(AssertionError):
        test_e4m3_encode_round_trip_ties_and_saturation()
    monkeypatch.undo()


def _check_layers_fp8(layers_fp8):
    """DraftContext.layers_fp8 with per-layer (K, V) scales: K/V values that
    are E4M3 codes times their own layer's scale come back unchanged, and
    values past 448 * scale saturate there.  The scales (0.3, 1.7, 0.11,
    5.0) are unrelated by powers of two, so a value stored with another
    layer's or the other tensor's scale is in general not representable and
    changes."""
    cfg = tiny_cfg(n_layers=2)
    rng = np.random.default_rng(33)
    ks, vs = [0.3, 0.11], [1.7, 5.0]
    ctx = O.DraftContext(cfg)
    shape = (30, cfg.n_kv_heads, cfg.head_dim)
    for l in range(2):
        codes_k = rng.integers(0x08, 0x7F, shape) | (rng.integers(0, 2, shape) << 7)
        codes_v = rng.integers(0x08, 0x7F, shape) | (rng.integers(0, 2, shape) << 7)
        ctx.k[l] = O.e4m3_decode(codes_k) * ks[l]
        ctx.v[l] = O.e4m3_decode(codes_v) * vs[l]
    ctx.k[1][0, 0, 0] = 1000.0 * ks[1]          # saturates at 448 * scale
    ctx.v[0][1, 1, 1] = -900.0 * vs[0]
    out = layers_fp8(ctx, ks, vs)
    assert len(out) == 2
    assert out[1][0][0, 0, 0] == 448.0 * ks[1] and out[0][1][1, 1, 1] == -448.0 * vs[0]
    ctx.k[1][0, 0, 0] = 448.0 * ks[1]
    ctx.v[0][1, 1, 1] = -448.0 * vs[0]
    for l in range(2):
        assert np.array_equal(out[l][0], ctx.k[l]) and np.array_equal(out[l][1], ctx.v[l]), l


def test_layers_fp8_uses_each_layers_own_scales():
    _check_layers_fp8(O.DraftContext.layers_fp8)


def test_layers_fp8_pin_catches_planted_mistakes():
    def swapped(self, ks, vs):
        return [O.fp8_kv(k, v, b, a) for k, v, a, b in zip(self.k, self.v, ks, vs)]

    def first_layer_scales(self, ks, vs):
        return [O.fp8_kv(k, v, ks[0], vs[0]) for k, v in zip(self.k, self.v)]

    def unscaled(self, ks, vs):
        return [O.fp8_kv(k, v, 1.0, 1.0) for k, v in zip(self.k, self.v)]

    for wrong in (swapped, first_layer_scales, unscaled):
        with pytest.raises(AssertionError):
            _check_layers_fp8(wrong)


# ----------------------------------------------------------- draft KV windowing
# [P1]: "with draft windowing enabled, the draft uses a private compact mapping
# over the shared global index space"; --speculative-dflash-draft-window-size.
# Reading: keep the most recent W_d committed rows at their positions; every
# block query sees exactly those rows (and the block); sliding layers still
# apply their own window.
def _masked_per_query(q, k, v, kb, vb, q_pos, kv_len, draft_window, layer_window):
    """Attention over the full context with the rows before kv_len - W_d
    hidden, one query at a time: for query j at kv_len + j a per-query window
    of W_d + j + 1 hides exactly those rows (block keys are always seen); a
    layer window W is the smaller of the two."""
    out = []
    for j in range(q.shape[0]):
        w = draft_window + j + 1
        if layer_window:
            w = min(w, layer_window)
        out.append(O.block_attention(q[j:j + 1], k, v, kb, vb, q_pos[j:j + 1],
                                     np.arange(kv_len), w))
    return np.concatenate(out, axis=0)


@pytest.mark.parametrize("draft_window,layer_window", [(7, 0), (7, 4), (25, 0), (1, 0)])
def test_compact_window_store_equals_masked_full_context(draft_window, layer_window):
    rng = np.random.default_rng(40 + draft_window + layer_window)
    kv_len, S, kvh, nh, D = 20, 4, 2, 4, 8
    k, v = rng.normal(size=(kv_len, kvh, D)), rng.normal(size=(kv_len, kvh, D))
    kb, vb = rng.normal(size=(S, kvh, D)), rng.normal(size=(S, kvh, D))
    q = rng.normal(size=(S, nh, D))
    q_pos = kv_len + np.arange(S)
    lo = max(0, kv_len - draft_window)
    compact = O.block_attention(q, k[lo:], v[lo:], kb, vb, q_pos, np.arange(lo, kv_len), layer_window)
    masked = _masked_per_query(q, k, v, kb, vb, q_pos, kv_len, draft_window, layer_window)
    assert np.allclose(compact, masked, rtol=1e-12, atol=1e-12)


def test_window_store_keeps_the_newest_rows_at_their_positions():
    cfg = tiny_cfg()
    rng = np.random.default_rng(41)
    W = tiny_weights(cfg, rng)
    ctx = O.DraftContext(cfg)
    ctx.inject([rng.normal(size=(9, cfg.target_hidden)) for _ in range(cfg.n_sel)], W)
    layers, pos = ctx.window_layers(4)
    assert pos.tolist() == [5, 6, 7, 8]
    assert np.array_equal(layers[0][0], ctx.k[0][5:]) and np.array_equal(layers[1][1], ctx.v[1][5:])
    # a window at least as long as the context changes nothing
    full, hf, _ = O.draft_block(cfg, W, 3, ctx.layers(), ctx.kv_len)
    same, hs, _ = O.draft_block_windowed(cfg, W, 3, ctx, 9)
    assert np.array_equal(full, same) and np.allclose(hf, hs, rtol=0, atol=0)
    # a short window does change the block's hidden states
    _, hw, _ = O.draft_block_windowed(cfg, W, 3, ctx, 2)
    assert not np.allclose(hw, hf)


def test_window_pins_catch_planted_mistakes(monkeypatch):
    """Re-basing the kept rows' positions to 0 breaks a layer window on top."""
    orig = O.DraftContext.window_layers

    def rebased(self, draft_window):
        layers, pos = orig(self, draft_window)
        return layers, np.arange(len(pos), dtype=np.int64)
    rng = np.random.default_rng(42)
    kv_len, S, kvh, nh, D = 20, 4, 2, 4, 8
    k, v = rng.normal(size=(kv_len, kvh, D)), rng.normal(size=(kv_len, kvh, D))
    kb, vb = rng.normal(size=(S, kvh, D)), rng.normal(size=(S, kvh, D))
    q = rng.normal(size=(S, nh, D))
    q_pos = kv_len + np.arange(S)
    ctx = SimpleNamespace(k=[k], v=[v], kv_len=kv_len)
    layers, pos = rebased(ctx, 7)
    wrong = O.block_attention(q, layers[0][0], layers[0][1], kb, vb, q_pos, pos, 4)
    right = _masked_per_query(q, k, v, kb, vb, q_pos, kv_len, 7, 4)
    assert not np.allclose(wrong, right)
