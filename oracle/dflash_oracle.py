"""Plain CPU oracle of the DFlash draft pass (test infrastructure only).

This module is the independent checker for the CUDA library in
``block_diffusion_speculative_fc_gb300``.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path never does.  It shares no code, tables or
constants with the CUDA path and imports nothing from it.

Everything is numpy in float64: inputs (weights, target features, which may
have been rounded to bf16 by the input generator) are widened to float64 and
every intermediate stays float64.  Contractions use ``numpy`` matmul; there is
no blocking, fusion or reordering beyond the definitions below.

Sources (three web pages on the method):
  [P1] "Inside SGLang: DFlash and DFlash 2 Implementation" (blog walkthrough).
  [P2] "[Feature] Spec V2 DFlash Support", sgl-project/sglang PR #23000.
  [P3] CSDN article "DFlash基本原理 / DFlash推理流程" (z-lab generate loop,
       Kimi-K2.6 draft config, SGLang flow, fused_kv_materialize).

Readings taken where the pages are silent (each is also pinned by a test):
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * g over the last axis.
  * q/k norm: RMSNorm per head over head_dim with one gain vector [D]
    shared by all heads.
  * RoPE: neox ("rotate half") on the full head_dim, frequency
    f_i = theta^(-2i/D) for i < D/2, pair (i, i + D/2).
  * attention: scale 1/sqrt(D); query head h reads KV head h // (n_h/KVH).
  * sliding window W > 0: a context key at position pk is visible to a
    query at position pq iff pq - pk < W; block keys are always visible.
  * no biases anywhere; argmax returns the lowest index among equal maxima.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
(worked examples printed on the pages, closed forms, invariants, brute force).
The DFlash 2 selector (compute_candidates, selector_walk,
draft_block_selector) and the sampled verification with a real proposal
(accept_block_sampled_q) are pinned by hand-built lattices, reductions to the
plain drafter and rule, and distribution tests of the walk and of
losslessness; the pages print no numeric selector example.  The FP8 KV
cache (e4m3_decode, e4m3_encode, fp8_kv) is pinned by the format's fixed
values, exhaustive round trips, ties and saturation, and the card's 12 KiB
per token.  Draft KV windowing (DraftContext.window_layers,
draft_block_windowed) is pinned against the full context masked per query.
The composition ``draft_forward`` has no printed numeric example on the pages;
it is pinned through its pinned parts and through an independent loop-level
restatement in the test suite ("parity unpinned by the pages" for the
composite as a whole).
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a):
    return np.asarray(a, dtype=F64)


# ---------------------------------------------------------------------------
# Step 1: context features.  [P3] "target model prefill": the feature of layer
# id j is hidden_states[j + 1] (index 0 holds the embedding output), and the
# selected states are concatenated along the feature axis in list order.
# ---------------------------------------------------------------------------
def extract_context_feature(hidden_states, layer_ids):
    """hidden_states: list (embedding output first) of [rows, H_t] arrays."""
    picked = [_f64(hidden_states[j + 1]) for j in layer_ids]
    return np.concatenate(picked, axis=-1)


def rms_norm(x, g, eps):
    """RMSNorm over the last axis."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(g)


def head_rms_norm(x, g, eps):
    """Per-head RMSNorm: x [..., heads, D], one gain g [D] for all heads."""
    return rms_norm(x, g, eps)


def rope_frequencies(head_dim, theta):
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * i / head_dim)


def rope_neox(x, positions, theta):
    """Rotate-half RoPE.  x [n, heads, D]; positions [n] (integers).

    Component i (i < D/2) and component i + D/2 form one plane, rotated by
    the angle positions * f_i.
    """
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(positions, dtype=F64)[:, None] * rope_frequencies(d, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def linear(x, w):
    """y = x w^T with w in [out, in] layout (no bias)."""
    return _f64(x) @ _f64(w).T


# [P1] Step 1 ("project_target_hidden(): fc + hidden_norm"); [P3] "target_hidden
# = self.hidden_norm(self.fc(target_hidden))".
def project_target_hidden(feats, fc_w, hidden_norm_g, eps):
    """feats: list of n_sel arrays [rows, H_t] in target_layer_ids order."""
    x = np.concatenate([_f64(f) for f in feats], axis=-1)
    return rms_norm(linear(x, fc_w), hidden_norm_g, eps)


def split_qkv(w_qkv, cfg):
    """Rows of the fused projection: q (n_h*D), then k (KVH*D), then v."""
    nq = cfg.n_heads * cfg.head_dim
    nk = cfg.n_kv_heads * cfg.head_dim
    return w_qkv[:nq], w_qkv[nq:nq + nk], w_qkv[nq + nk:nq + 2 * nk]


# [P1] Step 1 (kv_proj_only -> apply_k_norm -> apply_k_rope -> set_kv_buffer,
# once per draft layer); [P3] "fused_kv_materialize" computes the same thing.
def context_kv(y_hat, layer_w, positions, cfg):
    """K/V of projected context rows for one draft layer.

    Returns K, V of shape [rows, KVH, D]; K is k-normed then rotated.
    """
    _, wk, wv = split_qkv(layer_w["qkv"], cfg)
    rows = y_hat.shape[0]
    k = linear(y_hat, wk).reshape(rows, cfg.n_kv_heads, cfg.head_dim)
    v = linear(y_hat, wv).reshape(rows, cfg.n_kv_heads, cfg.head_dim)
    k = head_rms_norm(k, layer_w["k_norm"], cfg.rms_eps)
    k = rope_neox(k, positions, cfg.rope_theta)
    return k, v


def block_attention(q, k_ctx, v_ctx, k_blk, v_blk, q_pos, ctx_pos, window):
    """Non-causal block attention ([P1] Step 4; [P3] is_causal=False).

    q [S, n_h, D]; context keys/values [T, KVH, D] at positions ctx_pos [T];
    block keys/values [S, KVH, D], always visible to every block query.
    window > 0 keeps a context key only when q_pos - ctx_pos < window.
    """
    S, n_h, D = q.shape
    kvh = k_blk.shape[1]
    group = n_h // kvh
    keys = np.concatenate([_f64(k_ctx), _f64(k_blk)], axis=0)      # [T+S, KVH, D]
    vals = np.concatenate([_f64(v_ctx), _f64(v_blk)], axis=0)
    T, n_blk = k_ctx.shape[0], k_blk.shape[0]
    visible = np.ones((S, T + n_blk), dtype=bool)
    if window and window > 0 and T > 0:
        dist = np.asarray(q_pos, dtype=np.int64)[:, None] - np.asarray(ctx_pos, dtype=np.int64)[None, :]
        visible[:, :T] = dist < window
    out = np.empty((S, n_h, D), dtype=F64)
    scale = 1.0 / np.sqrt(F64(D))
    for h in range(n_h):
        kv = h // group
        scores = (_f64(q[:, h, :]) @ keys[:, kv, :].T) * scale     # [S, T+n_blk]
        scores = np.where(visible, scores, -np.inf)
        m = scores.max(axis=1, keepdims=True)
        p = np.exp(scores - m)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vals[:, kv, :]
    return out


def silu(x):
    return x / (1.0 + np.exp(-x))


def draft_layer(x, layer_w, k_ctx, v_ctx, positions, window, cfg, ctx_pos=None):
    """One DFlashDecoderLayer on the block rows of one request.

    x [S, H] residual stream; returns the updated residual stream.  The
    block K/V computed here live only for this pass and are never committed.
    ctx_pos: positions of the context rows (default 0, 1, ...).
    """
    S = x.shape[0]
    D = cfg.head_dim
    h = rms_norm(x, layer_w["in_norm"], cfg.rms_eps)
    wq, wk, wv = split_qkv(layer_w["qkv"], cfg)
    q = linear(h, wq).reshape(S, cfg.n_heads, D)
    k = linear(h, wk).reshape(S, cfg.n_kv_heads, D)
    v = linear(h, wv).reshape(S, cfg.n_kv_heads, D)
    q = rope_neox(head_rms_norm(q, layer_w["q_norm"], cfg.rms_eps), positions, cfg.rope_theta)
    k = rope_neox(head_rms_norm(k, layer_w["k_norm"], cfg.rms_eps), positions, cfg.rope_theta)
    if ctx_pos is None:
        ctx_pos = np.arange(k_ctx.shape[0], dtype=np.int64)
    a = block_attention(q, k_ctx, v_ctx, k, v, positions, ctx_pos, window)
    x = x + linear(a.reshape(S, cfg.n_heads * D), layer_w["o"])
    h2 = rms_norm(x, layer_w["post_norm"], cfg.rms_eps)
    gu = linear(h2, layer_w["gate_up"])
    gate, up = gu[:, :cfg.intermediate], gu[:, cfg.intermediate:]
    x = x + linear(silu(gate) * up, layer_w["down"])
    return x


# [P1] Step 3 (block_ids = [anchor, MASK...], positions = prefix + j) and
# Step 4 (backbone, final norm); [P3] "draft model predict".
def draft_forward(cfg, W, anchor, ctx_kv_layers, kv_len, ctx_pos=None):
    """Draft backbone for one request.

    ctx_kv_layers: per layer (K [kv_len, KVH, D], V) of the committed context
    (or, with ctx_pos, of the context rows at those positions).
    Returns the final-normed hidden states [S, H].
    """
    S = cfg.block_size
    ids = np.full(S, cfg.mask_token_id, dtype=np.int64)
    ids[0] = anchor
    x = _f64(W["embed"])[ids]
    positions = kv_len + np.arange(S, dtype=np.int64)
    for l in range(cfg.n_layers):
        kc, vc = ctx_kv_layers[l]
        x = draft_layer(x, W["layers"][l], kc[:kv_len], vc[:kv_len], positions,
                        cfg.sliding_window[l], cfg, ctx_pos)
    return rms_norm(x, W["final_norm"], cfg.rms_eps)


# [P1] Step 4 ("selects from draft_hidden[:, 1:, :] using the target vocabulary
# head"); plain DFlash proposes argmax tokens ([P1] Sampling).
def lm_head_argmax(hidden_rows, lm_head):
    """Greedy ids and the top-2 logit margin of each row.

    Ties resolve to the lowest index (numpy argmax convention).
    """
    logits = _f64(hidden_rows) @ _f64(lm_head).T
    ids = np.argmax(logits, axis=1)
    srt = np.sort(logits, axis=1)
    margin = srt[:, -1] - srt[:, -2] if logits.shape[1] > 1 else np.full(len(ids), np.inf)
    return ids.astype(np.int64), margin


def draft_block(cfg, W, anchor, ctx_kv_layers, kv_len):
    """Full draft pass for one request: ids [S] (col 0 = anchor), hidden [S, H], margins [S-1]."""
    hid = draft_forward(cfg, W, anchor, ctx_kv_layers, kv_len)
    ids, margin = lm_head_argmax(hid[1:], W["lm_head"])
    out = np.empty(cfg.block_size, dtype=np.int64)
    out[0] = anchor
    out[1:] = ids
    return out, hid, margin


def draft_block_windowed(cfg, W, anchor, ctx, draft_window):
    """draft_block over the compact store of the last draft_window rows."""
    layers, pos = ctx.window_layers(draft_window)
    hid = draft_forward(cfg, W, anchor, layers, ctx.kv_len, pos)
    ids, margin = lm_head_argmax(hid[1:], W["lm_head"])
    out = np.empty(cfg.block_size, dtype=np.int64)
    out[0] = anchor
    out[1:] = ids
    return out, hid, margin


# ---------------------------------------------------------------------------
# Step 3: verification.  [P3] "target model verify":
#   acceptance_length = sum(cumprod(block[1:] == posterior[:-1]))
# [P1] Step 6: commit_lens = accept_len + 1, bonus = posterior[accept_len],
# out_tokens = accepted drafts, then bonus, then padding.
# ---------------------------------------------------------------------------
def accept_block(draft, posterior):
    draft = np.asarray(draft, dtype=np.int64)
    posterior = np.asarray(posterior, dtype=np.int64)
    S = draft.shape[0]
    matches = (draft[1:] == posterior[:-1]).astype(np.int64)
    acc = int(np.cumprod(matches).sum()) if S > 1 else 0
    bonus = int(posterior[acc])
    out = np.zeros(S, dtype=np.int64)
    out[:acc] = draft[1:acc + 1]
    out[acc] = bonus
    return acc, bonus, acc + 1, out


# ---------------------------------------------------------------------------
# Lossless sampled verification ([P1] "Sampling: preserve the proposal
# distribution the walk actually used"): a proposed token y is accepted with
# probability min(1, p(y)/q(y)); at the first rejection the correction is drawn
# from the normalised positive residual [p - q]+; after full acceptance the
# target supplies a bonus token.  The plain DFlash drafter proposes argmax
# tokens (same section), so q is a point mass at y: y is accepted iff
# u < p(y), and [p - q]+ is p with y's entry set to 0 (p(y) - 1 <= 0).
# Random numbers are inputs: accept_u [S-1] uniform on [0, 1) and exp_noise
# [V] Exp(1) variates for the one draw the block needs.  A draw from weights
# w is argmax_v w(v) / e_v (the exponential race: the smallest of independent
# Exp(rate w_v) times e_v / w_v falls on v with probability w_v / sum w),
# lowest id on ties.  Decisions are taken in float32 (probabilities, uniforms,
# quotients), as the kernel takes them.
# ---------------------------------------------------------------------------
def exponential_race(weights, exp_noise):
    w = np.asarray(weights, dtype=np.float32)
    e = np.asarray(exp_noise, dtype=np.float32)
    keys = w / e
    return int(np.argmax(keys))


def accept_block_sampled(draft, probs, accept_u, exp_noise):
    """draft [S] int; probs [S, V] float32 target distribution at block
    position i (the target's choice for the token after draft[i]); accept_u
    [S-1]; exp_noise [V].  Returns (accept, bonus, commit, out_tokens) as
    accept_block does."""
    draft = np.asarray(draft, dtype=np.int64)
    probs = np.asarray(probs, dtype=np.float32)
    u = np.asarray(accept_u, dtype=np.float32)
    S = draft.shape[0]
    acc = 0
    while acc < S - 1 and u[acc] < probs[acc, draft[acc + 1]]:
        acc += 1
    w = probs[acc].copy()
    if acc < S - 1:
        w[draft[acc + 1]] = 0.0          # [p - q]+ with q the point mass at the rejected token
    bonus = exponential_race(w, exp_noise)
    out = np.zeros(S, dtype=np.int64)
    out[:acc] = draft[1:acc + 1]
    out[acc] = bonus
    return acc, bonus, acc + 1, out


# ---------------------------------------------------------------------------
# DFlash 2 candidate selector ([P1] "DFlash 2: replace selection, retain the
# serving loop").  After the one backbone pass, every draft position j = 1..S-1
# keeps the K highest lm_head logits as candidates (compute_candidates: ids
# and their "unary" logits U).  A transition from predecessor token p to
# candidate c at position j scores
#     score_j(p, c) = U_j(c) + < A[p] * (W_h h_j), B[c] >
# (the successor's unary logit plus a learned low-rank compatibility term;
# A, B: [V, r] token factors, W_h: [r, H], h_j the final-normed hidden state
# of position j).  The predecessor of the first prediction is the anchor; of
# every later one, the candidate the walk chose at the position before.  The
# walk goes left to right once, choosing greedily (highest score, earliest
# candidate on ties) or by sampling from softmax(score_j(p, .)) over the K
# candidates; it does not search for the best full path.  q_rows[j] is that
# softmax for the predecessor actually chosen: the proposal distribution a
# lossless sampled verification needs.
# Readings where the pages are silent: candidates are ordered by logit,
# highest first, lower id first among equal logits; no temperature (scores
# are used as they are); h_j is the same final-normed hidden state the lm_head
# reads; a sampled choice is the exponential race over q_rows[j] with one
# Exp(1) variate per candidate, as in the verification above.
# ---------------------------------------------------------------------------
def compute_candidates(hidden_rows, lm_head, K):
    """Top-K ids [R, K] (logit order, lower id first on ties) and their logits [R, K]."""
    logits = _f64(hidden_rows) @ _f64(lm_head).T
    V = logits.shape[1]
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= vocab")
    ids = np.empty((logits.shape[0], K), dtype=np.int64)
    for r in range(logits.shape[0]):
        ids[r] = np.argsort(-logits[r], kind="stable")[:K]
    return ids, np.take_along_axis(logits, ids, axis=1)


def selector_scores(unary_row, cand_row, pred, wh_row, A, B):
    """score(pred, c) for the K candidates c of one position."""
    return _f64(unary_row) + (_f64(A)[pred] * _f64(wh_row)) @ _f64(B)[np.asarray(cand_row)].T


def softmax(x):
    x = _f64(x)
    e = np.exp(x - x.max())
    return e / e.sum()


def selector_walk(anchor, cand, unary, wh, A, B, exp_noise=None):
    """cand, unary [S-1, K]; wh [S-1, r].  Greedy walk when exp_noise is None,
    else sampled with exp_noise [S-1, K] Exp(1) variates.  Returns the chosen
    ids [S-1], the chosen candidate slots [S-1] and q_rows [S-1, K] (float64)."""
    cand = np.asarray(cand, dtype=np.int64)
    n, K = cand.shape
    ids = np.empty(n, dtype=np.int64)
    slots = np.empty(n, dtype=np.int64)
    q = np.empty((n, K))
    pred = int(anchor)
    for j in range(n):
        sc = selector_scores(unary[j], cand[j], pred, wh[j], A, B)
        q[j] = softmax(sc)
        k = int(np.argmax(sc)) if exp_noise is None else exponential_race(q[j], exp_noise[j])
        slots[j] = k
        ids[j] = cand[j, k]
        pred = int(ids[j])
    return ids, slots, q


def draft_block_selector(cfg, W, sel, anchor, ctx_kv_layers, kv_len, K, exp_noise=None):
    """DFlash 2 draft pass for one request: ids [S] (col 0 = anchor), candidate
    ids [S-1, K], their logits [S-1, K], q_rows [S-1, K], wh [S-1, r] and the
    hidden states [S, H].  sel: {"A": [V, r], "B": [V, r], "W_h": [r, H]}."""
    hid = draft_forward(cfg, W, anchor, ctx_kv_layers, kv_len)
    cand, unary = compute_candidates(hid[1:], W["lm_head"], K)
    wh = hid[1:] @ _f64(sel["W_h"]).T
    ids, _, q = selector_walk(anchor, cand, unary, wh, sel["A"], sel["B"], exp_noise)
    out = np.empty(cfg.block_size, dtype=np.int64)
    out[0] = anchor
    out[1:] = ids
    return out, cand, unary, q, wh, hid


# Sampled verification of a drafter with a real proposal distribution (the
# selector's q_rows over its K candidates; zero elsewhere).  Proposed token y
# at position i is accepted iff u_i < p(y) / q(y); at the first rejection the
# correction is the exponential race over [p - q]+, after full acceptance over
# the target's last row.  Decisions in float32, as the kernel takes them.
def accept_block_sampled_q(draft, probs, cand, q_rows, accept_u, exp_noise):
    """draft [S]; probs [S, V] float32; cand [S-1, K] ids with q_rows [S-1, K]
    their proposal probabilities; accept_u [S-1]; exp_noise [V]."""
    draft = np.asarray(draft, dtype=np.int64)
    probs = np.asarray(probs, dtype=np.float32)
    cand = np.asarray(cand, dtype=np.int64)
    q = np.asarray(q_rows, dtype=np.float32)
    u = np.asarray(accept_u, dtype=np.float32)
    S = draft.shape[0]

    def q_of(i, y):
        hit = np.nonzero(cand[i] == y)[0]
        return q[i, hit[0]] if len(hit) else np.float32(0.0)

    acc = 0
    while acc < S - 1:
        y = draft[acc + 1]
        qy = q_of(acc, y)
        if not (qy > 0 and u[acc] < np.float32(probs[acc, y] / qy)):
            break
        acc += 1
    w = probs[acc].copy()
    if acc < S - 1:
        for k in range(cand.shape[1]):
            c = cand[acc, k]
            w[c] = np.maximum(np.float32(w[c] - q[acc, k]), np.float32(0.0))
    bonus = exponential_race(w, exp_noise)
    out = np.zeros(S, dtype=np.int64)
    out[:acc] = draft[1:acc + 1]
    out[acc] = bonus
    return acc, bonus, acc + 1, out


def commit_output(output_ids, start, draft, acc, bonus):
    """[P3] verify step: output_ids[start:start+acc+1] = block[:acc+1];
    output_ids[start+acc+1] = bonus; the new start (crop index) is start+acc+1."""
    output_ids = np.array(output_ids, copy=True)
    output_ids[start:start + acc + 1] = np.asarray(draft, dtype=np.int64)[:acc + 1]
    output_ids[start + acc + 1] = bonus
    return output_ids, start + acc + 1


# ---------------------------------------------------------------------------
# FP8 draft KV cache ([P3] Kimi-K2.6 draft card: "12 KiB / token (FP8)" for
# 6 layers x 2 (K, V) x 8 KV heads x 128 dims -- one byte per element and no
# per-token scale).  Readings where the pages are silent: the OCP 8-bit
# floating-point format E4M3 (1 sign bit, 4 exponent bits with bias 7, 3
# mantissa bits, subnormals, no infinities, S.1111.111 = NaN, largest finite
# value 448); an element x is stored as the code nearest to x / scale (ties
# to the code with an even mantissa, magnitudes beyond 448 saturate to 448,
# the sign is kept, NaN -> 0x7F), with one caller-given scale per layer and
# per tensor (K, V); attention reads code value * scale.
# ---------------------------------------------------------------------------
def e4m3_decode(code):
    """Value of E4M3 codes 0..255 (NaN for 0x7F and 0xFF)."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(F64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(F64)))
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x):
    """Nearest E4M3 code of each element (see the readings above): the two
    finite codes whose values bracket |x| (found by bisection over the
    ascending values of codes 0x00..0x7E), the nearer of the two, the one with
    the even mantissa when both are equally near."""
    x = np.asarray(x, dtype=F64)
    vals = e4m3_decode(np.arange(0x7F))               # 0x00 .. 0x7E, ascending values
    a = np.minimum(np.abs(x), 448.0).reshape(-1)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    even = np.where(lo % 2 == 0, lo, hi)              # the mantissa's last bit is the code's
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, even))
    pick = np.where(np.isnan(a), 0, pick)
    code = pick | np.where(np.signbit(x.reshape(-1)), 0x80, 0)
    code = np.where(np.isnan(x.reshape(-1)), 0x7F, code)
    return code.reshape(x.shape).astype(np.int64)


def fp8_kv(k, v, k_scale, v_scale):
    """K, V as an FP8 cache reads them back: decode(encode(x / scale)) * scale."""
    dq = lambda t, sc: e4m3_decode(e4m3_encode(_f64(t) / sc)) * sc  # noqa: E731
    return dq(k, k_scale), dq(v, v_scale)


class DraftContext:
    """Committed draft K/V of one request: per layer K, V [rows, KVH, D].

    Context row i sits at position i: rows are appended at positions
    kv_len .. kv_len + n - 1 and nothing is ever overwritten.
    """

    def __init__(self, cfg):
        self.cfg = cfg
        shape = (0, cfg.n_kv_heads, cfg.head_dim)
        self.k = [np.zeros(shape, F64) for _ in range(cfg.n_layers)]
        self.v = [np.zeros(shape, F64) for _ in range(cfg.n_layers)]

    @property
    def kv_len(self):
        return self.k[0].shape[0]

    def layers(self):
        return list(zip(self.k, self.v))

    # Draft KV windowing ([P1]: "with draft windowing enabled, the draft uses
    # a private compact mapping over the shared global index space";
    # --speculative-dflash-draft-window-size).  Reading: the draft keeps the
    # most recent draft_window committed rows of a request, at their original
    # positions (their K keeps the rotation of its position); every block
    # query sees exactly those rows and the block, and a sliding layer still
    # applies its own window on top.
    def window_layers(self, draft_window):
        """The compact store: per-layer (K, V) of the kept rows and their positions."""
        lo = max(0, self.kv_len - int(draft_window))
        return ([(k[lo:], v[lo:]) for k, v in zip(self.k, self.v)],
                np.arange(lo, self.kv_len, dtype=np.int64))

    def layers_fp8(self, k_scales, v_scales):
        """The committed K/V as an FP8 cache with per-layer scales holds them."""
        return [fp8_kv(k, v, ks, vs) for k, v, ks, vs in zip(self.k, self.v, k_scales, v_scales)]

    # [P1] Step 7: only the committed prefix rows of the verify features become
    # context (prefix-valid writes).
    def inject(self, feats, W):
        cfg = self.cfg
        y_hat = project_target_hidden(feats, W["fc"], W["hidden_norm"], cfg.rms_eps)
        self.append_projected(y_hat, W)
        return y_hat

    def append_projected(self, y_hat, W):
        """Append rows whose fc + hidden_norm projection is already known."""
        pos = self.kv_len + np.arange(y_hat.shape[0], dtype=np.int64)
        for l in range(self.cfg.n_layers):
            k, v = context_kv(y_hat, W["layers"][l], pos, self.cfg)
            self.k[l] = np.concatenate([self.k[l], k], axis=0)
            self.v[l] = np.concatenate([self.v[l], v], axis=0)
