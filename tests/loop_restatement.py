"""A second, loop-level statement of the draft backbone, for tiny shapes only.

Written independently of the oracle (explicit Python loops over rows,
features, heads and keys; math.* scalars), it pins how the oracle composes the
pinned parts: norm placement, residual adds, GQA head mapping, positions,
window and the SwiGLU order.  Source: "Inside SGLang: DFlash and DFlash 2
Implementation", Steps 3-4 (block ids, positions, decoder layers, final norm),
and the CSDN DFlash article, "draft model predict" (non-causal block pass).
"""
import math


def _rms(row, gain, eps):
    ms = sum(v * v for v in row) / len(row)
    r = 1.0 / math.sqrt(ms + eps)
    return [v * r * g for v, g in zip(row, gain)]


def _matvec(w, row):
    return [sum(w[o][i] * row[i] for i in range(len(row))) for o in range(len(w))]


def _rope(vec, pos, theta):
    d = len(vec)
    half = d // 2
    out = list(vec)
    for i in range(half):
        f = theta ** (-2.0 * i / d)
        c, s = math.cos(pos * f), math.sin(pos * f)
        a, b = vec[i], vec[i + half]
        out[i] = a * c - b * s
        out[i + half] = b * c + a * s
    return out


def draft_forward_loops(cfg, W, anchor, ctx_k, ctx_v, kv_len):
    """W: nested python lists; ctx_k/ctx_v[l][t][g][d]. Returns final hidden [S][H]."""
    S, H, D = cfg.block_size, cfg.hidden, cfg.head_dim
    nh, kvh = cfg.n_heads, cfg.n_kv_heads
    grp = nh // kvh
    eps = cfg.rms_eps
    x = [list(W["embed"][anchor if j == 0 else cfg.mask_token_id]) for j in range(S)]
    for l in range(cfg.n_layers):
        L = W["layers"][l]
        nq, nk = nh * D, kvh * D
        q_rows, k_rows, v_rows = L["qkv"][:nq], L["qkv"][nq:nq + nk], L["qkv"][nq + nk:]
        Q, K, V = [], [], []
        for j in range(S):
            h = _rms(x[j], L["in_norm"], eps)
            q, k, v = _matvec(q_rows, h), _matvec(k_rows, h), _matvec(v_rows, h)
            pos = kv_len + j
            Q.append([_rope(_rms(q[a * D:(a + 1) * D], L["q_norm"], eps), pos, cfg.rope_theta)
                      for a in range(nh)])
            K.append([_rope(_rms(k[g * D:(g + 1) * D], L["k_norm"], eps), pos, cfg.rope_theta)
                      for g in range(kvh)])
            V.append([v[g * D:(g + 1) * D] for g in range(kvh)])
        W_win = cfg.sliding_window[l]
        attn = []
        for j in range(S):
            pq = kv_len + j
            row = []
            for a in range(nh):
                g = a // grp
                keys, vals = [], []
                for t in range(kv_len):
                    if W_win == 0 or pq - t < W_win:
                        keys.append(ctx_k[l][t][g])
                        vals.append(ctx_v[l][t][g])
                for jj in range(S):
                    keys.append(K[jj][g])
                    vals.append(V[jj][g])
                sc = [sum(Q[j][a][d] * kk[d] for d in range(D)) / math.sqrt(D) for kk in keys]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                row.extend(sum(e[t] * vals[t][d] for t in range(len(vals))) / z for d in range(D))
            attn.append(row)
        for j in range(S):
            o = _matvec(L["o"], attn[j])
            x[j] = [x[j][i] + o[i] for i in range(H)]
            h2 = _rms(x[j], L["post_norm"], eps)
            gu = _matvec(L["gate_up"], h2)
            I = len(gu) // 2
            act = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
            dn = _matvec(L["down"], act)
            x[j] = [x[j][i] + dn[i] for i in range(H)]
    return [_rms(x[j], W["final_norm"], eps) for j in range(S)]
