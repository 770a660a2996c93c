"""Loop-only scalar restatement of the block, for tiny cases (test pin).

Pure Python floats and ``math``/``cmath``: no NumPy arithmetic, no
vectorisation, nothing shared with ``oracle/``. The rotary is written in the
complex form (pair (x_j, x_{j+r/2}) as x_j + i x_{j+r/2}, multiplied by
e^{i p theta_j}), a formulation independent of the oracle's cos/sin
expansion. Used only to pin the oracle on inputs of a few dozen numbers.
"""
from __future__ import annotations

import cmath
import math


def _vec(t):
    return [float(v) for v in t]


def _mat(t):
    return [[float(v) for v in row] for row in t]


def ln(row, g, b, eps):
    n = len(row)
    mu = sum(row) / n
    var = sum((v - mu) * (v - mu) for v in row) / n
    inv = 1.0 / math.sqrt(var + eps)
    return [(row[i] - mu) * inv * g[i] + (b[i] if b is not None else 0.0) for i in range(n)]


def rms(row, w, eps):
    n = len(row)
    inv = 1.0 / math.sqrt(sum(v * v for v in row) / n + eps)
    return [row[i] * inv * w[i] for i in range(n)]


def matvec(W, x, b=None):
    out = []
    for o in range(len(W)):
        acc = 0.0
        for i in range(len(x)):
            acc += W[o][i] * x[i]
        out.append(acc + (b[o] if b is not None else 0.0))
    return out


def rope_vec(vec, p, r, base):
    out = list(vec)
    h = r // 2
    for j in range(h):
        z = complex(vec[j], vec[j + h]) * cmath.exp(1j * p * base ** (-2.0 * j / r))
        out[j], out[j + h] = z.real, z.imag
    return out


def silu(z):
    return z / (1.0 + math.exp(-z))


def gelu_tanh(z):
    return 0.5 * z * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z * z * z)))


def block(cfg, x, weights):
    """y[b][s][:] for the block variant ``cfg`` (tiny sizes only)."""
    B, S, D = cfg.batch, cfg.seq, cfg.hidden
    H, Hk, d, r = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rotary_span
    W = {}
    for k_, t in weights.items():
        W[k_] = _mat(t) if t.dim() == 2 else _vec(t)
    X = [[_vec(x[b, s]) for s in range(S)] for b in range(B)]

    def norm(row, wn, bn):
        if cfg.norm == "layernorm":
            return ln(row, W[wn], W.get(bn), cfg.eps)
        return rms(row, W[wn], cfg.eps)

    def mlp(row):
        if cfg.act == "swiglu":
            g = matvec(W["w_gate"], row)
            u = matvec(W["w_up"], row)
            a = [silu(g[i]) * u[i] for i in range(len(g))]
        else:
            a = [gelu_tanh(z) for z in matvec(W["w_up"], row, W.get("b_up"))]
        return matvec(W["w_down"], a, W.get("b_down"))

    slopes = [2.0 ** (-8.0 * (i + 1) / H) for i in range(H)] if cfg.alibi else [0.0] * H
    Y = []
    for b in range(B):
        n1 = [norm(X[b][s], "attn_norm_w", "attn_norm_b") if cfg.norm_place == "pre"
              else list(X[b][s]) for s in range(S)]
        Q = [[None] * S for _ in range(H)]
        K = [[None] * S for _ in range(Hk)]
        V = [[None] * S for _ in range(Hk)]
        for s in range(S):
            y = matvec(W["w_qkv"], n1[s], W.get("b_qkv"))
            if cfg.qkv_layout == "stacked":
                qf = y[:H * d]
                kf = y[H * d:(H + Hk) * d]
                vf = y[(H + Hk) * d:]
            else:
                qf, kf, vf = [], [], []
                for h in range(H):
                    base_ = h * 3 * d
                    qf += y[base_:base_ + d]
                    kf += y[base_ + d:base_ + 2 * d]
                    vf += y[base_ + 2 * d:base_ + 3 * d]
            if cfg.qk_norm == "rms_full":
                qf = rms(qf, W["q_norm_w"], cfg.qk_norm_eps)
                kf = rms(kf, W["k_norm_w"], cfg.qk_norm_eps)
            for h in range(H):
                qh = qf[h * d:(h + 1) * d]
                if cfg.qk_norm == "ln_per_head":
                    qh = ln(qh, W["q_norm_w"][h], None, cfg.qk_norm_eps)
                Q[h][s] = rope_vec(qh, s, r, cfg.rope_base)
            for g in range(Hk):
                kh = kf[g * d:(g + 1) * d]
                if cfg.qk_norm == "ln_per_head":
                    kh = ln(kh, W["k_norm_w"][g], None, cfg.qk_norm_eps)
                K[g][s] = rope_vec(kh, s, r, cfg.rope_base)
                V[g][s] = vf[g * d:(g + 1) * d]
        rows = []
        for i in range(S):
            premix = []
            for h in range(H):
                g = h // (H // Hk)
                sc = []
                for j in range(i + 1):
                    dot = sum(Q[h][i][t] * K[g][j][t] for t in range(d))
                    sc.append(dot / math.sqrt(d) - slopes[h] * (i - j))
                m = max(sc)
                e = [math.exp(v - m) for v in sc]
                z = sum(e)
                premix += [sum(e[j] / z * V[g][j][t] for j in range(i + 1)) for t in range(d)]
            attn = matvec(W["w_o"], premix, W.get("b_o"))
            xs = X[b][i]
            if cfg.residual == "parallel":
                mo = mlp(n1[i])
                rows.append([xs[c] + attn[c] + mo[c] for c in range(D)])
            elif cfg.norm_place == "pre":
                h_ = [xs[c] + attn[c] for c in range(D)]
                mo = mlp(norm(h_, "mlp_norm_w", "mlp_norm_b"))
                rows.append([h_[c] + mo[c] for c in range(D)])
            else:
                an = rms(attn, W["post_attn_norm_w"], cfg.eps)
                h_ = [xs[c] + an[c] for c in range(D)]
                mn = rms(mlp(h_), W["post_mlp_norm_w"], cfg.eps)
                rows.append([h_[c] + mn[c] for c in range(D)])
        Y.append(rows)
    return Y
