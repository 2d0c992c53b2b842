"""Scalar, loop-by-loop restatement of the decoder forward for tiny sizes.

Used only to pin the fp64 oracle.  It is written as a different algorithm on
purpose: nested Python loops over scalars, rotary embedding as a complex
multiplication z * exp(i * pos * freq) with z = x_i + i x_{i+hd/2}, softmax
as exp / sum without max subtraction, no numpy.  A mistake shared with the
vectorised oracle would need the same error in both formulations.
"""
from __future__ import annotations

import cmath
import math


def matvec(w, x):
    """w: list of rows [out][in]; returns [out]."""
    return [sum(w[o][i] * x[i] for i in range(len(x))) for o in range(len(w))]


def rmsnorm(x, w, eps):
    ms = sum(v * v for v in x) / len(x)
    r = 1.0 / math.sqrt(ms + eps)
    return [w[i] * x[i] * r for i in range(len(x))]


def rotate(vec, pos, theta):
    hd = len(vec)
    half = hd // 2
    out = [0.0] * hd
    for i in range(half):
        freq = theta ** (-(2.0 * i) / hd)
        z = complex(vec[i], vec[i + half]) * cmath.exp(1j * pos * freq)
        out[i] = z.real
        out[i + half] = z.imag
    return out


def silu(z):
    return z / (1.0 + math.exp(-z))


def block(cfg, w, x, valid_start=None, rope=True, window=0, key_mask=None):
    """x: [B][T][d] nested lists; w: dict of nested lists.  rope=False leaves
    q and k unrotated (a NoPE block); window > 0 keeps only the `window` most
    recent keys of each query, its own included; key_mask[b][j] false hides
    key j of sequence b."""
    H, KV, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    B, T = len(x), len(x[0])
    out = []
    for b in range(B):
        vs = 0 if valid_start is None else int(valid_start[b])
        qs, ks, vs_ = [], [], []
        for t in range(T):
            pos = max(t - vs, 0)
            n = rmsnorm(x[b][t], w["attn_norm"], cfg.rms_eps)
            q = matvec(w["wq"], n)
            k = matvec(w["wk"], n)
            v = matvec(w["wv"], n)
            rot = (lambda u: rotate(u, pos, cfg.rope_theta)) if rope else (lambda u: list(u))
            qs.append([rot(q[h * hd:(h + 1) * hd]) for h in range(H)])
            ks.append([rot(k[h * hd:(h + 1) * hd]) for h in range(KV)])
            vs_.append([v[h * hd:(h + 1) * hd] for h in range(KV)])
        rows = []
        for t in range(T):
            o = []
            for h in range(H):
                kvh = h * KV // H
                keys = [j for j in range(T) if vs <= j <= t and (window == 0 or t - j < window)
                        and (key_mask is None or key_mask[b][j])]
                if not keys:
                    o.extend([0.0] * hd)
                    continue
                wts = [math.exp(sum(qs[t][h][c] * ks[j][kvh][c] for c in range(hd)) / math.sqrt(hd))
                       for j in keys]
                tot = sum(wts)
                for c in range(hd):
                    o.append(sum(wts[a] * vs_[j][kvh][c] for a, j in enumerate(keys)) / tot)
            attn = matvec(w["wo"], o)
            hrow = [x[b][t][i] + attn[i] for i in range(len(attn))]
            m = rmsnorm(hrow, w["mlp_norm"], cfg.rms_eps)
            g = matvec(w["wgate"], m)
            u = matvec(w["wup"], m)
            a = [silu(g[i]) * u[i] for i in range(len(g))]
            dn = matvec(w["wdown"], a)
            rows.append([hrow[i] + dn[i] for i in range(len(dn))])
        out.append(rows)
    return out


def model(cfg, layers, embed, final_norm, ids, kinds=None):
    """kinds: optional list of (rope, window) per layer."""
    x = [[list(embed[i]) for i in seq] for seq in ids]
    for l, w in enumerate(layers):
        rope, window = kinds[l] if kinds else (True, 0)
        x = block(cfg, w, x, rope=rope, window=window)
    logits = []
    for seq in x:
        logits.append([matvec(embed, rmsnorm(row, final_norm, cfg.rms_eps)) for row in seq])
    return logits
