"""Brute-force scalar MLA decode in pure Python, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Written independently
of ``oracle.mla``: plain lists and ``math``, no NumPy, no matrix routine, so
that a slip in the vectorised oracle (a transposed operand, a wrong slice, a
dropped term) shows up as a disagreement.

It follows the explicit definition on page "DeepSeek-V2：在“大力出奇迹”的AI军备
竞赛中，四两拨千斤" (liang.world), 第二章 §1-§3: compress, RoPE key, per-head
K/V up-projection, decoupled query/key concatenation, per-head softmax
attention, concatenation and W_O.  Readings (scale, RoPE form, orientation)
are the same stated assumptions as ``oracle.mla``.
"""
from __future__ import annotations

import math


def _matvec(W, x):
    """W given as a list of rows; returns W x."""
    out = []
    for row in W:
        acc = 0.0
        for a, b in zip(row, x):
            acc += a * b
        out.append(acc)
    return out


def _rot(x, pos, base):
    d = len(x)
    y = [0.0] * d
    for j in range(d // 2):
        ang = pos * base ** (-2.0 * j / d)
        x0, x1 = x[2 * j], x[2 * j + 1]
        y[2 * j] = x0 * math.cos(ang) - x1 * math.sin(ang)
        y[2 * j + 1] = x0 * math.sin(ang) + x1 * math.cos(ang)
    return y


def decode(dims, h, q, w, T):
    """h: list of S hidden rows (positions 0..S-1); q: [T][n_h][d_nope+d_R].

    Returns u as a list of T rows of length d.
    """
    H, dn, dv, dr = dims.n_heads, dims.d_nope, dims.d_v, dims.d_rope
    base = dims.rope_base
    scale = 1.0 / math.sqrt(dn + dr)
    S = len(h)
    c = [_matvec(w["w_dkv"], h[p]) for p in range(S)]
    kr = [_rot(_matvec(w["w_kr"], h[p]), p, base) for p in range(S)]
    u_all = []
    for t in range(T):
        s_pos = S - T + t
        concat_o = []
        for i in range(H):
            w_uk_i = w["w_uk"][i * dn:(i + 1) * dn]
            w_uv_i = w["w_uv"][i * dv:(i + 1) * dv]
            q_i = list(q[t][i][:dn]) + _rot(list(q[t][i][dn:]), s_pos, base)
            scores = []
            values = []
            for p in range(s_pos + 1):
                k_ip = _matvec(w_uk_i, c[p]) + kr[p]
                dot = 0.0
                for a, b in zip(q_i, k_ip):
                    dot += a * b
                scores.append(dot * scale)
                values.append(_matvec(w_uv_i, c[p]))
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            z = sum(e)
            o_i = [0.0] * dv
            for p in range(s_pos + 1):
                for k in range(dv):
                    o_i[k] += e[p] / z * values[p][k]
            concat_o.extend(o_i)
        u_all.append(_matvec(w["w_o"], concat_o))
    return u_all


def query(dims, h_row, w):
    """Scalar query of one hidden row: [n_h][d_nope + d_R], q^R un-rotated.

    c^Q = W^DQ h, q^C = W^UQ c^Q and q^R = W^QR h, head i taking its rows
    of each (the decode rotates q^R at the query position).
    """
    H, dn, dr = dims.n_heads, dims.d_nope, dims.d_rope
    c_q = _matvec(w["w_dq"], h_row)
    q_c = _matvec(w["w_uq"], c_q)
    q_r = _matvec(w["w_qr"], h_row)
    return [q_c[i * dn:(i + 1) * dn] + q_r[i * dr:(i + 1) * dr] for i in range(H)]


def decode_layers(dims, layers, h_new, T):
    """Scalar decode through a stack of layers: h_{j+1} = h_j + u_j.

    layers[j]: {"w": matrices as row lists, "prefix_h": hidden rows of the
    cached positions of layer j}; h_new: T rows of layer 0's new hidden
    states.  Each layer's cache is its prefix rows followed by the rows of
    its own input; its queries come from its own input.
    """
    h = [list(r) for r in h_new]
    for layer in layers:
        w = layer["w"]
        seq = [list(r) for r in layer["prefix_h"]] + h
        q = [query(dims, r, w) for r in h]
        u = decode(dims, seq, q, w, T)
        h = [[a + b for a, b in zip(hr, ur)] for hr, ur in zip(h, u)]
    return h
