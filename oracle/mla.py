"""Plain fp64 CPU oracle of Multi-head Latent Attention decode.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
the benchmark's CPU-baseline leg may import this module.  The CUDA library
never imports, links or calls it, and shares no code with it.

Sources (each function cites the place it follows):
  [V2-arch]   page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，四两拨千斤"
              (liang.world/post/deepseek-v2-architecture-revolution),
              第二章 "侠客甲——MLA": §1 (MHA), §2 (低秩键值联合压缩),
              §3 (解耦旋转位置嵌入).
  [DS-report] page "DeepSeek 系列模型技术深度解读"
              (tuntang.top/research/deepseek-technical-report), section
              "Multi-head Latent Attention (MLA)": "标准 MHA 的瓶颈",
              "MLA 的核心思想", table "MLA vs GQA 对比", "RoPE 的兼容性处理".
  [DS-pptc]   page www.pptc.cn/news/140720, §3.4 (cache the RoPE key too) and
              §6 问题二.

Readings where the pages are silent (each is a stated assumption):
  * softmax scale 1/sqrt(d_nope + d_rope) (1/sqrt(192) at V2 widths);
  * RoPE rotates interleaved pairs (x[2j], x[2j+1]) by angle pos * theta_j,
    theta_j = base**(-2j/d_rope), base 10000, positions counted from 0,
    as (x0 cos - x1 sin, x0 sin + x1 cos);
  * no biases and no normalisation on the latent;
  * matrices act on column vectors ("W h"): W^DKV [d_c, d], W^KR [d_R, d],
    W^UK [n_h*d_nope, d_c] and W^UV [n_h*d_v, d_c] with head i owning rows
    i*d_nope.. (resp. i*d_v..), W_O [d, n_h*d_v];
  * a query at position s sees cached positions 0..s (itself included).

Everything is float64 with no intermediate rounding.  Inputs are the exact
(bf16 or fp32) input values upcast to float64.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Closed forms of the cache size ([V2-arch] ch.2 §1 and §2, [DS-report] table)
# ---------------------------------------------------------------------------
def mha_cache_elems(n_heads: int, d_head: int, layers: int = 1) -> int:
    """Elements MHA caches per token: 2 * n_h * d_h per layer ([V2-arch] §1)."""
    return 2 * n_heads * d_head * layers


def mla_cache_elems(d_latent: int, d_rope: int, layers: int = 1) -> int:
    """Elements MLA caches per token: (d_c + d_h^R) per layer ([V2-arch] §2-3)."""
    return (d_latent + d_rope) * layers


def gqa_equivalent_groups(d_latent: int, d_rope: int, d_head: int) -> float:
    """GQA group count whose cache 2*n_g*d_h equals MLA's ([V2-arch] §3, end)."""
    return mla_cache_elems(d_latent, d_rope) / (2.0 * d_head)


# ---------------------------------------------------------------------------
# Decoupled RoPE ([V2-arch] ch.2 §3; [DS-report] "RoPE 的兼容性处理")
# ---------------------------------------------------------------------------
def rope(x: np.ndarray, pos, base: float = 10000.0) -> np.ndarray:
    """Rotate the last axis of ``x`` (even length d_R) to position ``pos``.

    ``pos`` is a scalar or an integer array broadcastable to x[..., 0].
    Pair j = (x[2j], x[2j+1]) turns by pos * base**(-2j/d_R).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    assert d % 2 == 0
    j = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * j / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (d,)))
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# ---------------------------------------------------------------------------
# Compression and the cached row ([V2-arch] ch.2 §2-3; [DS-report] "MLA 的核心思想")
# ---------------------------------------------------------------------------
def latent_rows(h: np.ndarray, w_dkv: np.ndarray, w_kr: np.ndarray,
                positions, base: float = 10000.0) -> np.ndarray:
    """Cached rows [c^KV_p ; k^R_p] for hidden states ``h`` [N, d].

    c^KV_p = W^DKV h_p ([V2-arch] §2); k^R_p = RoPE_p(W^KR h_p)
    ([DS-report] k_t formula; [V2-arch] §3: one k^R shared by all heads).
    Both parts are cached ([DS-pptc] §3.4, §6 问题二).  Returns [N, d_c+d_R].
    """
    h = np.asarray(h, dtype=np.float64)
    c = h @ np.asarray(w_dkv, dtype=np.float64).T
    kr = rope(h @ np.asarray(w_kr, dtype=np.float64).T, positions, base)
    return np.concatenate([c, kr], axis=1)


def slot_of(block_table: np.ndarray, b: int, pos: int, page_size: int) -> int:
    """Pool row holding token ``pos`` of sequence ``b`` in a paged cache.

    Paged addressing (plain definition): logical page pos // page_size of
    sequence b is physical page block_table[b, pos // page_size]; the token
    is row pos % page_size of that page.
    """
    return int(block_table[b, pos // page_size]) * page_size + pos % page_size


# ---------------------------------------------------------------------------
# Query path ([V2-arch] ch.2 §2, last paragraph: the query gets the same
# low-rank compression, c^Q; [DS-report] "RoPE 的兼容性处理":
# q_t = [W^UQ c_t^Q ; W^QR h_t . RoPE(t)])
# ---------------------------------------------------------------------------
def query_from_hidden(dims, h: np.ndarray, w_dq: np.ndarray, w_uq: np.ndarray,
                      w_qr: np.ndarray) -> np.ndarray:
    """Decode queries [N, n_h, d_nope + d_R] of hidden states ``h`` [N, d].

    c^Q = W^DQ h (reading: the query's down-projection, in the form of
    c^KV = W^DKV h; its width d_c' is not on the pages and is a parameter);
    q^C = W^UQ c^Q, head i owning rows i*d_nope..; q^R = W^QR h as the
    report writes it (input h, not c^Q), head i owning rows i*d_R...  The
    rotation of q^R is left to the decode, which applies it at the query's
    position, so the result has the layout of the decode's ``q`` input.
    Matrices act on column vectors: W^DQ [d_c', d], W^UQ [n_h*d_nope, d_c'],
    W^QR [n_h*d_R, d].
    """
    h = np.asarray(h, dtype=np.float64)
    H, dn, dr = dims.n_heads, dims.d_nope, dims.d_rope
    c_q = h @ np.asarray(w_dq, dtype=np.float64).T
    q_c = (c_q @ np.asarray(w_uq, dtype=np.float64).T).reshape(-1, H, dn)
    q_r = (h @ np.asarray(w_qr, dtype=np.float64).T).reshape(-1, H, dr)
    return np.concatenate([q_c, q_r], axis=2)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def _softmax(s: np.ndarray) -> np.ndarray:
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def decode_explicit(dims, rows: np.ndarray, q: np.ndarray, w: dict,
                    T: int, return_attn: bool = False) -> dict:
    """The pages' explicit (non-absorbed) decode of the last T tokens.

    ``rows`` [S, d_c+d_R] are the cached rows of positions 0..S-1 (the T new
    tokens included); ``q`` [T, n_h, d_nope+d_R] holds the un-rotated
    queries; query t sits at position S-T+t.  Per head i ([V2-arch] §1-3):
      k^C_{p,i} = W^UK_i c_p, v_{p,i} = W^UV_i c_p           (§2)
      q_i = [q^C_i ; RoPE_s(q^R_i)], k_{p,i} = [k^C_{p,i} ; k^R_p]   (§3)
      a_{i,p} = softmax_p(q_i . k_{p,i} * scale), o_i = sum_p a v   (§1)
      u = W_O [o_1; ...; o_{n_h}]                               (§1, output)
    K and V are materialised head by head.  Returns u [T, d], o [T, n_h, d_v]
    and, if asked, the attention weights a [T, n_h, S] (zero where masked).
    """
    dc, dr, dn, dv, H = dims.d_latent, dims.d_rope, dims.d_nope, dims.d_v, dims.n_heads
    rows = np.asarray(rows, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    S = rows.shape[0]
    c, kr = rows[:, :dc], rows[:, dc:]
    w_uk = np.asarray(w["w_uk"], dtype=np.float64)
    w_uv = np.asarray(w["w_uv"], dtype=np.float64)
    w_o = np.asarray(w["w_o"], dtype=np.float64)
    scale = dims.softmax_scale
    o = np.zeros((T, H, dv))
    attn = np.zeros((T, H, S)) if return_attn else None
    for i in range(H):
        k_c = c @ w_uk[i * dn:(i + 1) * dn].T          # [S, d_nope]
        v = c @ w_uv[i * dv:(i + 1) * dv].T            # [S, d_v]
        k = np.concatenate([k_c, kr], axis=1)          # [S, d_nope + d_R]
        for t in range(T):
            s_pos = S - T + t
            q_i = np.concatenate([q[t, i, :dn], rope(q[t, i, dn:], s_pos, dims.rope_base)])
            a = _softmax((k[:s_pos + 1] @ q_i) * scale)
            o[t, i] = a @ v[:s_pos + 1]
            if return_attn:
                attn[t, i, :s_pos + 1] = a
    u = o.reshape(T, H * dv) @ w_o.T
    out = {"u": u, "o": o}
    if return_attn:
        out["attn"] = attn
    return out


def decode_absorbed(dims, rows: np.ndarray, q: np.ndarray, w: dict, T: int) -> dict:
    """The same decode with W^UK folded into the query and W^UV applied after.

    Exact rewrite of ``decode_explicit`` by associativity ([V2-arch] §2, the
    absorption paragraph): q_i . W^UK_i c_p = (W^UK_i^T q_i) . c_p and
    sum_p a W^UV_i c_p = W^UV_i (sum_p a c_p).  Used where materialising K/V
    per head is too slow (long caches).  Returns u, o and the latent
    attention output o_lat [T, n_h, d_c] (= sum_p a c_p).
    """
    dc, dn, dv, H = dims.d_latent, dims.d_nope, dims.d_v, dims.n_heads
    rows = np.asarray(rows, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    S = rows.shape[0]
    c, kr = rows[:, :dc], rows[:, dc:]
    w_uk = np.asarray(w["w_uk"], dtype=np.float64).reshape(H, dn, dc)
    w_uv = np.asarray(w["w_uv"], dtype=np.float64).reshape(H, dv, dc)
    w_o = np.asarray(w["w_o"], dtype=np.float64)
    scale = dims.softmax_scale
    o_lat = np.zeros((T, H, dc))
    for t in range(T):
        s_pos = S - T + t
        q_abs = np.einsum("hkc,hk->hc", w_uk, q[t, :, :dn])          # [H, d_c]
        q_rot = rope(q[t, :, dn:], s_pos, dims.rope_base)             # [H, d_R]
        s = (q_abs @ c[:s_pos + 1].T + q_rot @ kr[:s_pos + 1].T) * scale
        a = _softmax(s)
        o_lat[t] = a @ c[:s_pos + 1]
    o = np.einsum("hvc,thc->thv", w_uv, o_lat)
    u = o.reshape(T, H * dv) @ w_o.T
    return {"u": u, "o": o, "o_lat": o_lat}


def decode_layers(dims, layers: list, h_new: np.ndarray, T: int, base: float | None = None,
                  form: str = "explicit") -> dict:
    """A decode step through a stack of MLA attention layers.

    The pages count the cache over all l layers of the model ([V2-arch] ch.2
    §2: (d_c + d_h^R) x l elements per token); each layer has its own weights
    and its own cache.  Reading (the pages give no block structure beyond
    attention and the MoE FFN, which is out of scope, and no normalisation):
    layer j + 1 takes h_{j+1} = h_j + u_j, the residual connection of a
    transformer block around the attention output.  ``layers[j]`` holds
    "w" (the eight matrices of ``query_from_hidden`` and the decode) and
    "prefix_rows" (layer j's cached rows of positions 0..S-T-1).  ``h_new``
    [T, d] are layer 0's hidden states of the T new tokens at positions
    S-T..S-1.  Each layer appends the rows of its own input h_j, makes the
    queries of its own input and decodes them.  Returns h_L [T, d] and the
    per-layer outputs u [L, T, d].
    """
    base = dims.rope_base if base is None else base
    h = np.asarray(h_new, dtype=np.float64)
    us = []
    for layer in layers:
        w = layer["w"]
        prefix = np.asarray(layer["prefix_rows"], dtype=np.float64)
        S = prefix.shape[0] + T
        new_rows = latent_rows(h, w["w_dkv"], w["w_kr"], np.arange(S - T, S), base)
        rows = np.concatenate([prefix, new_rows])
        q = query_from_hidden(dims, h, w["w_dq"], w["w_uq"], w["w_qr"])
        fn = decode_explicit if form == "explicit" else decode_absorbed
        u = fn(dims, rows, q, w, T)["u"]
        us.append(u)
        h = h + u
    return {"h": h, "u": np.stack(us)}


def attention_weights_absorbed(dims, rows, q, w, T, t, head) -> np.ndarray:
    """Softmax weights of one (query token, head) in the absorbed form."""
    dc, dn = dims.d_latent, dims.d_nope
    rows = np.asarray(rows, dtype=np.float64)
    S = rows.shape[0]
    s_pos = S - T + t
    w_uk = np.asarray(w["w_uk"], dtype=np.float64)[head * dn:(head + 1) * dn]
    q = np.asarray(q, dtype=np.float64)
    q_abs = w_uk.T @ q[t, head, :dn]
    q_rot = rope(q[t, head, dn:], s_pos, dims.rope_base)
    s = (rows[:s_pos + 1, :dc] @ q_abs + rows[:s_pos + 1, dc:] @ q_rot) * dims.softmax_scale
    return _softmax(s)


# ---------------------------------------------------------------------------
# Error measures used by every parity test (tolerances are the tests')
# ---------------------------------------------------------------------------
def error_stats(got: np.ndarray, ref: np.ndarray) -> dict:
    """max|err| / max|ref| and sum|err| / sum|ref| (mean relative error)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    return {
        "max_rel": float(err.max() / max(np.abs(ref).max(), 1e-300)),
        "mean_rel": float(err.sum() / max(np.abs(ref).sum(), 1e-300)),
    }
