"""Plain fp64 restatement of MLA decode (test infrastructure only).

Notation follows the pages: d model width, n_h = H heads, d_h head size,
d_c latent size, d_r = d^R_h decoupled rotary size, D = d_c + d_r cached
numbers per token.  A cached row is [c_s ; R_s k^R_s].

Readings where the pages are silent (each stated once, here):
  * RoPE (equation stripped on the pages; "Why position needs its own key"
    describes rotating each pair (x1, x2) by the angle m*theta with theta
    different per pair, citing RoFormer): adjacent pairs (x[2i], x[2i+1]),
    theta_i = base^(-2i/d_r), (x1, x2) -> (x1 cos - x2 sin, x1 sin + x2 cos),
    positions counted from 0.
  * Query t of a T_q-token step sits at position L - T_q + t, where L counts
    every cached row including the new ones; with the causal mask it sees
    keys 0..L-T_q+t (a token attends to itself and to earlier tokens).
  * Query compression is left out: q^C = W^Q h and q^R = W^QR h directly.
  * d_v = d_h.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "rope", "cache_rows", "project_queries", "absorb_query", "decode_attention",
    "decode_paged_logical", "absorb_output", "full_model_unabsorbed",
    "full_model_absorbed", "full_model_rope_on_reconstructed_keys",
    "mha_cache_numbers", "gqa_cache_numbers", "mla_cache_numbers",
    "mla_equivalent_gqa_groups", "bf16_to_f64", "rebuild_kv", "prefill_attention",
    "merge_output_weights", "absorb_output_merged",
]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns, as float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# rotary position embedding ("Why position needs its own key")
# --------------------------------------------------------------------------

def rope(x: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotate every adjacent pair of the last axis by position * theta_i.

    x: [..., n, d_r] with the token axis second to last; positions: [n]."""
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    assert d_r % 2 == 0
    i = np.arange(d_r // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / d_r)                           # [d_r/2]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    cos, sin = np.cos(ang), np.sin(ang)                        # [n, d_r/2]
    x1 = x[..., 0::2]
    x2 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * cos - x2 * sin
    out[..., 1::2] = x1 * sin + x2 * cos
    return out


# --------------------------------------------------------------------------
# the cache and the queries ("The MLA equations"; section 2 and 3)
# --------------------------------------------------------------------------

def cache_rows(c: np.ndarray, k_rope_raw: np.ndarray, positions: np.ndarray,
               base: float) -> np.ndarray:
    """Cached row of each token: [c_s ; R_s k^R_s]  ([n, d_c + d_r]).

    c = W^DKV h and k_rope_raw = W^KR h are computed by the caller; only the
    rotary part is rotated, the latent never is."""
    c = np.asarray(c, dtype=np.float64)
    kr = rope(k_rope_raw, positions, base)
    return np.concatenate([c, kr], axis=-1)


def project_queries(h, W_q, W_qr, H, d_h, d_r, positions, base):
    """q^C_h = (W^Q h)[h] and rotated q^R_h = R_t (W^QR h)[h]."""
    h = np.asarray(h, dtype=np.float64)
    n = h.shape[0]
    q_nope = (h @ np.asarray(W_q, np.float64).T).reshape(n, H, d_h)
    q_rope_raw = (h @ np.asarray(W_qr, np.float64).T).reshape(n, H, d_r)
    # rotate per head: move the head axis in front of the token axis
    q_rope = rope(q_rope_raw.transpose(1, 0, 2), positions, base).transpose(1, 0, 2)
    return q_nope, q_rope_raw, q_rope


def absorb_query(q_nope, q_rope_raw, positions, W_uk, base):
    """q_lat[n, h] = [W^UK_h^T q^C_h ; R_t q^R_h]   ([n, H, d_c + d_r]).

    W^UK is [H*d_h, d_c]; head h owns rows h*d_h .. (h+1)*d_h - 1."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    n, H, d_h = q_nope.shape
    W = np.asarray(W_uk, dtype=np.float64).reshape(H, d_h, -1)   # [H, d_h, d_c]
    q_c = np.stack([q_nope[:, hh, :] @ W[hh] for hh in range(H)], axis=1)   # [n, H, d_c]
    q_r = rope(np.asarray(q_rope_raw, np.float64).transpose(1, 0, 2),
               positions, base).transpose(1, 0, 2)
    return np.concatenate([q_c, q_r], axis=-1)


# --------------------------------------------------------------------------
# attention in latent space (the hot path)
# --------------------------------------------------------------------------

def decode_attention(q: np.ndarray, C: np.ndarray, d_c: int, scale: float,
                     causal: bool):
    """Latent-space softmax attention of one sequence.

    q: [T_q, H, D] latent queries (position L - T_q + t); C: [L, D] cached
    rows.  score_s = scale * q . C_s (content plus rotary term in one dot);
    p = softmax over the visible keys; o = sum_s p_s C_s[0:d_c] (the value is
    the first d_c numbers of the row).  Returns o [T_q, H, d_c] and the
    natural-log log-sum-exp of the scaled scores, lse [T_q, H]."""
    q = np.asarray(q, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    T_q, H, _ = q.shape
    L = C.shape[0]
    o = np.zeros((T_q, H, d_c))
    lse = np.zeros((T_q, H))
    for t in range(T_q):
        n = (L - T_q + t + 1) if causal else L
        z = scale * (q[t] @ C[:n].T)                 # [H, n]
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        s = e.sum(axis=1, keepdims=True)
        p = e / s
        o[t] = p @ C[:n, :d_c]
        lse[t] = m[:, 0] + np.log(s[:, 0])
    return o, lse


def decode_paged_logical(q_bits, cache_bits, offsets, d_c, scale, causal,
                         batch=None):
    """decode_attention for every sequence of a batch, read from the logical
    per-sequence rows (never from the paged pool).  Inputs are bfloat16 bit
    patterns, widened exactly.  Returns o [B, T_q, H, d_c], lse [B, T_q, H]."""
    B, T_q, H, _ = q_bits.shape
    seqs = range(B) if batch is None else batch
    o = np.zeros((B, T_q, H, d_c))
    lse = np.zeros((B, T_q, H))
    for b in seqs:
        C = bf16_to_f64(cache_bits[offsets[b]:offsets[b + 1]])
        o[b], lse[b] = decode_attention(bf16_to_f64(q_bits[b]), C, d_c, scale, causal)
    return o, lse


def absorb_output(o_lat, W_uv, W_o):
    """o_h = W^UV_h o_lat,h, then u = W^O [o_1; ...; o_H]   ([n, d])."""
    o_lat = np.asarray(o_lat, dtype=np.float64)
    n, H, d_c = o_lat.shape
    W = np.asarray(W_uv, dtype=np.float64).reshape(H, -1, d_c)   # [H, d_h, d_c]
    o = np.stack([o_lat[:, hh, :] @ W[hh].T for hh in range(H)], axis=1)    # [n, H, d_h]
    return o.reshape(n, -1) @ np.asarray(W_o, dtype=np.float64).T


# --------------------------------------------------------------------------
# W^UV folded into W^O ("How DeepSeek Rewrote the Transformer", the absorbed
# inference path: the value up-projection merges into the output projection)
# --------------------------------------------------------------------------

def merge_output_weights(W_uv, W_o, H):
    """One d x d_c matrix per head: M_h = W^O_h W^UV_h, where W^O_h is the
    column block of W^O that multiplies head h's values.  Returned side by
    side, [d, H * d_c]."""
    W_uv = np.asarray(W_uv, dtype=np.float64)
    W_o = np.asarray(W_o, dtype=np.float64)
    d_h = W_uv.shape[0] // H
    blocks = [W_o[:, hh * d_h:(hh + 1) * d_h] @ W_uv[hh * d_h:(hh + 1) * d_h] for hh in range(H)]
    return np.concatenate(blocks, axis=1)


def absorb_output_merged(o_lat, W_m):
    """u = sum_h M_h o_lat,h   ([n, d]); W_m = [M_1 ... M_H]."""
    o_lat = np.asarray(o_lat, dtype=np.float64)
    n, H, d_c = o_lat.shape
    return o_lat.reshape(n, H * d_c) @ np.asarray(W_m, dtype=np.float64).T


# --------------------------------------------------------------------------
# prefill over rebuilt per-head keys and values ("The MLA equations": the key
# of head h is [W^UK_h c_s ; R_s k^R_s], its value W^UV_h c_s)
# --------------------------------------------------------------------------

def rebuild_kv(C, H, W_uk, W_uv, d_c):
    """Per-head content keys and values of cached rows C [L, D].

    W^UK and W^UV are [H*d_h, d_c]; head h owns rows h*d_h .. (h+1)*d_h - 1.
    Returns k_nope [L, H, d_h] = W^UK_h c_s, v [L, H, d_h] = W^UV_h c_s and
    k_rope [L, d_r] = R_s k^R_s (the row's rotary part, stored rotated)."""
    C = np.asarray(C, dtype=np.float64)
    L = C.shape[0]
    c = C[:, :d_c]
    k_nope = (c @ np.asarray(W_uk, np.float64).T).reshape(L, H, -1)
    v = (c @ np.asarray(W_uv, np.float64).T).reshape(L, H, -1)
    return k_nope, v, C[:, d_c:].copy()


def prefill_attention(q_nope, q_rope_raw, positions, k_nope, v, k_rope, scale, base):
    """Causal softmax attention of one sequence's new tokens over per-head keys.

    q_nope [T, H, d_h] (content query q^C_h), q_rope_raw [T, H, d_r] (not yet
    rotated; rotated here by the query's position), positions [T];
    k_nope, v [L, H, d_h], k_rope [L, d_r].  Query i sees keys
    0 .. positions[i].  score = scale * ([q^C_h ; R_t q^R_h] . [k_nope ;
    k_rope]); o_h = sum_s p_s v_{s,h}.  Returns o [T, H, d_h] and the
    natural-log log-sum-exp of the scaled scores, lse [T, H]."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    T, H, d_h = q_nope.shape
    q_rope = rope(np.asarray(q_rope_raw, np.float64).transpose(1, 0, 2),
                  positions, base).transpose(1, 0, 2)
    k_nope = np.asarray(k_nope, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    k_rope = np.asarray(k_rope, dtype=np.float64)
    o = np.zeros((T, H, d_h))
    lse = np.zeros((T, H))
    for i in range(T):
        n = int(positions[i]) + 1
        z = scale * (np.einsum("hd,shd->hs", q_nope[i], k_nope[:n]) +
                     q_rope[i] @ k_rope[:n].T)            # [H, n]
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        s = e.sum(axis=1, keepdims=True)
        o[i] = np.einsum("hs,shd->hd", e / s, v[:n])
        lse[i] = m[:, 0] + np.log(s[:, 0])
    return o, lse


# --------------------------------------------------------------------------
# the full layer, two ways (the pages' associativity identity)
# --------------------------------------------------------------------------

def _latents(inp):
    s = inp.spec
    h = np.asarray(inp.h, dtype=np.float64)
    pos = np.arange(s.n_tokens)
    c = h @ np.asarray(inp.W_dkv, np.float64).T               # [n, d_c]
    kr_raw = h @ np.asarray(inp.W_kr, np.float64).T           # [n, d_r]
    return h, pos, c, kr_raw


def full_model_unabsorbed(inp):
    """Rebuild every head's keys and values, then textbook attention.

    k_{s,h} = [W^UK_h c_s ; R_s k^R_s], v_{s,h} = W^UV_h c_s,
    q_h = [q^C_h ; R_t q^R_h], score scaled by 1/sqrt(d_h + d_r), causal mask,
    o_h = sum p v, u = W^O concat_h o_h.  Returns u for the query tokens
    (the last n_query tokens) and the per-head o [n_query, H, d_h]."""
    s = inp.spec
    H, d_h, d_c = s.H, s.d_h, s.d_c
    h, pos, c, kr_raw = _latents(inp)
    kr = rope(kr_raw, pos, s.rope_base)                        # [n, d_r]
    W_uk = np.asarray(inp.W_uk, np.float64).reshape(H, d_h, d_c)
    W_uv = np.asarray(inp.W_uv, np.float64).reshape(H, d_h, d_c)
    k_c = np.stack([c @ W_uk[hh].T for hh in range(H)])      # [H, n, d_h]
    v = np.stack([c @ W_uv[hh].T for hh in range(H)])         # [H, n, d_h]
    q_nope, _, q_rope = project_queries(h, inp.W_q, inp.W_qr, H, d_h, s.d_r,
                                        pos, s.rope_base)
    qs = range(s.n_cached, s.n_tokens)
    o = np.zeros((len(qs), H, d_h))
    for i, t in enumerate(qs):
        for hh in range(H):
            k = np.concatenate([k_c[hh, :t + 1], kr[:t + 1]], axis=1)
            qv = np.concatenate([q_nope[t, hh], q_rope[t, hh]])
            z = (k @ qv) * s.softmax_scale
            e = np.exp(z - z.max())
            o[i, hh] = (e / e.sum()) @ v[hh, :t + 1]
    u = o.reshape(len(qs), H * d_h) @ np.asarray(inp.W_o, np.float64).T
    return u, o


def full_model_absorbed(inp):
    """Cache only [c ; R k^R], absorb W^UK into the query, attend in latent
    space, up-project the latent output once, then W^O.

    Returns u [n_query, d] and a dict of the intermediates."""
    s = inp.spec
    h, pos, c, kr_raw = _latents(inp)
    C = cache_rows(c, kr_raw, pos, s.rope_base)               # [n, D]
    q_nope, q_rope_raw, _ = project_queries(h, inp.W_q, inp.W_qr, s.H, s.d_h,
                                            s.d_r, pos, s.rope_base)
    qs = slice(s.n_cached, s.n_tokens)
    q_lat = absorb_query(q_nope[qs], q_rope_raw[qs], pos[qs], inp.W_uk, s.rope_base)
    o_lat, lse = decode_attention(q_lat, C, s.d_c, s.softmax_scale, causal=True)
    u = absorb_output(o_lat, inp.W_uv, inp.W_o)
    return u, dict(c=c, k_rope_raw=kr_raw, C=C, q_nope=q_nope[qs],
                   q_rope_raw=q_rope_raw[qs], q_lat=q_lat, o_lat=o_lat, lse=lse)


def full_model_rope_on_reconstructed_keys(inp):
    """Negative control ("Why position needs its own key"): rotate the
    rebuilt content keys k_h = W^UK_h c_s and the content query instead of
    keeping rotation in the decoupled key.  Absorption is then no longer an
    identity; tests check that the absorbed path disagrees with this."""
    s = inp.spec
    H, d_h, d_c = s.H, s.d_h, s.d_c
    h, pos, c, kr_raw = _latents(inp)
    kr = rope(kr_raw, pos, s.rope_base)
    W_uk = np.asarray(inp.W_uk, np.float64).reshape(H, d_h, d_c)
    W_uv = np.asarray(inp.W_uv, np.float64).reshape(H, d_h, d_c)
    k_c = rope(np.stack([c @ W_uk[hh].T for hh in range(H)]), pos, s.rope_base)
    v = np.stack([c @ W_uv[hh].T for hh in range(H)])
    q_nope, _, q_rope = project_queries(h, inp.W_q, inp.W_qr, H, d_h, s.d_r,
                                        pos, s.rope_base)
    q_nope_rot = rope(q_nope.transpose(1, 0, 2), pos, s.rope_base).transpose(1, 0, 2)
    qs = range(s.n_cached, s.n_tokens)
    o = np.zeros((len(qs), H, d_h))
    for i, t in enumerate(qs):
        for hh in range(H):
            k = np.concatenate([k_c[hh, :t + 1], kr[:t + 1]], axis=1)
            qv = np.concatenate([q_nope_rot[t, hh], q_rope[t, hh]])
            z = (k @ qv) * s.softmax_scale
            e = np.exp(z - z.max())
            o[i, hh] = (e / e.sum()) @ v[hh, :t + 1]
    return o.reshape(len(qs), H * d_h) @ np.asarray(inp.W_o, np.float64).T


# --------------------------------------------------------------------------
# cache sizes (section 4 and Exercise 1; "How big is the difference?")
# --------------------------------------------------------------------------

def mha_cache_numbers(n_heads: int, d_k: int, d_v: int | None = None) -> int:
    """Numbers cached per token per layer by multi-head attention: every
    head keeps one key and one value."""
    return n_heads * (d_k + (d_k if d_v is None else d_v))


def gqa_cache_numbers(n_kv_groups: int, d_h: int) -> int:
    """Grouped-query attention: one key and one value per KV group."""
    return 2 * n_kv_groups * d_h


def mla_cache_numbers(d_c: int, d_r: int) -> int:
    """MLA: the latent plus the decoupled rotary key, shared by all heads."""
    return d_c + d_r


def mla_equivalent_gqa_groups(d_c: float, d_r: float, d_h: float) -> float:
    """Groups n_g at which GQA caches as much as MLA: 2 n_g d_h = d_c + d_r."""
    return (d_c + d_r) / (2.0 * d_h)
