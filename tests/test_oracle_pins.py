"""Pins of the fp64 oracle against things other than itself.

Each test ties an oracle function to a figure printed on the pages, a
library routine, a brute-force loop, or a closed form / invariant, chosen so
that a dropped term, a wrong sign or index, or a transposed operand fails at
least one of them.  CPU only.
"""

import math
import os

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cache_figures.txt")


def golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, value = line.split()[:2]
            out[name] = float(value)
    return out


# --------------------------------------------------------------------------
# cache-size figures printed on the pages
# --------------------------------------------------------------------------

def test_cache_counts_v2_scale():
    g = golden()
    d, n_h = 5120, 128
    d_h = d // n_h
    mha = orc.mha_cache_numbers(n_h, d_h)
    gqa = orc.gqa_cache_numbers(8, d_h)
    mla = orc.mla_cache_numbers(512, 64)
    assert (mha, gqa, mla) == (g["mha_numbers_v2"], g["gqa_numbers_v2"], g["mla_numbers_v2"])
    assert round(mha / mla, 1) == g["mla_vs_mha_factor"]
    assert mha / gqa == g["gqa_vs_mha_factor"]


def test_cache_counts_small_example_is_tiny_workload_shape():
    # the proof's small example: full K (content + rotary) and V per head
    g = golden()
    s = mi.TINY_FULL_MODEL
    full = orc.mha_cache_numbers(s.H, s.d_h + s.d_r, s.d_h)
    lat = orc.mla_cache_numbers(s.d_c, s.d_r)
    assert full == g["small_full_kv"] and lat == g["small_latent_rope"]
    assert round(full / lat, 1) == g["small_factor"]


def test_cache_counts_deepseek_v3():
    g = golden()
    layers, heads, bytes_per = 61, 128, 2
    per_tok = layers * orc.mla_cache_numbers(512, 64) * bytes_per
    assert per_tok == g["v3_bytes_per_token"]
    assert round(per_tok / 1024, 1) == g["v3_kib_per_token"]
    mha = layers * orc.mha_cache_numbers(heads, 128 + 64, 128) * bytes_per
    assert mha / 1024 == g["v3_mha_kib_per_token"]
    assert round(mha / per_tok) == g["v3_mha_factor_approx"]
    video = layers * orc.mha_cache_numbers(heads, 128) * bytes_per
    assert video == g["v3_video_mha_count"]
    assert round(video / per_tok, 1) == g["v3_video_factor"]


def test_gqa_equivalent_groups():
    g = golden()
    d_h = 128.0
    assert orc.mla_equivalent_gqa_groups(4 * d_h, d_h / 2, d_h) == g["gqa_equiv_groups"]


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_matches_complex_rotation():
    # RoFormer's complex form: pair (x0, x1) as x0 + i x1, times e^{i m theta_j}
    rng = np.random.default_rng(11)
    d_r, base = 16, 10000.0
    x = rng.standard_normal((7, d_r))
    pos = np.array([0, 1, 2, 5, 63, 128, 131071])
    z = x[:, 0::2] + 1j * x[:, 1::2]
    j = np.arange(d_r // 2)
    w = np.exp(1j * np.outer(pos, np.power(base, -2.0 * j / d_r)))
    zr = z * w
    got = orc.rope(x, pos, base)
    np.testing.assert_allclose(got[:, 0::2], zr.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[:, 1::2], zr.imag, rtol=0, atol=1e-12)


def test_rope_identity_norm_and_first_pair():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((5, 64))
    np.testing.assert_array_equal(orc.rope(x, np.zeros(5), 10000.0), x)   # R_0 = I
    pos = np.arange(5) * 997
    y = orc.rope(x, pos, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1),
                               rtol=1e-13)
    # the first pair turns by exactly m radians (theta_0 = 1), anticlockwise
    e = np.zeros((1, 64)); e[0, 0] = 1.0
    r = orc.rope(e, np.array([1.0]), 10000.0)
    assert abs(r[0, 0] - math.cos(1.0)) < 1e-15 and abs(r[0, 1] - math.sin(1.0)) < 1e-15


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(13)
    q, k = rng.standard_normal((2, 1, 64))
    base = 10000.0
    ref = (orc.rope(q, [7], base) @ orc.rope(k, [3], base).T).item()
    for m, n in [(4, 0), (104, 100), (5004, 5000)]:
        v = (orc.rope(q, [m], base) @ orc.rope(k, [n], base).T).item()
        assert abs(v - ref) < 1e-9


# --------------------------------------------------------------------------
# latent-space decode attention
# --------------------------------------------------------------------------

def brute_force_decode(q, C, d_c, scale, causal):
    """Pure-Python loops: the textbook definition, element by element."""
    T_q, H, D = len(q), len(q[0]), len(q[0][0])
    L = len(C)
    o = [[[0.0] * d_c for _ in range(H)] for _ in range(T_q)]
    lse = [[0.0] * H for _ in range(T_q)]
    for t in range(T_q):
        last = L - T_q + t if causal else L - 1
        for h in range(H):
            z = []
            for s in range(last + 1):
                acc = 0.0
                for k in range(D):
                    acc += q[t][h][k] * C[s][k]
                z.append(acc * scale)
            m = max(z)
            w = [math.exp(v - m) for v in z]
            tot = sum(w)
            for j in range(d_c):
                o[t][h][j] = sum(w[s] * C[s][j] for s in range(last + 1)) / tot
            lse[t][h] = m + math.log(tot)
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("T_q,H,L,d_c,d_r,causal", [
    (1, 1, 1, 4, 2, False), (1, 3, 9, 8, 4, False), (2, 2, 7, 10, 2, True),
    (3, 2, 5, 6, 6, True), (1, 2, 9, 12, 0, False)])
def test_decode_matches_brute_force(T_q, H, L, d_c, d_r, causal):
    rng = np.random.default_rng(100 + L)
    D = d_c + d_r
    q = rng.standard_normal((T_q, H, D))
    C = rng.standard_normal((L, D))
    scale = 1.0 / math.sqrt(D)
    o, lse = orc.decode_attention(q, C, d_c, scale, causal)
    ob, lb = brute_force_decode(q.tolist(), C.tolist(), d_c, scale, causal)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


@pytest.mark.parametrize("T_q,H,L,causal", [(1, 128, 300, False), (2, 16, 129, True),
                                            (4, 8, 64, True)])
def test_decode_matches_torch_sdpa(T_q, H, L, causal):
    """A single shared key/value head: keys are the whole 576-wide rows and
    values their first 512 numbers, so this is library attention."""
    rng = np.random.default_rng(200 + L)
    d_c, d_r = 512, 64
    q = rng.standard_normal((T_q, H, d_c + d_r))
    C = rng.standard_normal((L, d_c + d_r))
    scale = 1.0 / math.sqrt(192.0)
    o, _ = orc.decode_attention(q, C, d_c, scale, causal)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]                  # [1,H,T_q,D]
    tk = torch.from_numpy(C)[None, None].expand(1, H, L, d_c + d_r)
    tv = torch.from_numpy(C[:, :d_c])[None, None].expand(1, H, L, d_c)
    mask = None
    if causal:
        t = torch.arange(T_q)[:, None]
        s = torch.arange(L)[None, :]
        mask = s <= (L - T_q + t)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                           scale=scale)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-13)


def test_decode_single_row_returns_that_row():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 20))
    C = rng.standard_normal((1, 20))
    o, lse = orc.decode_attention(q, C, 16, 0.3, False)
    np.testing.assert_array_equal(o[0], np.broadcast_to(C[0, :16], (4, 16)))
    np.testing.assert_allclose(lse[0], 0.3 * (q[0] @ C[0]), rtol=1e-15)


def test_decode_zero_query_averages_rows():
    rng = np.random.default_rng(4)
    C = rng.standard_normal((37, 24))
    o, lse = orc.decode_attention(np.zeros((1, 2, 24)), C, 20, 1.0, False)
    np.testing.assert_allclose(o[0, 0], C[:, :20].mean(axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(37), rtol=1e-15)


def test_decode_shared_rotary_key_shifts_scores_uniformly():
    """Giving every cached row the same rotary part adds one constant to all
    of a head's scores: o is unchanged, lse moves by exactly that constant."""
    rng = np.random.default_rng(5)
    d_c, d_r = 16, 8
    q = rng.standard_normal((1, 3, d_c + d_r))
    C = rng.standard_normal((40, d_c + d_r))
    C0 = C.copy(); C0[:, d_c:] = 0.0
    C1 = C.copy(); C1[:, d_c:] = C[0, d_c:]
    o0, l0 = orc.decode_attention(q, C0, d_c, 0.25, False)
    o1, l1 = orc.decode_attention(q, C1, d_c, 0.25, False)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-14)
    np.testing.assert_allclose((l1 - l0)[0], 0.25 * (q[0, :, d_c:] @ C[0, d_c:]), atol=1e-13)


def test_decode_output_in_convex_hull_and_causal_prefix():
    rng = np.random.default_rng(6)
    C = rng.standard_normal((50, 12))
    q = 3.0 * rng.standard_normal((2, 5, 12))
    o, _ = orc.decode_attention(q, C, 8, 1.0, True)
    lo, hi = C[:, :8].min(axis=0), C[:, :8].max(axis=0)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)
    # causal query 0 of 2 sees exactly the first 49 rows
    o49, _ = orc.decode_attention(q[:1], C[:49], 8, 1.0, False)
    np.testing.assert_allclose(o[0], o49[0], rtol=0, atol=1e-15)


def test_paged_logical_reads_each_sequence():
    spec = mi.DecodeSpec("t", seed=9, B=3, H=2, T_q=2, d_c=8, d_r=4,
                         seqlens=(3, 70, 64), causal=True, softmax_scale=0.5)
    inp = mi.make_decode_inputs(spec)
    o, lse = orc.decode_paged_logical(inp.q_bits, inp.cache_bits, inp.offsets,
                                      8, 0.5, True)
    for b in range(3):
        C = orc.bf16_to_f64(inp.seq_rows(b))
        ob, lb = brute_force_decode(orc.bf16_to_f64(inp.q_bits[b]).tolist(),
                                    C.tolist(), 8, 0.5, True)
        np.testing.assert_allclose(o[b], ob, atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse[b], lb, atol=1e-13, rtol=0)


# --------------------------------------------------------------------------
# the full layer: absorbed == unabsorbed (the pages' identity)
# --------------------------------------------------------------------------

def small_spec(**kw):
    base = dict(name="s", seed=21, d=48, H=3, d_h=8, d_c=12, d_r=6, n_cached=20,
                n_query=2)
    base.update(kw)
    return mi.FullModelSpec(**base)


@pytest.mark.parametrize("spec", [mi.TINY_FULL_MODEL, small_spec(),
                                  small_spec(seed=22, H=5, d_h=4, d_c=20, d_r=2,
                                             n_cached=7, n_query=3)],
                         ids=["tiny_full_model", "small_a", "small_b"])
def test_absorbed_equals_unabsorbed(spec):
    g = golden()
    inp = mi.make_full_model_inputs(spec)
    u_full, _ = orc.full_model_unabsorbed(inp)
    u_abs, _ = orc.full_model_absorbed(inp)
    diff = np.abs(u_full - u_abs).max()
    rel = np.linalg.norm(u_full - u_abs) / np.linalg.norm(u_full)
    assert rel < 1e-12
    # same order of rounding noise as the page's fp64 proof
    assert diff < 1e3 * g["absorbed_vs_full_diff"]


def test_unabsorbed_heads_match_library_attention():
    """Rebuilt per-head keys/values through torch's attention with its
    default scale 1/sqrt(query width) = 1/sqrt(d_h + d_r)."""
    spec = small_spec(n_query=3)
    inp = mi.make_full_model_inputs(spec)
    H, d_h, d_c, d_r = spec.H, spec.d_h, spec.d_c, spec.d_r
    n = spec.n_tokens
    h = torch.from_numpy(inp.h.astype(np.float64))
    W = {k: torch.from_numpy(getattr(inp, k).astype(np.float64))
         for k in ("W_dkv", "W_kr", "W_q", "W_qr", "W_uk", "W_uv")}
    pos = np.arange(n)
    c = h @ W["W_dkv"].T
    kr = torch.from_numpy(orc.rope((h @ W["W_kr"].T).numpy(), pos, spec.rope_base))
    kc = (c @ W["W_uk"].T).view(n, H, d_h)
    v = (c @ W["W_uv"].T).view(n, H, d_h)
    qc = (h @ W["W_q"].T).view(n, H, d_h)
    qr = torch.from_numpy(orc.rope((h @ W["W_qr"].T).view(n, H, d_r)
                                   .permute(1, 0, 2).numpy(), pos, spec.rope_base))
    k = torch.cat([kc.permute(1, 0, 2), kr[None].expand(H, n, d_r)], -1)   # [H,n,48]
    q = torch.cat([qc.permute(1, 0, 2), qr], -1)                            # [H,n,48]
    mask = torch.ones(n, n, dtype=torch.bool).tril()
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None],
                                                           v.permute(1, 0, 2)[None],
                                                           attn_mask=mask)[0]
    _, o = orc.full_model_unabsorbed(inp)
    want = ref.permute(1, 0, 2)[spec.n_cached:].numpy()
    np.testing.assert_allclose(o, want, rtol=0, atol=1e-13)


def test_rope_on_reconstructed_keys_breaks_absorption():
    inp = mi.make_full_model_inputs(mi.TINY_FULL_MODEL)
    u_abs, _ = orc.full_model_absorbed(inp)
    u_bad = orc.full_model_rope_on_reconstructed_keys(inp)
    rel = np.linalg.norm(u_bad - u_abs) / np.linalg.norm(u_abs)
    assert rel > 1e-3


def test_folding_identity_per_head():
    """q . (W^UK_h c) == (W^UK_h^T q) . c for every head (section 2, Exercise 3)."""
    rng = np.random.default_rng(31)
    H, d_h, d_c, d_r = 4, 5, 7, 4
    W_uk = rng.standard_normal((H * d_h, d_c))
    q_nope = rng.standard_normal((1, H, d_h))
    q_rope = rng.standard_normal((1, H, d_r))
    c = rng.standard_normal(d_c)
    q_lat = orc.absorb_query(q_nope, q_rope, np.zeros(1), W_uk, 10000.0)
    k = (W_uk @ c).reshape(H, d_h)
    for hh in range(H):
        assert abs(q_lat[0, hh, :d_c] @ c - q_nope[0, hh] @ k[hh]) < 1e-12
        np.testing.assert_array_equal(q_lat[0, hh, d_c:], q_rope[0, hh])  # R_0 = I


def test_absorb_output_against_explicit_values():
    """sum_s p_s (W^UV_h c_s) == W^UV_h (sum_s p_s c_s), then W^O."""
    rng = np.random.default_rng(32)
    H, d_h, d_c, d, L = 3, 4, 6, 10, 9
    W_uv = rng.standard_normal((H * d_h, d_c))
    W_o = rng.standard_normal((d, H * d_h))
    C = rng.standard_normal((L, d_c))
    p = rng.random((H, L)); p /= p.sum(axis=1, keepdims=True)
    o_lat = (p @ C)[None]                                  # [1, H, d_c]
    vals = np.stack([C @ W_uv[hh * d_h:(hh + 1) * d_h].T for hh in range(H)])  # [H,L,d_h]
    o = np.stack([p[hh] @ vals[hh] for hh in range(H)]).reshape(1, -1)
    np.testing.assert_allclose(orc.absorb_output(o_lat, W_uv, W_o), o @ W_o.T,
                               rtol=0, atol=1e-12)


def test_merged_output_equals_the_two_projections():
    """Associativity: W^O [W^UV_h o_h]_h == sum_h (W^O_h W^UV_h) o_h.  The
    merged form multiplies in the other order, so a transposed block or a
    wrong head offset on either side breaks the equality."""
    rng = np.random.default_rng(33)
    H, d_h, d_c, d, n = 5, 3, 7, 11, 4
    W_uv = rng.standard_normal((H * d_h, d_c))
    W_o = rng.standard_normal((d, H * d_h))
    o_lat = rng.standard_normal((n, H, d_c))
    W_m = orc.merge_output_weights(W_uv, W_o, H)
    assert W_m.shape == (d, H * d_c)
    np.testing.assert_allclose(orc.absorb_output_merged(o_lat, W_m), orc.absorb_output(o_lat, W_uv, W_o),
                               rtol=0, atol=1e-12)


def test_merged_weights_special_cases():
    """W^UV_h = [I 0] (the first d_h latents) makes M_h the column block
    W^O_h padded with zeros; a W^O that selects one value coordinate of one
    head makes a row of M equal a row of W^UV."""
    rng = np.random.default_rng(34)
    H, d_h, d_c, d = 3, 2, 5, 4
    W_uv = np.zeros((H * d_h, d_c))
    for hh in range(H):
        W_uv[hh * d_h:(hh + 1) * d_h, :d_h] = np.eye(d_h)
    W_o = rng.standard_normal((d, H * d_h))
    W_m = orc.merge_output_weights(W_uv, W_o, H)
    for hh in range(H):
        np.testing.assert_array_equal(W_m[:, hh * d_c:hh * d_c + d_h], W_o[:, hh * d_h:(hh + 1) * d_h])
        np.testing.assert_array_equal(W_m[:, hh * d_c + d_h:(hh + 1) * d_c], 0.0)
    W_uv = rng.standard_normal((H * d_h, d_c))
    W_o = np.zeros((d, H * d_h))
    W_o[2, 1 * d_h + 1] = 1.0                      # output 2 = value coordinate 1 of head 1
    W_m = orc.merge_output_weights(W_uv, W_o, H)
    np.testing.assert_array_equal(W_m[2, d_c:2 * d_c], W_uv[1 * d_h + 1])
    assert np.count_nonzero(W_m[[0, 1, 3]]) == 0 and np.count_nonzero(W_m[2, :d_c]) == 0


# --------------------------------------------------------------------------
# bfloat16 decoding: fixed bit patterns from the format's definition (1 sign,
# 8 exponent bits with bias 127, 7 fraction bits), and torch's own decoding
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0),                 # exponent 127, fraction 0
    (0xC000, -2.0),                # sign, exponent 128
    (0x3FC0, 1.5),                 # fraction 0b1000000 = 1/2
    (0x4049, 3.140625),            # 2 * (1 + 73/128)
    (0x0001, 2.0 ** -133),         # smallest subnormal: 2^-126 * 2^-7
    (0x0080, 2.0 ** -126),         # smallest normal
    (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127),   # largest finite
    (0x8000, -0.0),
    (0x7F80, math.inf),
    (0xFF80, -math.inf),
])
def test_bf16_to_f64_fixed_patterns(bits, value):
    got = orc.bf16_to_f64(np.array([bits], dtype=np.uint16))
    assert got.dtype == np.float64
    assert got[0] == value
    assert math.copysign(1.0, got[0]) == math.copysign(1.0, value)


def test_bf16_to_f64_nan_and_random_bits_match_torch():
    assert np.isnan(orc.bf16_to_f64(np.array([0x7FC0, 0xFFC1], dtype=np.uint16))).all()
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 16, size=50000, dtype=np.uint16)
    got = orc.bf16_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(want)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(got[~finite & ~np.isnan(want)], want[~finite & ~np.isnan(want)])
