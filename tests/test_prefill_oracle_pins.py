"""Pins of the oracle's prefill functions (rebuilt per-head keys and values).

Each pin ties oracle.rebuild_kv / oracle.prefill_attention to something
other than themselves:
  * the pages' identity: attention over rebuilt keys and values equals the
    absorbed latent-space attention followed by W^UV_h ("Multi-head latent
    attention (MLA)", section 2; "Attention, Part 2: MQA, GQA and MLA", the
    absorbed inference path), with the latent path pinned on its own by the
    decode pins;
  * torch's scaled_dot_product_attention in float64 with an explicit mask;
  * brute force on tiny inputs and special cases (constant values, a zero
    query, keys past the query's position that must not matter).
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc


def _case(seed, L, T, H, d_h, d_c, d_r):
    rng = np.random.default_rng(seed)
    C = rng.standard_normal((L, d_c + d_r))
    W_uk = rng.standard_normal((H * d_h, d_c)) / math.sqrt(d_c)
    W_uv = rng.standard_normal((H * d_h, d_c)) / math.sqrt(d_c)
    q_nope = rng.standard_normal((T, H, d_h))
    q_rope = rng.standard_normal((T, H, d_r))
    pos = np.arange(L - T, L)
    return C, W_uk, W_uv, q_nope, q_rope, pos


@pytest.mark.parametrize("L,T,H,d_h,d_c,d_r", [
    (20, 5, 3, 8, 16, 4), (7, 7, 2, 4, 6, 2), (33, 1, 4, 16, 24, 8), (64, 17, 1, 8, 8, 6)])
def test_prefill_equals_absorbed_latent_path(L, T, H, d_h, d_c, d_r):
    C, W_uk, W_uv, q_nope, q_rope, pos = _case(L * 7 + T, L, T, H, d_h, d_c, d_r)
    scale, base = 1 / math.sqrt(d_h + d_r), 10000.0
    k, v, kr = orc.rebuild_kv(C, H, W_uk, W_uv, d_c)
    o, lse = orc.prefill_attention(q_nope, q_rope, pos, k, v, kr, scale, base)
    q_lat = orc.absorb_query(q_nope, q_rope, pos, W_uk, base)
    o_lat, lse_lat = orc.decode_attention(q_lat, C, d_c, scale, causal=True)
    o_abs = np.einsum("thc,hdc->thd", o_lat, W_uv.reshape(H, d_h, d_c))
    np.testing.assert_allclose(o, o_abs, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_lat, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L,T,H", [(40, 9, 3), (5, 5, 2)])
def test_prefill_matches_torch_sdpa(L, T, H):
    d_h, d_c, d_r = 8, 12, 4
    C, W_uk, W_uv, q_nope, q_rope, pos = _case(L + 100 * T, L, T, H, d_h, d_c, d_r)
    scale, base = 0.3, 500.0
    k, v, kr = orc.rebuild_kv(C, H, W_uk, W_uv, d_c)
    o, _ = orc.prefill_attention(q_nope, q_rope, pos, k, v, kr, scale, base)
    q_rot = orc.rope(q_rope.transpose(1, 0, 2), pos, base).transpose(1, 0, 2)
    q = torch.from_numpy(np.concatenate([q_nope, q_rot], -1)).permute(1, 0, 2)      # [H, T, 12]
    kk = torch.from_numpy(np.concatenate([k, np.broadcast_to(kr[:, None, :], (L, H, d_r))], -1))
    mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])                   # [T, L]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, kk.permute(1, 0, 2), torch.from_numpy(v).permute(1, 0, 2), attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_rebuild_kv_brute_force():
    rng = np.random.default_rng(5)
    L, H, d_h, d_c, d_r = 3, 2, 3, 4, 2
    C = rng.standard_normal((L, d_c + d_r))
    W_uk = rng.standard_normal((H * d_h, d_c))
    W_uv = rng.standard_normal((H * d_h, d_c))
    k, v, kr = orc.rebuild_kv(C, H, W_uk, W_uv, d_c)
    for s in range(L):
        for h in range(H):
            for i in range(d_h):
                row = h * d_h + i
                assert k[s, h, i] == pytest.approx(sum(W_uk[row, j] * C[s, j] for j in range(d_c)), abs=1e-12)
                assert v[s, h, i] == pytest.approx(sum(W_uv[row, j] * C[s, j] for j in range(d_c)), abs=1e-12)
        assert np.array_equal(kr[s], C[s, d_c:])


def test_prefill_special_cases():
    L, T, H, d_h, d_r = 12, 4, 2, 4, 2
    rng = np.random.default_rng(9)
    k = rng.standard_normal((L, H, d_h))
    kr = rng.standard_normal((L, d_r))
    pos = np.arange(L - T, L)
    # constant values: the output is that constant whatever the weights
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25, 3.0]), (L, H, d_h)).copy()
    o, _ = orc.prefill_attention(rng.standard_normal((T, H, d_h)), rng.standard_normal((T, H, d_r)),
                                 pos, k, v, kr, 0.7, 10000.0)
    np.testing.assert_allclose(o, np.broadcast_to(v[0], o.shape), rtol=1e-14)
    # a zero query: uniform weights over the visible keys, lse = log(count)
    v = rng.standard_normal((L, H, d_h))
    o, lse = orc.prefill_attention(np.zeros((T, H, d_h)), np.zeros((T, H, d_r)), pos, k, v, kr,
                                   0.7, 10000.0)
    for i, p in enumerate(pos):
        np.testing.assert_allclose(o[i], v[:p + 1].mean(axis=0), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[i], math.log(p + 1), rtol=1e-14)
    # keys and values past a query's position do not change its output
    q_n, q_r = rng.standard_normal((T, H, d_h)), rng.standard_normal((T, H, d_r))
    o1, l1 = orc.prefill_attention(q_n, q_r, pos, k, v, kr, 0.7, 10000.0)
    k2, v2, kr2 = k.copy(), v.copy(), kr.copy()
    k2[pos[0] + 1:] *= 5.0
    v2[pos[0] + 1:] = 1e6
    kr2[pos[0] + 1:] = -3.0
    o2, l2 = orc.prefill_attention(q_n[:1], q_r[:1], pos[:1], k2, v2, kr2, 0.7, 10000.0)
    np.testing.assert_array_equal(o2[0], o1[0])
    np.testing.assert_array_equal(l2[0], l1[0])


def test_prefill_inputs_are_seeded_and_laid_out():
    import mla_inputs as mi
    spec = mi.PrefillSpec("layout", seed=21, B=3, H=2, T_q=5, seqlens=(5, 70, 129), d_h=16,
                          d_c=32, d_r=8)
    a = mi.make_prefill_inputs(spec, with_kv=True)
    b = mi.make_prefill_inputs(spec, with_kv=True)
    for x, y in ((a.q_nope_bits, b.q_nope_bits), (a.w_uv_bits, b.w_uv_bits),
                 (a.k_nope_bits, b.k_nope_bits), (a.cache.pool_bits, b.cache.pool_bits)):
        assert np.array_equal(x, y)                       # same seed, same bits
    R = mi.prefill_kv_rows(a.cache.max_blocks)
    assert R % 128 == 0 and R >= 64 * a.cache.max_blocks
    assert a.q_nope_bits.shape == (3, 5, 2, 16) and a.q_rope_bits.shape == (3, 5, 2, 8)
    assert a.w_uk_bits.shape == (2 * 16, 32)
    assert a.k_nope_bits.shape == (3, 2, R, 16) and a.k_rope_bits.shape == (3, R, 8)
    for bi, L in enumerate(spec.seqlens):
        assert not np.any(a.k_nope_bits[bi, :, L:]) and not np.any(a.v_bits[bi, :, L:])
        assert not np.any(a.k_rope_bits[bi, L:]) and np.any(a.k_nope_bits[bi, :, :L])
        # the paged pool holds exactly the logical rows of each sequence
        rows = a.cache.seq_rows(bi)
        for s in (0, L - 1):
            blk = a.cache.block_table[bi, s // 64]
            assert np.array_equal(a.cache.pool_bits[blk, s % 64], rows[s])
