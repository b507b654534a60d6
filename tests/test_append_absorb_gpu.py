"""Parity of mla_cache_append, mla_absorb_query, mla_absorb_output and the
whole four-call layer (tiny fp32 full-model workload) with the fp64 oracle."""

import numpy as np
import pytest
import torch

import head_latent_attention_28_b300 as mla
import mla_inputs as mi
import oracle as orc
from gpu_util import F32_MAX_ABS, bits_to_device

pytestmark = pytest.mark.gpu


def bf16_ulp(x):
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - 7)


@pytest.mark.parametrize("cache_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("in_dtype", [torch.float32, torch.bfloat16])
def test_cache_append_matches_oracle(cache_dtype, in_dtype):
    rng = np.random.default_rng(40)
    d_c, d_r, B, maxb, nb = 512, 64, 3, 4, 16
    n_new = 37
    bt = rng.permutation(nb)[: B * maxb].reshape(B, maxb).astype(np.int32)
    # distinct (sequence, position) pairs, including both ends of the table
    flat = rng.choice(B * maxb * 64 - 3, n_new - 3, replace=False) + 3
    flat = np.concatenate([[0, 63, maxb * 64 - 1], flat]).astype(np.int64)
    seq_ids = (flat // (maxb * 64)).astype(np.int32)
    positions = (flat % (maxb * 64)).astype(np.int32)
    c = rng.standard_normal((n_new, d_c)).astype(np.float32)
    kr = rng.standard_normal((n_new, d_r)).astype(np.float32)
    if in_dtype == torch.bfloat16:
        c = mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(c)).reshape(c.shape)
        kr = mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(kr)).reshape(kr.shape)
    cache = torch.full((nb, 64, d_c + d_r), float("nan"), dtype=cache_dtype, device="cuda")
    mla.mla_cache_append(torch.from_numpy(c).cuda().to(in_dtype),
                         torch.from_numpy(kr).cuda().to(in_dtype),
                         torch.from_numpy(seq_ids).cuda(), torch.from_numpy(positions).cuda(),
                         torch.from_numpy(bt).cuda(), cache, rope_base=10000.0)
    assert mla.mla_check_status() == mla.MLA_OK
    got = cache.double().cpu().numpy()
    want = orc.cache_rows(c, kr, positions, 10000.0)
    for i in range(n_new):
        row = got[bt[seq_ids[i], positions[i] // 64], positions[i] % 64]
        if cache_dtype == torch.float32:
            np.testing.assert_allclose(row, want[i], rtol=0, atol=1e-6)
        else:
            # the latent is only cast: bitwise; the rotated key within one bf16 step
            cb = mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(c[i])).astype(np.float64)
            np.testing.assert_array_equal(row[:d_c], cb)
            assert np.all(np.abs(row[d_c:] - want[i, d_c:]) <= bf16_ulp(want[i, d_c:]))
    # untouched rows keep their contents
    written = {(bt[seq_ids[i], positions[i] // 64], positions[i] % 64) for i in range(n_new)}
    untouched = [(k, r) for k in range(nb) for r in range(64) if (k, r) not in written]
    assert all(np.isnan(got[k, r]).all() for k, r in untouched[:200])


def test_cache_append_bad_position_reports_status():
    cache = torch.zeros((4, 64, 80), device="cuda")
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    c = torch.ones((2, 64), device="cuda")
    kr = torch.ones((2, 16), device="cuda")
    mla.mla_cache_append(c, kr, torch.tensor([0, 5], dtype=torch.int32, device="cuda"),
                         torch.tensor([3, 0], dtype=torch.int32, device="cuda"), bt, cache)
    assert mla.mla_check_status() == mla.MLA_ERR_BAD_INDEX
    assert cache[0, 3, 0].item() == 1.0            # the valid row was written


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_absorb_query_matches_oracle(dtype):
    rng = np.random.default_rng(41)
    N, H, d_h, d_c, d_r = 5, 128, 128, 512, 64
    qn = rng.standard_normal((N, H, d_h)).astype(np.float32)
    qr = rng.standard_normal((N, H, d_r)).astype(np.float32)
    w = (rng.standard_normal((H * d_h, d_c)) / np.sqrt(d_c)).astype(np.float32)
    pos = np.array([0, 1, 4095, 70000, 131071], dtype=np.int32)
    if dtype == torch.bfloat16:
        qn, qr, w = (mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(x)).reshape(x.shape)
                     for x in (qn, qr, w))
    out = mla.mla_absorb_query(torch.from_numpy(qn).cuda().to(dtype),
                               torch.from_numpy(qr).cuda().to(dtype),
                               torch.from_numpy(pos).cuda(),
                               torch.from_numpy(w).cuda().to(dtype), q_dtype=torch.float32)
    torch.cuda.synchronize()
    want = orc.absorb_query(qn, qr, pos, w, 10000.0)
    np.testing.assert_allclose(out.double().cpu().numpy(), want, rtol=0, atol=2e-5)


@pytest.mark.parametrize("d_h", [64, 128])
def test_absorb_query_tensor_core_tiles(d_h):
    """bf16 inputs with d_c = 512 take the tensor-core kernel: 200 tokens are
    two tiles of 128 (the second ragged); bf16 output within one rounding step
    of the fp64 oracle, fp32 output within float accumulation error."""
    rng = np.random.default_rng(44 + d_h)
    N, H, d_c, d_r = 200, 16, 512, 64
    qn, qr = (mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(x)).reshape(x.shape) for x in
              (rng.standard_normal((N, H, d_h)).astype(np.float32),
               rng.standard_normal((N, H, d_r)).astype(np.float32)))
    w = (rng.standard_normal((H * d_h, d_c)) / np.sqrt(d_h)).astype(np.float32)
    w = mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(w)).reshape(w.shape)
    pos = rng.integers(0, 1 << 17, size=N).astype(np.int32)
    args = [torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (qn, qr)]
    want = orc.absorb_query(qn, qr, pos, w, 10000.0)
    out32 = mla.mla_absorb_query(args[0], args[1], torch.from_numpy(pos).cuda(),
                                 torch.from_numpy(w).cuda().to(torch.bfloat16), q_dtype=torch.float32)
    out16 = mla.mla_absorb_query(args[0], args[1], torch.from_numpy(pos).cuda(),
                                 torch.from_numpy(w).cuda().to(torch.bfloat16), q_dtype=torch.bfloat16)
    assert mla.mla_check_status() == mla.MLA_OK
    np.testing.assert_allclose(out32.double().cpu().numpy(), want, rtol=0, atol=2e-5)
    got = out16.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= bf16_ulp(want) + 1e-5)


def test_absorb_query_bf16_output_rounds_once():
    rng = np.random.default_rng(42)
    N, H, d_h, d_c, d_r = 3, 16, 64, 512, 64
    qn = rng.standard_normal((N, H, d_h)).astype(np.float32)
    qr = rng.standard_normal((N, H, d_r)).astype(np.float32)
    w = (rng.standard_normal((H * d_h, d_c)) / 8).astype(np.float32)
    pos = np.array([5, 77, 2048], dtype=np.int32)
    out = mla.mla_absorb_query(torch.from_numpy(qn).cuda(), torch.from_numpy(qr).cuda(),
                               torch.from_numpy(pos).cuda(), torch.from_numpy(w).cuda(),
                               q_dtype=torch.bfloat16)
    want = orc.absorb_query(qn, qr, pos, w, 10000.0)
    got = out.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= bf16_ulp(want) + 1e-5)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_absorb_output_matches_oracle(dtype):
    rng = np.random.default_rng(43)
    N, H, d_h, d_c, d = 4, 128, 128, 512, 5120
    o_lat = rng.standard_normal((N, H, d_c)).astype(np.float32)
    w_uv = (rng.standard_normal((H * d_h, d_c)) / np.sqrt(d_c)).astype(np.float32)
    w_o = (rng.standard_normal((d, H * d_h)) / np.sqrt(H * d_h)).astype(np.float32)
    if dtype == torch.bfloat16:
        w_uv, w_o = (mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(x)).reshape(x.shape)
                     for x in (w_uv, w_o))
    out = mla.mla_absorb_output(torch.from_numpy(o_lat).cuda(),
                                torch.from_numpy(w_uv).cuda().to(dtype),
                                torch.from_numpy(w_o).cuda().to(dtype))
    want = orc.absorb_output(o_lat, w_uv, w_o)
    np.testing.assert_allclose(out.double().cpu().numpy(), want, rtol=0, atol=5e-5)


def test_tiny_full_model_end_to_end_fp32():
    """Four calls in sequence on the tiny fp32 workload (128 cached tokens +
    1 new, d=256, 8 heads): projections by the caller (float32 torch
    matmuls, no TF32), then append -> absorb query -> decode -> absorb
    output; u must match the oracle's UNabsorbed layer to 1e-4."""
    torch.backends.cuda.matmul.allow_tf32 = False
    spec = mi.TINY_FULL_MODEL
    inp = mi.make_full_model_inputs(spec)
    dev = "cuda"
    T = lambda x: torch.from_numpy(x).to(dev)
    h = T(inp.h)
    c = h @ T(inp.W_dkv).T
    kr_raw = h @ T(inp.W_kr).T
    n = spec.n_tokens
    # paged float32 cache: 3 blocks of a shuffled 8-block pool
    rng = np.random.default_rng(7)
    bt = mi.shuffled_block_table(rng, n, 8)
    cache = torch.full((8, 64, spec.d_c + spec.d_r), float("nan"), device=dev)
    mla.mla_cache_append(c.contiguous(), kr_raw.contiguous(),
                         torch.zeros(n, dtype=torch.int32, device=dev),
                         torch.arange(n, dtype=torch.int32, device=dev), T(bt), cache,
                         rope_base=spec.rope_base)
    qs = slice(spec.n_cached, n)
    q_nope = (h[qs] @ T(inp.W_q).T).view(-1, spec.H, spec.d_h).contiguous()
    q_rope = (h[qs] @ T(inp.W_qr).T).view(-1, spec.H, spec.d_r).contiguous()
    pos = torch.arange(spec.n_cached, n, dtype=torch.int32, device=dev)
    q_lat = mla.mla_absorb_query(q_nope, q_rope, pos, T(inp.W_uk), rope_base=spec.rope_base)
    o_lat, _ = mla.mla_decode_paged(q_lat.view(1, spec.n_query, spec.H, -1).contiguous(), cache,
                                    T(bt), torch.tensor([n], dtype=torch.int32, device=dev),
                                    d_c=spec.d_c, softmax_scale=spec.softmax_scale, causal=True)
    u = mla.mla_absorb_output(o_lat.view(spec.n_query, spec.H, spec.d_c).contiguous(),
                              T(inp.W_uv), T(inp.W_o))
    assert mla.mla_check_status() == mla.MLA_OK
    want, _ = orc.full_model_unabsorbed(inp)
    err = np.abs(u.double().cpu().numpy() - want).max()
    assert err <= F32_MAX_ABS, err
    # and the intermediate latent output against the absorbed oracle
    _, mid = orc.full_model_absorbed(inp)
    assert np.abs(o_lat.double().cpu().numpy()[0] - mid["o_lat"]).max() <= F32_MAX_ABS
