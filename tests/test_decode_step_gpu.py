"""mla_decode_step (absorb the new queries, append the new tokens' rows and
attend, in one call) against the three separate calls, bit for bit, and
against the fp64 oracle of the same chain."""

import math

import numpy as np
import pytest
import torch

import head_latent_attention_28_b300 as mla
import mla_inputs as mi
import oracle as orc
from gpu_util import assert_decode_close, bits_to_device

pytestmark = pytest.mark.gpu

CASES = [
    # tensor-core decode and absorption
    (mi.DecodeSpec("step_h128", seed=50, B=3, H=128, seqlens=(70, 300, 129)), 128),
    (mi.DecodeSpec("step_h16_tq2", seed=51, B=3, H=16, T_q=2, causal=True,
                   seqlens=(2, 200, 65), softmax_scale=1 / math.sqrt(192)), 64),
    # multi-token step with 256 query rows per sequence: two row groups
    (mi.DecodeSpec("step_h128_tq2_row_groups", seed=53, B=2, H=128, T_q=2, causal=True,
                   seqlens=(2, 333)), 128),
    # CUDA-core decode and plain absorption
    (mi.DecodeSpec("step_small_dims", seed=52, B=2, H=8, d_c=64, d_r=16, seqlens=(129, 40),
                   softmax_scale=1 / math.sqrt(48)), 32),
]


def new_token_inputs(spec, d_h, seed):
    rng = np.random.default_rng(seed)
    N = spec.B * spec.T_q

    def draw(*shape, scale=1.0):
        return mi.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))

    return dict(qn=draw(N, spec.H, d_h), qr=draw(N, spec.H, spec.d_r),
                w=draw(spec.H * d_h, spec.d_c, scale=1 / math.sqrt(d_h)),
                c=draw(N, spec.d_c), kr=draw(N, spec.d_r))


def positions_of(spec, seqlens):
    return np.array([seqlens[i // spec.T_q] - spec.T_q + i % spec.T_q
                     for i in range(spec.B * spec.T_q)], dtype=np.int32)


@pytest.mark.parametrize("spec,d_h", CASES, ids=[c[0].name for c in CASES])
def test_step_equals_separate_calls_and_oracle(spec, d_h):
    inp = mi.make_decode_inputs(spec)
    new = new_token_inputs(spec, d_h, spec.seed + 100)
    dev = {k: bits_to_device(v) for k, v in new.items()}
    bt = torch.from_numpy(inp.block_table).cuda()
    sl = torch.from_numpy(inp.seqlens).cuda()
    pool = bits_to_device(inp.pool_bits)
    pool_step, pool_sep = pool.clone(), pool.clone()
    N, D = spec.B * spec.T_q, spec.d_c + spec.d_r

    o1, l1 = mla.mla_decode_step(dev["qn"], dev["qr"], dev["w"], dev["c"], dev["kr"], pool_step,
                                 bt, sl, softmax_scale=spec.softmax_scale, causal=spec.causal)
    assert mla.mla_check_status() == mla.MLA_OK

    pos = positions_of(spec, inp.seqlens)
    pos_t = torch.from_numpy(pos).cuda()
    sid_t = torch.from_numpy((np.arange(N) // spec.T_q).astype(np.int32)).cuda()
    q_lat = mla.mla_absorb_query(dev["qn"], dev["qr"], pos_t, dev["w"], q_dtype=torch.bfloat16)
    mla.mla_cache_append(dev["c"], dev["kr"], sid_t, pos_t, bt, pool_sep)
    o2, l2 = mla.mla_decode_paged(q_lat.view(spec.B, spec.T_q, spec.H, D), pool_sep, bt, sl,
                                  d_c=spec.d_c, softmax_scale=spec.softmax_scale,
                                  causal=spec.causal)
    assert mla.mla_check_status() == mla.MLA_OK
    # bit patterns: unused pool rows hold NaN (poison), which never compares equal
    assert torch.equal(pool_step.view(torch.int16), pool_sep.view(torch.int16))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

    # the oracle: fp64 absorption and rows, rounded to bf16 as stored, then attention
    f = lambda bits: mi.bf16_bits_to_f32(bits).reshape(bits.shape).astype(np.float64)
    q = orc.absorb_query(f(new["qn"]), f(new["qr"]), pos, f(new["w"]), 10000.0)
    q_bits = mi.f32_to_bf16_bits(q.astype(np.float32)).reshape(spec.B, spec.T_q, spec.H, D)
    rows = orc.cache_rows(f(new["c"]), f(new["kr"]), pos, 10000.0)
    cache_bits = inp.cache_bits.copy()
    for i in range(N):
        cache_bits[inp.offsets[i // spec.T_q] + pos[i]] = mi.f32_to_bf16_bits(
            rows[i].astype(np.float32))
    want_o, want_lse = orc.decode_paged_logical(q_bits, cache_bits, inp.offsets, spec.d_c,
                                                spec.softmax_scale, spec.causal)
    assert_decode_close(o1.double().cpu().numpy(), want_o, what=spec.name)
    np.testing.assert_allclose(l1.double().cpu().numpy(), want_lse, rtol=0, atol=2e-2)


def test_step_rejects_small_workspace():
    spec, d_h = CASES[0]
    inp = mi.make_decode_inputs(spec)
    new = {k: bits_to_device(v) for k, v in new_token_inputs(spec, d_h, 7).items()}
    pool = bits_to_device(inp.pool_bits)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MLAError):
        mla.mla_decode_step(new["qn"], new["qr"], new["w"], new["c"], new["kr"], pool,
                            torch.from_numpy(inp.block_table).cuda(),
                            torch.from_numpy(inp.seqlens).cuda(),
                            softmax_scale=spec.softmax_scale, workspace=small)
