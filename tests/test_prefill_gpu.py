"""Prefill over rebuilt per-head keys and values (mla_prefill_kv,
mla_prefill_attention) against the fp64 oracle.

Tolerances:
  * rebuilt keys and values are stored in bf16: the kernel accumulates the
    512-term products in fp32 and rounds once, so a value may land one bf16
    step from the oracle's fp64 value rounded (|err| <= 2^-8 |x| plus 2e-3
    for the fp32 accumulation of terms of size ~1); the rotary key is a copy,
    bit for bit; rows past the sequence end are exact zeros;
  * attention outputs carry the bf16 rounding of the probabilities and of the
    rotated query (each a relative 2^-9 per element): the decode tolerances,
    max abs 2e-2 and relative L2 5e-3, and 2e-2 on the log-sum-exp.
"""
import numpy as np
import pytest
import torch

import head_latent_attention_28_b300 as mla
import mla_inputs as mi
import oracle as orc
from gpu_util import assert_decode_close, bits_to_device

pytestmark = pytest.mark.gpu

CASES = [
    # three query tokens at the end of a 1000-row sequence, and a 3-row one
    mi.PrefillSpec("pf_small_chunk_h4", seed=62, B=2, H=4, T_q=3, seqlens=(3, 1000)),
    # pure prefill of 200 tokens (two query tiles, a ragged second one)
    mi.PrefillSpec("pf_pure_t200_h8", seed=60, B=1, H=8, T_q=200, seqlens=(200,)),
    # chunked prefill with earlier context; 12 heads (head groups of 8 and 4)
    mi.PrefillSpec("pf_chunk_ragged_h12", seed=61, B=3, H=12, T_q=130, seqlens=(130, 400, 259)),
    # DeepSeek-V2 head count, 256 new tokens after 128 cached ones
    mi.PrefillSpec("pf_h128_t256", seed=63, B=1, H=128, T_q=256, seqlens=(384,)),
    # one new token after 699 cached rows, one head: a work item whose second
    # query tile does not exist and whose first holds one real row
    mi.PrefillSpec("pf_one_token_h1", seed=66, B=1, H=1, T_q=1, seqlens=(700,)),
    # 129 new tokens: the item's second query tile holds one real row
    mi.PrefillSpec("pf_t129_h3", seed=67, B=2, H=3, T_q=129, seqlens=(129, 300)),
]
IDS = [c.name for c in CASES]


def f64(bits):
    return mi.bf16_bits_to_f32(bits).reshape(bits.shape).astype(np.float64)


def upload(inp):
    c = inp.cache
    return dict(pool=bits_to_device(c.pool_bits), bt=torch.from_numpy(c.block_table).cuda(),
                sl=torch.from_numpy(c.seqlens).cuda(), qn=bits_to_device(inp.q_nope_bits),
                qr=bits_to_device(inp.q_rope_bits), wuk=bits_to_device(inp.w_uk_bits),
                wuv=bits_to_device(inp.w_uv_bits))


def positions(inp, b):
    L = int(inp.cache.seqlens[b])
    return np.arange(L - inp.spec.T_q, L)


def oracle_chain(inp, b):
    """fp64: rebuild the sequence's keys and values, then attend."""
    s, c = inp.spec, inp.cache
    k, v, kr = orc.rebuild_kv(f64(c.seq_rows(b)), s.H, f64(inp.w_uk_bits), f64(inp.w_uv_bits), s.d_c)
    return orc.prefill_attention(f64(inp.q_nope_bits[b]), f64(inp.q_rope_bits[b]), positions(inp, b),
                                 k, v, kr, s.softmax_scale, s.rope_base)


@pytest.mark.parametrize("spec", CASES, ids=IDS)
def test_prefill_kv_matches_oracle(spec):
    inp = mi.make_prefill_inputs(spec)
    dev = upload(inp)
    k, v, kr = mla.mla_prefill_kv(dev["pool"], dev["bt"], dev["sl"], dev["wuk"], dev["wuv"], H=spec.H)
    assert mla.mla_check_status() == mla.MLA_OK
    R = mi.prefill_kv_rows(inp.cache.max_blocks)
    assert k.shape == (spec.B, spec.H, R, spec.d_h) and R == mla.mla_prefill_kv_rows(inp.cache.max_blocks)
    # head-major buffers, compared as [b, s, h, :]
    k = k.float().cpu().numpy().transpose(0, 2, 1, 3)
    v = v.float().cpu().numpy().transpose(0, 2, 1, 3)
    kr_bits = kr.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(spec.B):
        L = int(inp.cache.seqlens[b])
        rows = inp.cache.seq_rows(b)
        want_k, want_v, _ = orc.rebuild_kv(f64(rows), spec.H, f64(inp.w_uk_bits), f64(inp.w_uv_bits), spec.d_c)
        for got, want, what in ((k[b, :L], want_k, "k_nope"), (v[b, :L], want_v, "v")):
            err = np.abs(got - want)
            bound = 2.0 ** -8 * np.abs(want) + 2e-3
            assert np.all(err <= bound), f"{spec.name} {what}: worst {np.max(err - bound):.3e} over bound"
        # the rotary key is copied bit for bit; the padding rows of the last tile are zeros
        assert np.array_equal(kr_bits[b, :L], rows[:, spec.d_c:])
        pad = (L + 127) // 128 * 128
        assert not np.any(k[b, L:pad]) and not np.any(v[b, L:pad]) and not np.any(kr_bits[b, L:pad])


@pytest.mark.parametrize("spec", CASES, ids=IDS)
def test_prefill_attention_matches_oracle(spec):
    inp = mi.make_prefill_inputs(spec, with_kv=True)
    dev = upload(inp)
    kn, vv, kr = (bits_to_device(x) for x in (inp.k_nope_bits, inp.v_bits, inp.k_rope_bits))
    o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], kn, vv, kr, dev["sl"],
                                       max_blocks_per_seq=inp.cache.max_blocks,
                                       softmax_scale=spec.softmax_scale, rope_base=spec.rope_base)
    assert mla.mla_check_status() == mla.MLA_OK
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for b in range(spec.B):
        want_o, want_lse = orc.prefill_attention(
            f64(inp.q_nope_bits[b]), f64(inp.q_rope_bits[b]), positions(inp, b),
            f64(inp.k_nope_bits[b]).transpose(1, 0, 2), f64(inp.v_bits[b]).transpose(1, 0, 2),
            f64(inp.k_rope_bits[b]), spec.softmax_scale, spec.rope_base)
        assert_decode_close(o[b], want_o, what=f"{spec.name} b={b}")
        np.testing.assert_allclose(lse[b], want_lse, rtol=0, atol=2e-2)


@pytest.mark.parametrize("spec", CASES, ids=IDS)
def test_prefill_chain_matches_oracle(spec):
    inp = mi.make_prefill_inputs(spec)
    dev = upload(inp)
    k, v, kr = mla.mla_prefill_kv(dev["pool"], dev["bt"], dev["sl"], dev["wuk"], dev["wuv"], H=spec.H)
    o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], k, v, kr, dev["sl"],
                                       max_blocks_per_seq=inp.cache.max_blocks,
                                       softmax_scale=spec.softmax_scale, rope_base=spec.rope_base)
    assert mla.mla_check_status() == mla.MLA_OK
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for b in range(spec.B):
        want_o, want_lse = oracle_chain(inp, b)
        assert_decode_close(o[b], want_o, what=f"{spec.name} b={b}")
        np.testing.assert_allclose(lse[b], want_lse, rtol=0, atol=2e-2)


def test_prefill_attention_schedules_agree():
    """The attention kernel is persistent: its CTAs take work items (two
    query tiles of one head) from a counter kept per stream and zeroed by the
    kernel for the next launch, or in a fixed order on the per-thread default
    stream.  384 items (the last pair of each head has one tile) over at most
    one CTA per SM: sampled queries match the oracle, and repeated launches,
    fresh streams and the fixed order all give the same bits."""
    from cuda.bindings import runtime as cudart
    spec = mi.PrefillSpec("pf_sched_h64_t640", seed=65, B=2, H=64, T_q=640, seqlens=(640, 900))
    inp = mi.make_prefill_inputs(spec, with_kv=True)
    dev = upload(inp)
    kn, vv, kr = (bits_to_device(x) for x in (inp.k_nope_bits, inp.v_bits, inp.k_rope_bits))

    def run(stream=None):
        o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], kn, vv, kr, dev["sl"],
                                           max_blocks_per_seq=inp.cache.max_blocks,
                                           softmax_scale=spec.softmax_scale, rope_base=spec.rope_base,
                                           stream=stream)
        torch.cuda.synchronize()
        if stream is not None:
            cudart.cudaStreamSynchronize(stream)
        return o, lse

    torch.cuda.synchronize()
    ref_o, ref_lse = run()
    assert mla.mla_check_status() == mla.MLA_OK
    queries = np.array([0, 127, 128, 255, 256, 383, 384, 511, 512, 639])
    for b in range(spec.B):
        want_o, want_lse = orc.prefill_attention(
            f64(inp.q_nope_bits[b, queries]), f64(inp.q_rope_bits[b, queries]), positions(inp, b)[queries],
            f64(inp.k_nope_bits[b]).transpose(1, 0, 2), f64(inp.v_bits[b]).transpose(1, 0, 2),
            f64(inp.k_rope_bits[b]), spec.softmax_scale, spec.rope_base)
        assert_decode_close(ref_o[b, queries].double().cpu().numpy(), want_o, what=f"sampled queries b={b}")
        np.testing.assert_allclose(ref_lse[b, queries].double().cpu().numpy(), want_lse, rtol=0, atol=2e-2)
    outs = [run(), run(2)]                      # 2 = cudaStreamPerThread: the fixed order
    streams = []
    for _ in range(3):
        err, st = cudart.cudaStreamCreate()
        assert err == cudart.cudaError_t.cudaSuccess
        streams.append(st)
        outs += [run(int(st)), run(int(st))]
    # two launches in flight at once on two streams (two counters in use together)
    pair = []
    for st in streams[:2]:
        pair.append(mla.mla_prefill_attention(dev["qn"], dev["qr"], kn, vv, kr, dev["sl"],
                                              max_blocks_per_seq=inp.cache.max_blocks,
                                              softmax_scale=spec.softmax_scale, rope_base=spec.rope_base,
                                              stream=int(st)))
    for st in streams:
        cudart.cudaStreamSynchronize(st)
        cudart.cudaStreamDestroy(st)
    torch.cuda.synchronize()
    outs += pair
    assert mla.mla_check_status() == mla.MLA_OK
    for o, lse in outs:
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


def test_prefill_bad_length_reports_and_writes_zeros():
    spec = mi.PrefillSpec("pf_bad_len", seed=64, B=2, H=4, T_q=5, seqlens=(5, 300))
    inp = mi.make_prefill_inputs(spec, with_kv=True)
    dev = upload(inp)
    kn, vv, kr = (bits_to_device(x) for x in (inp.k_nope_bits, inp.v_bits, inp.k_rope_bits))
    sl = dev["sl"].clone()
    sl[0] = 4                                   # fewer rows than new tokens
    o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], kn, vv, kr, sl,
                                       max_blocks_per_seq=inp.cache.max_blocks,
                                       softmax_scale=spec.softmax_scale)
    assert mla.mla_check_status() == mla.MLA_ERR_BAD_INDEX
    assert not torch.any(o[0]) and not torch.any(lse[0])
    want_o, _ = orc.prefill_attention(
        f64(inp.q_nope_bits[1]), f64(inp.q_rope_bits[1]), positions(inp, 1),
        f64(inp.k_nope_bits[1]).transpose(1, 0, 2), f64(inp.v_bits[1]).transpose(1, 0, 2),
        f64(inp.k_rope_bits[1]), spec.softmax_scale, spec.rope_base)
    assert_decode_close(o[1].double().cpu().numpy(), want_o, what="valid sequence next to a bad one")


def test_prefill_rejects_unsupported_and_bad_args():
    spec = CASES[0]
    inp = mi.make_prefill_inputs(spec, with_kv=True)
    dev = upload(inp)
    kn, vv, kr = (bits_to_device(x) for x in (inp.k_nope_bits, inp.v_bits, inp.k_rope_bits))
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_prefill_attention(dev["qn"], dev["qr"], kn, vv, kr, dev["sl"],
                                  max_blocks_per_seq=inp.cache.max_blocks, softmax_scale=0.0)
    assert ei.value.status == mla.MLA_ERR_INVALID_ARG
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_prefill_kv(dev["pool"].float(), dev["bt"], dev["sl"], dev["wuk"].float(),
                           dev["wuv"].float(), H=spec.H)
    assert ei.value.status == mla.MLA_ERR_UNSUPPORTED


@pytest.mark.slow
def test_prefill_full_size_sampled():
    """The bench workload (one 4096-token prompt, 128 heads), every output of
    the rebuild checked on sampled rows and the attention on sampled queries."""
    spec = mi.V2_PREFILL
    inp = mi.make_prefill_inputs(spec)
    dev = upload(inp)
    k, v, kr = mla.mla_prefill_kv(dev["pool"], dev["bt"], dev["sl"], dev["wuk"], dev["wuv"], H=spec.H)
    o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], k, v, kr, dev["sl"],
                                       max_blocks_per_seq=inp.cache.max_blocks,
                                       softmax_scale=spec.softmax_scale, rope_base=spec.rope_base)
    assert mla.mla_check_status() == mla.MLA_OK
    rows = f64(inp.cache.seq_rows(0))
    want_k, want_v, want_kr = orc.rebuild_kv(rows, spec.H, f64(inp.w_uk_bits), f64(inp.w_uv_bits), spec.d_c)
    rng = np.random.default_rng(11)
    sample_rows = np.concatenate([[0, 127, 128, 4095], rng.integers(0, 4096, 12)])
    kk = k[0][:, sample_rows].float().cpu().numpy().transpose(1, 0, 2)
    vv = v[0][:, sample_rows].float().cpu().numpy().transpose(1, 0, 2)
    for got, want in ((kk, want_k[sample_rows]), (vv, want_v[sample_rows])):
        assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 2e-3)
    queries = np.concatenate([[0, 1, 127, 128, 4095], rng.integers(0, 4096, 7)])
    pos = positions(inp, 0)[queries]
    want_o, want_lse = orc.prefill_attention(f64(inp.q_nope_bits[0, queries]), f64(inp.q_rope_bits[0, queries]),
                                             pos, want_k, want_v, want_kr, spec.softmax_scale, spec.rope_base)
    assert_decode_close(o[0, queries].double().cpu().numpy(), want_o, what="full-size sampled queries")
    np.testing.assert_allclose(lse[0, queries].double().cpu().numpy(), want_lse, rtol=0, atol=2e-2)


def test_prefill_lazy_rescale_after_a_jump():
    """Keys 200-259 scaled by 16: every row's score maximum jumps by far more
    than 2^8 (8 log2 units) after the first 128-key tile, so the kernel must
    rescale its output accumulator in tensor memory mid-sequence (the lazy
    O-rescale).  The jump is checked on the oracle's scores first."""
    spec = mi.PrefillSpec("pf_lazy_rescale", seed=65, B=1, H=8, T_q=64, seqlens=(512,))
    inp = mi.make_prefill_inputs(spec, with_kv=True)
    kn = f64(inp.k_nope_bits)                                   # [B, H, R, d_h]
    kn[:, :, 200:260, :] *= 16.0
    inp.k_nope_bits = mi.f32_to_bf16_bits(kn.astype(np.float32)).reshape(kn.shape)
    pos = positions(inp, 0)
    qn = f64(inp.q_nope_bits[0])                                # [T, H, d_h]
    qr = orc.rope(f64(inp.q_rope_bits[0]).transpose(1, 0, 2), pos, spec.rope_base).transpose(1, 0, 2)
    k = f64(inp.k_nope_bits[0]).transpose(1, 0, 2)              # [R, H, d_h]
    kr = f64(inp.k_rope_bits[0])                                # [R, d_r]
    s = spec.softmax_scale * (np.einsum("thd,shd->ths", qn, k) + np.einsum("thd,sd->ths", qr, kr))
    jump = (s[:, :, 128:int(pos[-1]) + 1].max(axis=2) - s[:, :, :128].max(axis=2)) / np.log(2.0)
    assert jump.min() > 8.0, jump.min()
    dev = upload(inp)
    kd, vd, krd = (bits_to_device(x) for x in (inp.k_nope_bits, inp.v_bits, inp.k_rope_bits))
    o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], kd, vd, krd, dev["sl"],
                                       max_blocks_per_seq=inp.cache.max_blocks,
                                       softmax_scale=spec.softmax_scale, rope_base=spec.rope_base)
    assert mla.mla_check_status() == mla.MLA_OK
    want_o, want_lse = orc.prefill_attention(qn, f64(inp.q_rope_bits[0]), pos, k,
                                             f64(inp.v_bits[0]).transpose(1, 0, 2), kr,
                                             spec.softmax_scale, spec.rope_base)
    assert_decode_close(o.double().cpu().numpy()[0], want_o, what="lazy rescale")
    np.testing.assert_allclose(lse.double().cpu().numpy()[0], want_lse, rtol=0, atol=2e-2)



def test_chunked_prefill_two_chunks_rebuilds_only_new_rows():
    """Two chunks per sequence: the first rebuilds rows [0, L1) in full, the
    second (mla_prefill_kv_chunk) only its T_new rows into the same buffers.
    The buffers then equal one full rebuild at L2 bit for bit, rows of the
    first chunk untouched by the second call (checked by planting a marker
    where it must not write), and the second chunk's attention matches the
    oracle chain."""
    spec = mi.PrefillSpec("pf_two_chunks", seed=66, B=2, H=12, T_q=130, seqlens=(430, 200))
    inp = mi.make_prefill_inputs(spec)
    dev = upload(inp)
    sl2 = dev["sl"]
    sl1 = sl2 - spec.T_q                                     # 300 and 70 rows before the chunk
    k, v, kr = mla.mla_prefill_kv(dev["pool"], dev["bt"], sl1, dev["wuk"], dev["wuv"], H=spec.H)
    # a marker in rows of the first chunk: the chunk's call must leave it
    k[:, :, 5, :] = 7.0
    mla.mla_prefill_kv(dev["pool"], dev["bt"], sl2, dev["wuk"], dev["wuv"], H=spec.H, out=(k, v, kr),
                       T_new=spec.T_q)
    assert mla.mla_check_status() == mla.MLA_OK
    assert torch.all(k[:, :, 5, :] == 7.0)
    k[:, :, 5, :] = mla.mla_prefill_kv(dev["pool"], dev["bt"], sl1, dev["wuk"], dev["wuv"], H=spec.H)[0][:, :, 5, :]
    kf, vf, krf = mla.mla_prefill_kv(dev["pool"], dev["bt"], sl2, dev["wuk"], dev["wuv"], H=spec.H)
    assert mla.mla_check_status() == mla.MLA_OK
    for b in range(spec.B):          # rows the calls write: up to L2 rounded up to 128
        n = (int(inp.cache.seqlens[b]) + 127) // 128 * 128
        assert torch.equal(k[b, :, :n], kf[b, :, :n]) and torch.equal(v[b, :, :n], vf[b, :, :n])
        assert torch.equal(kr[b, :n], krf[b, :n])
    o, lse = mla.mla_prefill_attention(dev["qn"], dev["qr"], k, v, kr, sl2,
                                       max_blocks_per_seq=inp.cache.max_blocks,
                                       softmax_scale=spec.softmax_scale, rope_base=spec.rope_base)
    assert mla.mla_check_status() == mla.MLA_OK
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for b in range(spec.B):
        want_o, want_lse = oracle_chain(inp, b)
        assert_decode_close(o[b], want_o, what=f"second chunk b={b}")
        np.testing.assert_allclose(lse[b], want_lse, rtol=0, atol=2e-2)
