"""Parity of mla_decode_paged (through the C ABI) with the fp64 oracle.

Medium cases are compared element by element over the whole output; the
five full-size workloads are run in the launch configuration the benchmark
times and compared on sampled sequences the oracle computes one by one.
"""

import math

import numpy as np
import pytest
import torch

import head_latent_attention_28_b300 as mla
import mla_inputs as mi
import oracle as orc
from gpu_util import (BF16_MAX_ABS, BF16_REL_L2, F32_MAX_ABS, assert_decode_close,
                      bits_to_device, run_decode, upload_decode)

pytestmark = pytest.mark.gpu


def oracle_all(inp, batch=None):
    s = inp.spec
    return orc.decode_paged_logical(inp.q_bits, inp.cache_bits, inp.offsets, s.d_c,
                                    s.softmax_scale, s.causal, batch=batch)


MEDIUM = [
    mi.DecodeSpec("h128_ragged", seed=10, B=3, H=128, seqlens=(65, 1000, 3000)),
    mi.DecodeSpec("h128_edges", seed=11, B=6, H=128, seqlens=(1, 63, 64, 65, 128, 129)),
    mi.DecodeSpec("h128_one_long", seed=12, B=1, H=128, seqlens=(20000,)),
    mi.DecodeSpec("h128_pool_gaps", seed=13, B=4, H=128, seqlens=(700, 1, 2000, 130),
                  num_blocks=200),
    mi.DecodeSpec("h16_tq2_causal", seed=14, B=5, H=16, T_q=2, causal=True,
                  seqlens=(2, 64, 65, 700, 2500)),
    mi.DecodeSpec("h64_tq2_causal", seed=15, B=3, H=64, T_q=2, causal=True,
                  seqlens=(2, 300, 4000)),
    mi.DecodeSpec("h32_tq4_causal", seed=16, B=3, H=32, T_q=4, causal=True,
                  seqlens=(4, 67, 1500)),
    # more than 128 query rows: the tensor-core kernel takes them in row groups
    # of 128 over the same pages (the last group may be short)
    mi.DecodeSpec("h128_tq2_causal_row_groups", seed=26, B=3, H=128, T_q=2, causal=True,
                  seqlens=(2, 1000, 2050)),
    mi.DecodeSpec("h32_tq8_causal_row_groups", seed=27, B=2, H=32, T_q=8, causal=True,
                  seqlens=(300, 1500)),
    mi.DecodeSpec("h64_tq3_causal_short_group", seed=28, B=3, H=64, T_q=3, causal=True,
                  seqlens=(3, 200, 1300)),
    mi.DecodeSpec("h128_tq4_four_groups", seed=29, B=2, H=128, T_q=4, causal=True,
                  seqlens=(65, 700)),
    # row counts that are not a multiple of 32: the last 32-row group of the
    # epilogue is partial (72 = 2 x 32 + 8 rows; 40 = 32 + 8)
    mi.DecodeSpec("h24_tq3_rows72", seed=31, B=5, H=24, T_q=3,
                  seqlens=(3, 700, 1500, 64, 2100)),
    mi.DecodeSpec("h40_causal_tq1_rows40", seed=32, B=3, H=40, seqlens=(129, 1, 900)),
    mi.DecodeSpec("h20_tq2_causal_rows40", seed=33, B=3, H=20, T_q=2, causal=True,
                  seqlens=(2, 500, 1200)),
    # a causal chunk of 32 new tokens (chunked prefill through the absorbed
    # path): 32 row groups of 128 rows over the same pages, each query token
    # sees the cache up to itself
    mi.DecodeSpec("h128_chunk32_causal", seed=30, B=2, H=128, T_q=32, causal=True,
                  seqlens=(32, 500)),
    mi.DecodeSpec("h8_small_rows", seed=17, B=2, H=8, d_c=64, d_r=16, seqlens=(129, 40),
                  softmax_scale=1 / math.sqrt(48)),
    mi.DecodeSpec("many_short_seqs", seed=18, B=600, H=16, seqlen_range=(1, 200)),
    # more than 64 work items per worker: the planner hands them out in batches
    mi.DecodeSpec("items_beyond_one_batch", seed=34, B=5000, H=8, seqlen_range=(1, 64)),
]


@pytest.mark.parametrize("spec", MEDIUM, ids=[s.name for s in MEDIUM])
def test_decode_medium_matches_oracle(spec):
    inp = mi.make_decode_inputs(spec)
    o, lse = run_decode(inp)
    want_o, want_lse = oracle_all(inp)
    assert_decode_close(o, want_o, what=spec.name)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=2e-2)


def test_decode_float32_cache_tight_tolerance():
    """float32 queries and cache go through float FFMA: max abs 1e-4."""
    spec = mi.DecodeSpec("f32", seed=19, B=3, H=8, d_c=64, d_r=16, seqlens=(129, 1, 700),
                         softmax_scale=1 / math.sqrt(48))
    inp = mi.make_decode_inputs(spec)
    q = torch.from_numpy(mi.bf16_bits_to_f32(inp.q_bits).reshape(inp.q_bits.shape)).cuda()
    pool = mi.bf16_bits_to_f32(inp.pool_bits.reshape(-1)).reshape(inp.pool_bits.shape)
    pool = torch.from_numpy(pool).cuda()
    # perturb below bf16 resolution so the test sees float, not bf16, inputs
    g = torch.Generator(device="cuda").manual_seed(0)
    q = q + 1e-3 * torch.randn(q.shape, device="cuda", generator=g)
    valid = torch.isfinite(pool)
    pool = torch.where(valid, pool + 1e-3 * torch.randn(pool.shape, device="cuda", generator=g),
                       pool)
    bt = torch.from_numpy(inp.block_table).cuda()
    sl = torch.from_numpy(inp.seqlens).cuda()
    o, lse = mla.mla_decode_paged(q, pool, bt, sl, d_c=64, softmax_scale=spec.softmax_scale)
    assert mla.mla_check_status() == mla.MLA_OK
    qn = q.double().cpu().numpy()
    pn = pool.double().cpu().numpy()
    for b in range(3):
        L = int(inp.seqlens[b])
        rows = np.concatenate([pn[inp.block_table[b, j]] for j in range((L + 63) // 64)])[:L]
        wo, wl = orc.decode_attention(qn[b], rows, 64, spec.softmax_scale, False)
        assert np.abs(o[b].double().cpu().numpy() - wo).max() <= F32_MAX_ABS
        assert np.abs(lse[b].double().cpu().numpy() - wl).max() <= F32_MAX_ABS


# --------------------------------------------------------------------------
# bit-exact indexing
# --------------------------------------------------------------------------

def test_one_hot_probe_returns_exact_row():
    """Give one token a score that beats every other by >1000 (natural
    units): p is exactly 1 there and 0 elsewhere, so o must equal that
    token's latent bitwise.  A decoy with an even larger score sits in the
    row just past the sequence end and must be ignored."""
    spec = mi.DecodeSpec("probe", seed=20, B=2, H=128, seqlens=(300, 129))
    inp = mi.make_decode_inputs(spec)
    d_c, D = spec.d_c, spec.D
    pool = inp.pool_bits.copy()
    q = np.zeros_like(inp.q_bits)
    big = mi.f32_to_bf16_bits(np.array([128.0], np.float32))[0]
    huge = mi.f32_to_bf16_bits(np.array([256.0], np.float32))[0]
    zero = np.uint16(0)
    for b in range(2):
        L = int(inp.seqlens[b])
        for j in range((L + 63) // 64):
            blk = inp.block_table[b, j]
            n = min(64, L - 64 * j)
            pool[blk, :n, d_c:] = zero                  # rotary parts 0 for valid rows
        q[b, 0, :, d_c] = big                            # every head looks at dim d_c
    dev = upload_decode(inp)
    dev["q"] = bits_to_device(q)
    targets = {0: [0, 63, 64, 127, 128, 255, 256, 299], 1: [0, 64, 127, 128]}
    for b, tlist in targets.items():
        L = int(inp.seqlens[b])
        last_blk = inp.block_table[b, (L - 1) // 64]
        decoy_row = L % 64                               # row just past the end
        for t in tlist:
            p = pool.copy()
            blk, r = inp.block_table[b, t // 64], t % 64
            p[blk, r, d_c] = big
            if decoy_row:
                p[last_blk, decoy_row, :] = mi.f32_to_bf16_bits(np.full(D, 3.0, np.float32))
                p[last_blk, decoy_row, d_c] = huge
            dev["pool"] = bits_to_device(p)
            o, _ = run_decode(inp, dev)
            want = mi.bf16_bits_to_f32(p[blk, r, :d_c]).astype(np.float64)
            np.testing.assert_array_equal(o[b, 0], np.broadcast_to(want, (128, d_c)),
                                          err_msg=f"seq {b} target token {t}")


def test_layout_invariance_bitwise():
    """The same logical cache under two different block permutations gives
    bitwise identical outputs (the split plan depends only on lengths)."""
    spec = mi.DecodeSpec("perm", seed=21, B=5, H=128, seqlens=(3000, 64, 1, 1500, 777),
                         num_blocks=300)
    inp = mi.make_decode_inputs(spec)
    o1, l1 = run_decode(inp)
    rng = np.random.default_rng(99)
    perm = rng.permutation(spec.num_blocks).astype(np.int32)
    bt2 = np.where(inp.block_table >= 0, perm[np.maximum(inp.block_table, 0)], -1).astype(np.int32)
    pool2 = np.full_like(inp.pool_bits, mi.BF16_NAN)
    used = inp.block_table[inp.block_table >= 0]
    pool2[perm[used]] = inp.pool_bits[used]
    inp2 = mi.DecodeInputs(spec, inp.seqlens, inp.offsets, bt2, inp.q_bits, inp.cache_bits, pool2)
    o2, l2 = run_decode(inp2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_batch_order_invariance():
    """A sequence's output does not depend on its neighbours beyond the
    split plan: running it alone changes only rounding.  (On the tensor-core
    path the probabilities are rounded to bf16 relative to each worker's
    running max, so a different split rounds differently: the bf16 decode
    tolerance applies, not a float one.)"""
    spec = mi.DecodeSpec("order", seed=22, B=3, H=128, seqlens=(5000, 100, 2500))
    inp = mi.make_decode_inputs(spec)
    o, _ = run_decode(inp)
    for b in range(3):
        sub = mi.DecodeSpec("one", seed=22, B=1, H=128, seqlens=(int(inp.seqlens[b]),))
        one = mi.DecodeInputs(sub, inp.seqlens[b:b + 1], np.array([0, inp.seqlens[b]]),
                              inp.block_table[b:b + 1], inp.q_bits[b:b + 1],
                              inp.seq_rows(b), inp.pool_bits)
        ob, _ = run_decode(one)
        assert_decode_close(ob[0], o[b], what=f"seq {b} alone vs in batch")


# --------------------------------------------------------------------------
# device-side errors (bounds checks turn bad indices into a status, no fault)
# --------------------------------------------------------------------------

def test_bad_block_id_reports_status():
    spec = mi.DecodeSpec("badblk", seed=23, B=2, H=128, seqlens=(200, 100))
    inp = mi.make_decode_inputs(spec)
    dev = upload_decode(inp)
    bt = inp.block_table.copy()
    bt[1, 0] = spec.num_blocks if spec.num_blocks else inp.num_blocks   # one past the pool
    dev["bt"] = torch.from_numpy(bt).cuda()
    o, _ = mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], d_c=512,
                                softmax_scale=spec.softmax_scale)
    assert mla.mla_check_status() == mla.MLA_ERR_BAD_INDEX
    assert mla.mla_check_status() == mla.MLA_OK          # cleared by the read
    want, _ = oracle_all(inp, batch=[0])
    assert_decode_close(o[0:1].double().cpu().numpy(), want[0:1], what="good sequence")


def test_bad_seqlen_reports_status_and_zeroes_that_sequence():
    spec = mi.DecodeSpec("badlen", seed=24, B=3, H=16, T_q=2, causal=True,
                         seqlens=(300, 100, 500))
    inp = mi.make_decode_inputs(spec)
    dev = upload_decode(inp)
    sl = inp.seqlens.copy()
    sl[1] = 1                                            # shorter than T_q
    sl[2] = inp.max_blocks * 64 + 1                      # beyond the block table
    dev["sl"] = torch.from_numpy(sl).cuda()
    o, lse = mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], d_c=512,
                                  softmax_scale=spec.softmax_scale, causal=True)
    assert mla.mla_check_status() == mla.MLA_ERR_BAD_INDEX
    on = o.double().cpu().numpy()
    assert np.all(on[1:] == 0.0)
    want, _ = oracle_all(inp, batch=[0])
    assert_decode_close(on[0:1], want[0:1], what="valid sequence")


def test_workspace_too_small_is_rejected():
    spec = mi.DecodeSpec("ws", seed=25, B=2, H=128, seqlens=(100, 100))
    inp = mi.make_decode_inputs(spec)
    dev = upload_decode(inp)
    need = mla.mla_decode_workspace_size(2, 1, 128, 512, 64)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], d_c=512,
                             softmax_scale=0.07, workspace=ws)
    assert ei.value.status == mla.MLA_ERR_WORKSPACE


# --------------------------------------------------------------------------
# full-size workloads, sampled
# --------------------------------------------------------------------------

FULL = [mi.V2_DECODE, mi.RAGGED_SERVING, mi.LONG_CONTEXT, mi.FEW_HEAD_MTP]


def straddling_sequences(inp):
    """Sequences whose pages the decode's split plan gives to more than one
    worker (their results go through the log-sum-exp merge)."""
    s = inp.spec
    W = mla.mla_decode_num_workers(s.B, s.T_q, s.H, s.d_c, s.d_r, mla.MLA_BF16)
    C = mla.mla_decode_item_cost(s.T_q, s.H, s.d_c, s.d_r, mla.MLA_BF16)
    fw, lw, _ = mla.mla_decode_split_plan(inp.seqlens, s.T_q, inp.block_table.shape[1], W, C)
    return [b for b in range(s.B) if fw[b] != lw[b]]


def sample_sequences(inp, n, prefer=()):
    """Both ends, the longest and shortest, up to n // 2 of `prefer`, then
    seeded random picks, n in all (at least 4)."""
    L = inp.seqlens
    picks = {0, len(L) - 1, int(np.argmax(L)), int(np.argmin(L))}
    rng = np.random.default_rng(inp.spec.seed + 1000)
    prefer = list(prefer)
    if prefer:
        picks |= set(rng.choice(prefer, size=min(n // 2, len(prefer)), replace=False).tolist())
    rest = [b for b in rng.permutation(len(L)).tolist() if b not in picks]
    return sorted(picks | set(rest[: max(0, max(n, 4) - len(picks))]))


@pytest.mark.parametrize("spec", FULL, ids=[s.name for s in FULL])
def test_full_size_workload_sampled(spec):
    inp = mi.make_decode_inputs(spec)
    o, lse = run_decode(inp)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    # the ragged batch: about 24 sequences, half of them split across workers
    n = 2 if spec.B <= 4 else 24 if spec is mi.RAGGED_SERVING else 6
    batch = sample_sequences(inp, n, straddling_sequences(inp) if spec is mi.RAGGED_SERVING else ())
    if spec is mi.RAGGED_SERVING:
        assert len(batch) >= 24 and len(set(batch) & set(straddling_sequences(inp))) >= 8
    want_o, want_l = oracle_all(inp, batch=batch)
    for b in batch:
        assert_decode_close(o[b], want_o[b], what=f"{spec.name} seq {b}")
        np.testing.assert_allclose(lse[b], want_l[b], rtol=0, atol=2e-2)


def _random_specs(n, seed):
    """Seeded random shapes: any head count and query-token count (row groups
    and partial 32-row epilogue groups), causal or not, ragged lengths."""
    rng = np.random.default_rng(seed)
    specs = []
    for k in range(n):
        H, T_q = int(rng.integers(1, 129)), int(rng.integers(1, 9))
        B = int(rng.integers(1, 5))
        causal = bool(rng.random() < 0.5)
        lens = tuple(int(x) for x in rng.integers(T_q, 1500, size=B))
        specs.append(mi.DecodeSpec(f"random{k}_h{H}_tq{T_q}", seed=seed * 100 + k, B=B, H=H,
                                   T_q=T_q, causal=causal, seqlens=lens))
    return specs


RANDOM = _random_specs(10, 61)


@pytest.mark.parametrize("spec", RANDOM, ids=[s.name for s in RANDOM])
def test_random_shapes_match_oracle(spec):
    inp = mi.make_decode_inputs(spec)
    o, lse = run_decode(inp)
    want_o, want_lse = oracle_all(inp)
    assert_decode_close(o, want_o, what=spec.name)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=2e-2)


# --------------------------------------------------------------------------
# split invariance: the same batch with 1, 2, 7 and 74 split workers
# --------------------------------------------------------------------------

SPLIT_SPEC = mi.DecodeSpec("forced_splits", seed=77, B=3, H=128, seqlens=(5000, 300, 12000))


@pytest.mark.parametrize("splits", [1, 2, 7, 74])
def test_forced_splits_match_oracle(splits):
    """Every split count gives the oracle's result at the decode tolerance;
    one worker holds everything at 1 split, the long sequences straddle
    workers at 7 and 74."""
    s = SPLIT_SPEC
    inp = mi.make_decode_inputs(s)
    natural = mla.mla_decode_num_workers(s.B, s.T_q, s.H, s.d_c, s.d_r, mla.MLA_BF16)
    try:
        mla.mla_test_force_splits(splits)
        W = mla.mla_decode_num_workers(s.B, s.T_q, s.H, s.d_c, s.d_r, mla.MLA_BF16)
        assert W == min(splits, natural)
        o, lse = run_decode(inp)
        C = mla.mla_decode_item_cost(s.T_q, s.H, s.d_c, s.d_r, mla.MLA_BF16)
        fw, lw, _ = mla.mla_decode_split_plan(inp.seqlens, s.T_q, inp.block_table.shape[1], W, C)
    finally:
        mla.mla_test_force_splits(0)
    assert mla.mla_decode_num_workers(s.B, s.T_q, s.H, s.d_c, s.d_r, mla.MLA_BF16) == natural
    if splits == 1:
        assert list(fw) == [0, 0, 0] and list(lw) == [0, 0, 0]
    if splits >= 7:
        assert lw[2] > fw[2] and lw[0] > fw[0]
    want_o, want_l = oracle_all(inp)
    for b in range(s.B):
        assert_decode_close(o[b], want_o[b], what=f"{splits} splits, seq {b}")
        np.testing.assert_allclose(lse[b], want_l[b], rtol=0, atol=2e-2)
