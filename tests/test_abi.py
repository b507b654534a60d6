"""CPU checks of the C ABI: the library loads, exports every declared entry
point, rejects bad arguments on the host before touching a device, and its
split planner partitions pages as documented."""

import os
import re

import numpy as np
import pytest
import torch

import head_latent_attention_28_b300 as mla

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(mla_\w+)\s*\(", text))


def test_header_declarations_match_binding_and_exports():
    decl = declared_functions()
    assert decl, "no declarations parsed"
    assert decl == set(mla.SIGNATURES), decl ^ set(mla.SIGNATURES)
    lib = mla.load_library()
    for name in decl:
        assert hasattr(lib, name)


def test_status_strings_and_version():
    for code in range(7):
        assert mla.mla_status_string(code)
    assert mla.lib().mla_version() >= 100


def test_decode_rejects_bad_arguments_on_host():
    lib = mla.lib()
    P = 16  # a non-null, 16-byte aligned dummy address; never dereferenced
    ok = dict(q=P, kv=P, dt=1, bt=P, sl=P, B=1, T_q=1, H=128, d_c=512, d_r=64, page=64,
              maxb=4, nb=4, scale=0.07, causal=0, ws=P, wsb=1 << 30, o=P, lse=None, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.mla_decode_paged(a["q"], a["kv"], a["dt"], a["bt"], a["sl"], a["B"], a["T_q"],
                                    a["H"], a["d_c"], a["d_r"], a["page"], a["maxb"], a["nb"],
                                    a["scale"], a["causal"], a["ws"], a["wsb"], a["o"], a["lse"],
                                    a["s"])
    bad = [dict(q=None), dict(kv=None), dict(bt=None), dict(sl=None), dict(o=None),
           dict(B=0), dict(T_q=0), dict(H=0), dict(d_c=0), dict(d_c=513), dict(d_r=-1),
           dict(d_r=600), dict(page=32), dict(maxb=0), dict(nb=0), dict(scale=0.0),
           dict(dt=7), dict(q=P + 2)]
    for kw in bad:
        assert call(**kw) == mla.MLA_ERR_INVALID_ARG, kw


def test_other_calls_reject_bad_arguments_on_host():
    lib = mla.lib()
    P = 16
    # append: odd d_r, bad page size, null cache
    assert lib.mla_cache_append(P, P, 1, P, P, 1, P, 1, 4, P, 1, 4, 64, 512, 63, 1e4, None) == 1
    assert lib.mla_cache_append(P, P, 1, P, P, 1, P, 1, 4, P, 1, 4, 32, 512, 64, 1e4, None) == 1
    assert lib.mla_cache_append(P, P, 1, P, P, 1, P, 1, 4, None, 1, 4, 64, 512, 64, 1e4, None) == 1
    assert lib.mla_cache_append(P, P, 1, P, P, 0, P, 1, 4, P, 1, 4, 64, 512, 64, 1e4, None) == 0
    # absorb query / output
    assert lib.mla_absorb_query(None, P, P, P, 1, 1, 8, 32, 64, 16, 1e4, P, 1, None) == 1
    assert lib.mla_absorb_query(P, P, P, P, 1, 1, 8, 32, 64, 15, 1e4, P, 1, None) == 1
    assert lib.mla_absorb_output(P, P, P, 1, 1, 8, 32, 64, 0, P, None) == 1
    assert lib.mla_absorb_output(P, P, P, 1, 1, 256, 256, 64, 64, P, None) == 1  # H*d_h too big


def brute_force_plan(seqlens, T_q, max_blocks, W, C=0):
    """Explicit unit list: each valid sequence contributes C item-cost units,
    then one unit per page; with W' = min(W, U // (C + 1)) active workers,
    unit u goes to the worker w with floor(U w / W') <= u < floor(U (w+1) / W').
    Returns first/last owner of each sequence's pages, T, and per active
    worker (pages, items)."""
    cap = max_blocks * 64
    units = []                              # (sequence, is_page)
    for b, L in enumerate(seqlens):
        if T_q <= L <= cap:
            units += [(b, False)] * C + [(b, True)] * ((L + 63) // 64)
    U = len(units)
    T = sum(1 for _, pg in units if pg)
    Wa = min(W, U // (C + 1))
    owners = []
    for w in range(Wa):
        owners += [w] * ((U * (w + 1)) // Wa - (U * w) // Wa)
    first = [-1] * len(seqlens)
    last = [-1] * len(seqlens)
    work = [[0, set()] for _ in range(Wa)]
    for (b, pg), w in zip(units, owners):
        if not pg:
            continue
        if first[b] < 0:
            first[b] = w
        last[b] = w
        work[w][0] += 1
        work[w][1].add(b)
    return first, last, T, [(n, len(items)) for n, items in work]


@pytest.mark.parametrize("C", [0, 3, 5])
@pytest.mark.parametrize("W", [1, 3, 74, 148, 1000])
def test_split_plan_matches_brute_force(W, C):
    rng = np.random.default_rng(W + 7 * C)
    for trial in range(5):
        B = int(rng.integers(1, 60))
        seqlens = rng.integers(0, 3000, size=B).astype(np.int32)
        seqlens[rng.random(B) < 0.1] = 5000       # over capacity -> invalid
        f, l, T = mla.mla_decode_split_plan(seqlens, 2, 64, W, C)
        bf, bl, bT, work = brute_force_plan(seqlens.tolist(), 2, 64, W, C)
        assert T == bT
        np.testing.assert_array_equal(f, bf)
        np.testing.assert_array_equal(l, bl)
        # no active worker is empty, and the cost pages + C * items of the
        # workers differs by at most 2 C + 1 units (a range holds floor or
        # ceil of U / W' units; a worker starting inside a sequence's pages
        # pays C for that item outside its units, and one whose range ends
        # inside a sequence's C units holds units it does not pay for)
        assert all(n >= 1 for n, _ in work)
        costs = [n + C * k for n, k in work]
        assert max(costs) - min(costs) <= 2 * C + 1
        # partial slots b + w are distinct over all (sequence, worker) pairs,
        # and every worker between a sequence's first and last holds part of it
        slots = [b + w for b in range(B) if f[b] >= 0 and f[b] != l[b]
                 for w in range(f[b], l[b] + 1)]
        assert len(slots) == len(set(slots))
        assert all(s < B + W for s in slots)
        valid = [b for b in range(B) if f[b] >= 0]
        for b0, b1 in zip(valid, valid[1:]):
            assert f[b1] in (l[b0], l[b0] + 1)   # contiguous, no skipped worker

    # few pages, many workers: the case where idle workers would leave holes
    f, l, T = mla.mla_decode_split_plan(np.array([300, 129], np.int32), 1, 8, W, C)
    assert T == 8 and f[0] == 0 and l[1] == min(W, (8 + 2 * C) // (C + 1)) - 1


def test_item_cost_per_kernel():
    # tensor-core shapes: grows with the query rows (5 pages at 128 rows, 3 at 32)
    assert mla.mla_decode_item_cost(1, 128, 512, 64) == 5
    assert mla.mla_decode_item_cost(2, 16, 512, 64) == 3
    assert mla.mla_decode_item_cost(1, 1, 512, 64) == 2
    # the CUDA-core kernel splits pages evenly
    assert mla.mla_decode_item_cost(1, 128, 512, 64, dtype=torch.float32) == 0
    assert mla.mla_decode_item_cost(1, 8, 64, 16) == 0
    # more than 128 rows: row groups of 128 on the tensor-core kernel
    assert mla.mla_decode_item_cost(1, 256, 512, 64) == 5
    assert mla.mla_decode_item_cost(3, 24, 512, 64) == 4      # 72 rows
    # invalid dims
    assert mla.mla_decode_item_cost(0, 128, 512, 64) == -1
    # the host plan rejects a negative cost
    with pytest.raises(mla.MLAError):
        mla.mla_decode_split_plan(np.array([100], np.int32), 1, 8, 4, -1)


def test_row_groups_per_kernel():
    assert mla.mla_decode_row_groups(1, 128, 512, 64) == 1
    assert mla.mla_decode_row_groups(2, 128, 512, 64) == 2
    assert mla.mla_decode_row_groups(3, 64, 512, 64) == 2      # 192 rows: 128 + 64
    assert mla.mla_decode_row_groups(8, 128, 512, 64) == 8
    assert mla.mla_decode_row_groups(2, 128, 512, 64, dtype=torch.float32) == 1
    assert mla.mla_decode_row_groups(1, 8, 64, 16) == 1
    assert mla.mla_decode_row_groups(0, 8, 512, 64) == -1
    # the tensor-core path takes any row count for d_c = 512, d_r = 64, bf16
    assert mla.lib().mla_decode_path(2, 128, 512, 64, mla.MLA_BF16) == 1
    assert mla.lib().mla_decode_path(2, 128, 512, 64, mla.MLA_F32) == 0


def test_prefill_rows_and_host_checks():
    lib = mla.lib()
    # rows per sequence of the rebuilt K/V: 64 * max_blocks rounded up to 128
    assert [mla.mla_prefill_kv_rows(m) for m in (1, 2, 3, 64, 65)] == [128, 128, 256, 4096, 4224]
    assert mla.mla_prefill_kv_rows(0) == 0
    P = 16  # a non-null, 16-byte aligned dummy address; never dereferenced
    kv = dict(cache=P, dt=1, bt=P, sl=P, B=1, d_c=512, d_r=64, page=64, maxb=4, nb=4,
              wuk=P, wuv=P, H=8, d_h=128, k=P, v=P, kr=P, s=None)

    def call_kv(**kw):
        a = dict(kv, **kw)
        return lib.mla_prefill_kv(a["cache"], a["dt"], a["bt"], a["sl"], a["B"], a["d_c"], a["d_r"],
                                  a["page"], a["maxb"], a["nb"], a["wuk"], a["wuv"], a["H"], a["d_h"],
                                  a["k"], a["v"], a["kr"], a["s"])
    for bad in (dict(cache=None), dict(bt=None), dict(sl=None), dict(wuk=None), dict(wuv=P + 8),
                dict(k=None), dict(v=None), dict(kr=None), dict(B=-1), dict(H=0), dict(page=32),
                dict(maxb=0), dict(nb=0), dict(dt=7)):
        assert call_kv(**bad) == mla.MLA_ERR_INVALID_ARG, bad
    for unsup in (dict(dt=0), dict(d_c=256), dict(d_r=32), dict(d_h=64)):
        assert call_kv(**unsup) == mla.MLA_ERR_UNSUPPORTED, unsup
    assert call_kv(B=0) == mla.MLA_OK          # nothing to do, no device touched

    at = dict(qn=P, qr=P, dt=1, k=P, v=P, kr=P, sl=P, B=1, T_q=4, H=8, d_h=128, d_r=64, maxb=4,
              base=10000.0, scale=0.07, o=P, lse=None, s=None)

    def call_at(**kw):
        a = dict(at, **kw)
        return lib.mla_prefill_attention(a["qn"], a["qr"], a["dt"], a["k"], a["v"], a["kr"], a["sl"],
                                         a["B"], a["T_q"], a["H"], a["d_h"], a["d_r"], a["maxb"],
                                         a["base"], a["scale"], a["o"], a["lse"], a["s"])
    for bad in (dict(qn=None), dict(qr=None), dict(k=None), dict(v=P + 4), dict(kr=None),
                dict(sl=None), dict(o=None), dict(lse=P + 2), dict(T_q=0), dict(H=0), dict(B=-1),
                dict(maxb=0), dict(scale=0.0), dict(scale=-1.0), dict(scale=float("inf")),
                dict(base=0.0), dict(dt=7)):
        assert call_at(**bad) == mla.MLA_ERR_INVALID_ARG, bad
    for unsup in (dict(dt=0), dict(d_h=64), dict(d_r=16)):
        assert call_at(**unsup) == mla.MLA_ERR_UNSUPPORTED, unsup
    assert call_at(B=0) == mla.MLA_OK


def test_prefill_path_choice():
    use = mla.mla_prefill_use_rebuild
    # a single new token, or a handful, stay on the absorbed decode; a prompt goes to the rebuild
    assert use(1, 4096, 128) == 0 and use(16, 4096, 128) == 0 and use(64, 131072, 128) == 0
    assert use(4096, 4096, 128) == 1 and use(512, 32768, 128) == 1
    # at 128 heads the switch sits near 66 new tokens whatever the length
    for L in (4096, 32768, 131072):
        flips = [T for T in range(1, 200) if use(T, L, 128) == 1]
        assert flips and 55 <= flips[0] <= 80, (L, flips[:3])
        assert all(use(T, L, 128) == 1 for T in range(flips[0], 200))
    # fewer heads form fewer 128-row groups, so the absorbed decode stays longer
    assert use(64, 4096, 16) == 0 and use(1024, 4096, 16) == 1
    # shapes the rebuild kernels do not take, and invalid input
    assert use(4096, 4096, 128, d_h=64) == 0
    assert use(4096, 4096, 128, dtype=torch.float32) == 0
    assert use(0, 10, 8) == -1 and use(5, 4, 8) == -1 and use(1, 10, 0) == -1
