"""Failure detection on the GPU: a bounded device wait that runs out.

The test hook mla_test_set_wait_fault makes the tensor-core decode leave out
one page load of split worker 0 and lowers every bounded wait to a few
milliseconds.  The wait for that page must run out without a trap or a hang:
the kernel records MLA_ERR_TIMEOUT, drains its copies and MMAs, frees its
tensor memory and returns.  The context stays usable: with the hook off the
next call is MLA_OK and gives the same bits as before.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("skip", [1, 2])
def test_decode_wait_runs_out_then_the_next_call_is_clean(skip):
    import head_latent_attention_28_b300 as mla
    from gpu_util import assert_decode_close, run_decode, upload_decode
    # 512 pages over 74 split workers: worker 0 holds two pages
    spec = mi.DecodeSpec("wait_fault", seed=41, B=2, H=128, seqlens=(16384, 16383))
    inp = mi.make_decode_inputs(spec)
    dev = upload_decode(inp)
    o_ref, lse_ref = run_decode(inp, dev)
    kw = dict(d_c=spec.d_c, softmax_scale=spec.softmax_scale, causal=spec.causal)
    try:
        mla.mla_test_set_wait_fault(skip, 2000)
        mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], **kw)
        torch.cuda.synchronize()
        status = mla.mla_check_status()
    finally:
        mla.mla_test_set_wait_fault(0, 0)
    assert status == mla.MLA_ERR_TIMEOUT, mla.mla_status_string(status)
    # the device and the library are usable again, and nothing is left over
    o, lse = run_decode(inp, dev)
    assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)
    o64, lse64 = orc.decode_paged_logical(inp.q_bits, inp.cache_bits, inp.offsets, spec.d_c,
                                          spec.softmax_scale, spec.causal)
    assert_decode_close(o, o64, what="after the timeout")


def test_merge_without_its_partial_pass_reports_a_bad_record():
    import head_latent_attention_28_b300 as mla
    from gpu_util import upload_decode
    spec = mi.DecodeSpec("bad_record", seed=42, B=2, H=128, seqlens=(4096, 4096))
    inp = mi.make_decode_inputs(spec)
    dev = upload_decode(inp)
    ws = mla.alloc_workspace(spec.B, spec.T_q, spec.H, spec.d_c, spec.d_r, torch.bfloat16, "cuda")
    ws.zero_()
    # merge records (first worker, last worker) that no partial pass wrote:
    # the last before the first
    ws[:16].view(torch.int32).copy_(torch.tensor([5, 2, 5, 2], dtype=torch.int32))
    o, lse = mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], d_c=spec.d_c,
                                  softmax_scale=spec.softmax_scale, workspace=ws, stage="combine")
    assert mla.mla_check_status() == mla.MLA_ERR_BAD_RECORD
    assert torch.count_nonzero(o).item() == 0
