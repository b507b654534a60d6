"""The no-allocation decode entry point (mla_decode_paged_noalloc).

It runs the same kernels as mla_decode_paged but keeps the split workspace in
the library's own device scratch, for callers that cannot get device memory at
the call (a host with only the pointers it was handed, or a server that gave
all free memory to its cache pool).  On the same inputs both must give the same
bits, on two calls in a row (the scratch is reused, nothing in it has to start
at zero), and shapes whose workspace exceeds the scratch are refused.  This
file is collected last so that it also runs after every other GPU test.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _inputs(spec):
    from gpu_util import upload_decode
    inp = mi.make_decode_inputs(spec)
    return inp, upload_decode(inp)


@pytest.mark.parametrize("spec", [
    # tensor-core path (128 query rows), ragged lengths with a partial last page
    mi.DecodeSpec("noalloc_tc", seed=31, B=6, H=128, d_c=512, d_r=64,
                  seqlens=(1000, 4096, 65, 3000, 130, 2500)),
    # 32 query rows (padded to 128 in the MMAs), two query tokens with the causal mask
    mi.DecodeSpec("noalloc_few_rows", seed=32, B=5, H=16, T_q=2, d_c=512, d_r=64,
                  seqlens=(300, 2049, 64, 1500, 777), causal=True),
])
def test_noalloc_matches_workspace_entry_twice(spec):
    import head_latent_attention_28_b300 as mla
    inp, dev = _inputs(spec)
    assert mla.mla_decode_workspace_size(spec.B, spec.T_q, spec.H, spec.d_c, spec.d_r) <= SCRATCH_BYTES
    kw = dict(d_c=spec.d_c, softmax_scale=spec.softmax_scale, causal=spec.causal)
    o_ref, lse_ref = mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], **kw)
    for _ in range(2):
        o, lse = mla.mla_decode_paged_noalloc(dev["q"], dev["pool"], dev["bt"], dev["sl"], **kw)
        torch.cuda.synchronize()
        assert mla.mla_check_status() == mla.MLA_OK
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, lse_ref)


def test_noalloc_refuses_a_workspace_larger_than_its_scratch():
    import head_latent_attention_28_b300 as mla
    B, T_q, H, d_c, d_r = 256, 1, 128, 512, 64
    assert mla.mla_decode_workspace_size(B, T_q, H, d_c, d_r) > SCRATCH_BYTES
    q = torch.zeros((B, T_q, H, d_c + d_r), device="cuda", dtype=torch.bfloat16)
    pool = torch.zeros((4, 64, d_c + d_r), device="cuda", dtype=torch.bfloat16)
    bt = torch.zeros((B, 1), device="cuda", dtype=torch.int32)
    sl = torch.ones((B,), device="cuda", dtype=torch.int32)
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_paged_noalloc(q, pool, bt, sl, d_c=d_c, softmax_scale=0.1)
    assert ei.value.status == mla.MLA_ERR_WORKSPACE
