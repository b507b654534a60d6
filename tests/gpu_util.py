"""Helpers for the GPU tests: upload seeded inputs, call the library, compare.

Nothing here computes any part of the method; expected values always come
from the oracle package."""

from __future__ import annotations

import numpy as np
import torch

import head_latent_attention_28_b300 as mla
import mla_inputs as mi

# tolerances of the decode path (float accumulation over bfloat16 operands)
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_MAX_ABS = 1e-4


def bits_to_device(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def upload_decode(inp: mi.DecodeInputs, device="cuda"):
    return dict(
        q=bits_to_device(inp.q_bits, device),
        pool=bits_to_device(inp.pool_bits, device),
        bt=torch.from_numpy(inp.block_table).to(device),
        sl=torch.from_numpy(inp.seqlens).to(device),
    )


def run_decode(inp: mi.DecodeInputs, dev=None, workspace=None):
    dev = dev or upload_decode(inp)
    s = inp.spec
    o, lse = mla.mla_decode_paged(dev["q"], dev["pool"], dev["bt"], dev["sl"], d_c=s.d_c,
                                  softmax_scale=s.softmax_scale, causal=s.causal,
                                  workspace=workspace)
    st = mla.mla_check_status()
    assert st == mla.MLA_OK, mla.mla_status_string(st)
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_decode_close(got: np.ndarray, want: np.ndarray, max_abs=BF16_MAX_ABS,
                        rel_l2=BF16_REL_L2, what=""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e} > {max_abs}"
    assert rel <= rel_l2, f"{what}: rel L2 err {rel:.3e} > {rel_l2}"
    return float(err.max()), float(rel)
