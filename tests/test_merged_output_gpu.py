"""Parity of the merged output projection (W^UV folded into W^O) with the
fp64 oracle: mla_merge_output_weights against the oracle's merge, and
mla_absorb_output_merged against the oracle's two projections (equal to the
merged form by associativity, pinned on the CPU)."""

import numpy as np
import pytest
import torch

import head_latent_attention_28_b300 as mla
import mla_inputs as mi
import oracle as orc

pytestmark = pytest.mark.gpu

# bf16 weights and a bf16 copy of o_lat, fp32 sums: the decode tolerance for
# bf16 data with fp32 accumulation
MAX_ABS, REL_L2 = 2e-2, 5e-3


def bf16_round(x):
    return mi.bf16_bits_to_f32(mi.f32_to_bf16_bits(np.asarray(x, np.float32))).reshape(np.shape(x))


def bf16_ulp(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - 7)


def weights(rng, H, d_h, d_c, d):
    """W^UV and W^O scaled so the projections keep unit-size numbers, as bf16 values."""
    w_uv = bf16_round(rng.standard_normal((H * d_h, d_c)) / np.sqrt(d_c))
    w_o = bf16_round(rng.standard_normal((d, H * d_h)) / np.sqrt(H * d_h))
    return w_uv, w_o


def dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)


def check_close(got, want, what):
    err = np.abs(got - want)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert np.all(np.isfinite(got)), what
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert rel <= REL_L2, f"{what}: rel L2 err {rel:.3e}"


@pytest.mark.parametrize("H,d_h,d_c,d", [(3, 64, 40, 200), (2, 128, 264, 136)])
def test_merged_weights_match_oracle(H, d_h, d_c, d):
    """Ragged tiles both ways (d rows per 128, d_c columns per 256)."""
    rng = np.random.default_rng(50 + d)
    w_uv, w_o = weights(rng, H, d_h, d_c, d)
    w_m = mla.mla_merge_output_weights(dev_bf16(w_uv), dev_bf16(w_o), H)
    torch.cuda.synchronize()
    assert mla.mla_check_status() == mla.MLA_OK
    got = w_m.double().cpu().numpy()
    want = orc.merge_output_weights(w_uv, w_o, H)
    # fp32 sums of exact bf16 products, rounded once to bf16
    assert np.all(np.abs(got - want) <= bf16_ulp(want) + 1e-6), np.abs(got - want).max()


def test_merged_weights_full_shape_sampled():
    """H=128, d_h=128, d_c=512, d=5120: sampled rows of three heads against
    the oracle's merge of the same slices (the merge is separable by row and
    by head)."""
    rng = np.random.default_rng(53)
    H, d_h, d_c, d = 128, 128, 512, 5120
    w_uv, w_o = weights(rng, H, d_h, d_c, d)
    w_m = mla.mla_merge_output_weights(dev_bf16(w_uv), dev_bf16(w_o), H)
    torch.cuda.synchronize()
    assert mla.mla_check_status() == mla.MLA_OK
    rows = np.concatenate([[0, 127, 128, 2559, 5119], rng.choice(d, 11, replace=False)])
    for hh in (0, 77, 127):
        want = orc.merge_output_weights(w_uv[hh * d_h:(hh + 1) * d_h], w_o[rows, hh * d_h:(hh + 1) * d_h], 1)
        got = w_m[torch.from_numpy(rows).cuda(), hh * d_c:(hh + 1) * d_c].double().cpu().numpy()
        assert np.all(np.abs(got - want) <= bf16_ulp(want) + 1e-6), (hh, np.abs(got - want).max())


@pytest.mark.parametrize("N", [1, 5, 130])
def test_merged_output_matches_oracle(N):
    """Ragged rows (130 = one full 128-row tile and 2 more), ragged output
    columns (264 = 256 + 8) and K = H * d_c split across the grid."""
    rng = np.random.default_rng(60 + N)
    H, d_h, d_c, d = 4, 64, 64, 264
    w_uv, w_o = weights(rng, H, d_h, d_c, d)
    o_lat = rng.standard_normal((N, H, d_c)).astype(np.float32)
    w_m = mla.mla_merge_output_weights(dev_bf16(w_uv), dev_bf16(w_o), H)
    out = mla.mla_absorb_output_merged(torch.from_numpy(o_lat).cuda(), w_m)
    torch.cuda.synchronize()
    assert mla.mla_check_status() == mla.MLA_OK
    check_close(out.double().cpu().numpy(), orc.absorb_output(o_lat, w_uv, w_o), f"N={N}")


def test_merged_output_full_shape_and_against_unmerged():
    """N=32 decode rows at H=128, d_h=128, d_c=512, d=5120: the merged path
    against the oracle and against the library's unmerged path; the merged
    path is deterministic (fixed split order)."""
    rng = np.random.default_rng(61)
    N, H, d_h, d_c, d = 32, 128, 128, 512, 5120
    w_uv, w_o = weights(rng, H, d_h, d_c, d)
    o_lat = rng.standard_normal((N, H, d_c)).astype(np.float32)
    o_dev = torch.from_numpy(o_lat).cuda()
    w_m = mla.mla_merge_output_weights(dev_bf16(w_uv), dev_bf16(w_o), H)
    ws = torch.empty(mla.mla_absorb_output_merged_workspace_size(N, H, d_c, d), dtype=torch.uint8, device="cuda")
    out1 = mla.mla_absorb_output_merged(o_dev, w_m, workspace=ws)
    out2 = mla.mla_absorb_output_merged(o_dev, w_m, workspace=ws)
    un = mla.mla_absorb_output(o_dev, dev_bf16(w_uv), dev_bf16(w_o))
    torch.cuda.synchronize()
    assert mla.mla_check_status() == mla.MLA_OK
    assert torch.equal(out1, out2)
    want = orc.absorb_output(o_lat, w_uv, w_o)
    check_close(out1.double().cpu().numpy(), want, "merged")
    check_close(out1.double().cpu().numpy(), un.double().cpu().numpy(), "merged vs unmerged")


def test_merged_output_host_errors():
    H, d_c, d = 2, 64, 128
    o = torch.zeros((3, H, d_c), device="cuda")
    w32 = torch.zeros((d, H * d_c), device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.mla_absorb_output_merged(o, w32)             # fp32 weights: no tensor-core form
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED
    w16 = w32.to(torch.bfloat16)
    need = mla.mla_absorb_output_merged_workspace_size(3, H, d_c, d)
    assert need > 0
    with pytest.raises(mla.MLAError) as e:
        mla.mla_absorb_output_merged(o, w16, workspace=torch.empty(need - 256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == mla.MLA_ERR_WORKSPACE
    with pytest.raises(mla.MLAError) as e:                # d_h % 64 != 0
        mla.mla_merge_output_weights(torch.zeros((H * 32, d_c), dtype=torch.bfloat16, device="cuda"),
                                     torch.zeros((d, H * 32), dtype=torch.bfloat16, device="cuda"), H)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED
    assert mla.mla_check_status() == mla.MLA_OK


@pytest.mark.parametrize("N", [1, 130])
def test_unmerged_tensor_core_path_ragged(N):
    """mla_absorb_output with bf16 weights runs on the tensor cores with
    o_lat and o split into bf16 value + remainder: about fp32 accuracy on
    ragged rows (130), ragged output columns (264) and a K split."""
    rng = np.random.default_rng(70 + N)
    H, d_h, d_c, d = 4, 64, 64, 264
    w_uv, w_o = weights(rng, H, d_h, d_c, d)
    o_lat = rng.standard_normal((N, H, d_c)).astype(np.float32)
    out = mla.mla_absorb_output(torch.from_numpy(o_lat).cuda(), dev_bf16(w_uv), dev_bf16(w_o))
    torch.cuda.synchronize()
    assert mla.mla_check_status() == mla.MLA_OK
    want = orc.absorb_output(o_lat, w_uv, w_o)
    np.testing.assert_allclose(out.double().cpu().numpy(), want, rtol=0, atol=5e-5)
