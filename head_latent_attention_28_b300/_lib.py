"""ctypes binding of libmla.so: argument marshalling only.

Every function here takes torch tensors that already live on the GPU, checks
their shapes/dtypes, passes raw device pointers and sizes to the C ABI
(include/mla.h) and raises MLAError on a non-zero status.  There is no
fallback: if the library is missing the import of this module fails.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_CUDA = 3
MLA_ERR_WORKSPACE = 4
MLA_ERR_TIMEOUT = 5
MLA_ERR_BAD_INDEX = 6
MLA_ERR_BAD_RECORD = 7
MLA_F32 = 0
MLA_BF16 = 1
PAGE_SIZE = 64

# name -> (restype, argtypes); mirrors include/mla.h
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "mla_cache_append": (_I, [_P, _P, _I, _P, _P, _I, _P, _I, _I, _P, _I, _I, _I, _I, _I, _F, _P]),
    "mla_absorb_query": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P]),
    "mla_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "mla_decode_paged": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                              _P, _SZ, _P, _P, _P]),
    "mla_decode_paged_noalloc": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                      _I, _P, _P, _P]),
    "mla_decode_paged_partial": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                      _I, _P, _SZ, _P, _P, _P]),
    "mla_decode_combine": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                _P, _SZ, _P, _P, _P]),
    "mla_absorb_output": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "mla_merge_output_weights": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "mla_absorb_output_merged_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "mla_absorb_output_merged": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P, _P]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_last_cuda_error": (ctypes.c_char_p, []),
    "mla_check_status": (_I, [_P]),
    "mla_test_set_wait_fault": (_I, [_I, ctypes.c_uint]),
    "mla_test_force_splits": (_I, [_I]),
    "mla_version": (_I, []),
    "mla_decode_split_plan": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "mla_decode_item_cost": (_I, [_I, _I, _I, _I, _I]),
    "mla_decode_row_groups": (_I, [_I, _I, _I, _I, _I]),
    "mla_decode_step_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "mla_decode_step": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I,
                             _I, _I, _F, _I, _F, _P, _SZ, _P, _P, _P]),
    "mla_decode_num_workers": (_I, [_I, _I, _I, _I, _I, _I]),
    "mla_decode_path": (_I, [_I, _I, _I, _I, _I]),
    "mla_prefill_kv_rows": (_I, [_I]),
    "mla_prefill_use_rebuild": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "mla_prefill_kv": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P]),
    "mla_prefill_kv_chunk": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P,
                                  _P]),
    "mla_prefill_attention": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F,
                                   _P, _P, _P]),
}


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().mla_status_string(status).decode()
        if status == MLA_ERR_CUDA:
            msg += " (" + lib().mla_last_cuda_error().decode() + ")"
        super().__init__(f"{where}: {msg}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libmla.so not built ({path}); run "
                          "`python head_latent_attention_28_b300/build.py`")
    cdll = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(cdll, name)
        fn.restype, fn.argtypes = res, args
    return cdll


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MLAError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MLA_F32
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# --------------------------------------------------------------------------
# the four calls
# --------------------------------------------------------------------------

def mla_cache_append(c, k_rope, seq_ids, positions, block_table, kv_cache, *,
                     rope_base=10000.0, stream=None):
    """Write rows [c ; RoPE(k_rope)] of n_new tokens into the paged cache."""
    n_new, d_c = c.shape
    d_r = k_rope.shape[1]
    B, max_blocks = block_table.shape
    num_blocks, page, D = kv_cache.shape
    if D != d_c + d_r or k_rope.shape[0] != n_new or k_rope.dtype != c.dtype:
        raise ValueError("shape/dtype mismatch")
    st = lib().mla_cache_append(
        _dev(c, "c"), _dev(k_rope, "k_rope"), _dtype_code(c),
        _dev(seq_ids, "seq_ids", torch.int32), _dev(positions, "positions", torch.int32), n_new,
        _dev(block_table, "block_table", torch.int32), B, max_blocks,
        _dev(kv_cache, "kv_cache"), _dtype_code(kv_cache), num_blocks, page,
        d_c, d_r, float(rope_base), _stream(stream))
    _check(st, "mla_cache_append")


def mla_absorb_query(q_nope, q_rope, positions, w_uk, *, rope_base=10000.0,
                     q_dtype=None, out=None, stream=None):
    """q_lat = [W^UK_h^T q_nope ; RoPE(q_rope)]  -> [N, H, d_c + d_r]."""
    N, H, d_h = q_nope.shape
    d_r = q_rope.shape[2]
    d_c = w_uk.shape[1]
    if w_uk.shape[0] != H * d_h or q_rope.shape[:2] != (N, H):
        raise ValueError("shape mismatch")
    if q_nope.dtype != w_uk.dtype or q_rope.dtype != w_uk.dtype:
        raise TypeError("q_nope, q_rope and w_uk must share a dtype")
    if out is None:
        out = torch.empty((N, H, d_c + d_r), device=q_nope.device,
                          dtype=q_dtype or q_nope.dtype)
    st = lib().mla_absorb_query(
        _dev(q_nope, "q_nope"), _dev(q_rope, "q_rope"), _dev(positions, "positions", torch.int32),
        _dev(w_uk, "w_uk"), _dtype_code(w_uk), N, H, d_h, d_c, d_r, float(rope_base),
        _dev(out, "q_lat"), _dtype_code(out), _stream(stream))
    _check(st, "mla_absorb_query")
    return out


def mla_decode_workspace_size(B, T_q, H, d_c, d_r, dtype=torch.bfloat16) -> int:
    code = MLA_BF16 if dtype == torch.bfloat16 else MLA_F32
    return int(lib().mla_decode_workspace_size(B, T_q, H, d_c, d_r, code))


def alloc_workspace(B, T_q, H, d_c, d_r, dtype=torch.bfloat16, device="cuda"):
    n = mla_decode_workspace_size(B, T_q, H, d_c, d_r, dtype)
    if n == 0:
        raise ValueError("invalid decode dims")
    return torch.empty(n, dtype=torch.uint8, device=device)


def mla_decode_paged(q_lat, kv_cache, block_table, seqlens, *, d_c, softmax_scale,
                     causal=False, workspace=None, o_lat=None, lse=None, want_lse=True,
                     stream=None, stage="both"):
    """Latent-space attention of q_lat [B, T_q, H, D] over the paged cache.

    stage: "both" (mla_decode_paged), "partial" (mla_decode_paged_partial)
    or "combine" (mla_decode_combine).
    Returns (o_lat [B, T_q, H, d_c] float32, lse [B, T_q, H] float32 or None)."""
    B, T_q, H, D = q_lat.shape
    num_blocks, page, Dc = kv_cache.shape
    d_r = D - d_c
    if Dc != D or block_table.shape[0] != B or seqlens.shape != (B,):
        raise ValueError("shape mismatch")
    if q_lat.dtype != kv_cache.dtype:
        raise TypeError("q_lat and kv_cache must share a dtype")
    dev = q_lat.device
    if workspace is None:
        workspace = alloc_workspace(B, T_q, H, d_c, d_r, q_lat.dtype, dev)
    if o_lat is None:
        o_lat = torch.empty((B, T_q, H, d_c), device=dev, dtype=torch.float32)
    if lse is None and want_lse:
        lse = torch.empty((B, T_q, H), device=dev, dtype=torch.float32)
    L = lib()
    fn = (L.mla_decode_paged if stage == "both" else L.mla_decode_paged_partial if stage == "partial"
          else L.mla_decode_combine if stage == "combine" else None)
    if fn is None:
        raise ValueError(f"unknown stage {stage!r}")
    st = fn(
        _dev(q_lat, "q_lat"), _dev(kv_cache, "kv_cache"), _dtype_code(q_lat),
        _dev(block_table, "block_table", torch.int32), _dev(seqlens, "seqlens", torch.int32),
        B, T_q, H, d_c, d_r, page, block_table.shape[1], num_blocks,
        float(softmax_scale), 1 if causal else 0,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(o_lat, "o_lat", torch.float32),
        _dev(lse, "lse", torch.float32) if lse is not None else None, _stream(stream))
    _check(st, "mla_decode_paged" + ("" if stage == "both" else "_" + stage))
    return o_lat, lse


def mla_decode_paged_noalloc(q_lat, kv_cache, block_table, seqlens, *, d_c, softmax_scale,
                             causal=False, o_lat=None, lse=None, want_lse=True, stream=None):
    """mla_decode_paged with the library's own 64 MiB device scratch instead of a
    caller workspace (raises MLAError(MLA_ERR_WORKSPACE) for larger shapes), for
    callers that cannot get device memory at the call (no allocator of their
    own, or all free memory already given to the cache pool).  Calls that
    overlap on one device race on the scratch.  Returns (o_lat, lse or None)."""
    B, T_q, H, D = q_lat.shape
    num_blocks, page, Dc = kv_cache.shape
    d_r = D - d_c
    if Dc != D or block_table.shape[0] != B or seqlens.shape != (B,):
        raise ValueError("shape mismatch")
    if q_lat.dtype != kv_cache.dtype:
        raise TypeError("q_lat and kv_cache must share a dtype")
    dev = q_lat.device
    if o_lat is None:
        o_lat = torch.empty((B, T_q, H, d_c), device=dev, dtype=torch.float32)
    if lse is None and want_lse:
        lse = torch.empty((B, T_q, H), device=dev, dtype=torch.float32)
    st = lib().mla_decode_paged_noalloc(
        _dev(q_lat, "q_lat"), _dev(kv_cache, "kv_cache"), _dtype_code(q_lat),
        _dev(block_table, "block_table", torch.int32), _dev(seqlens, "seqlens", torch.int32),
        B, T_q, H, d_c, d_r, page, block_table.shape[1], num_blocks,
        float(softmax_scale), 1 if causal else 0,
        _dev(o_lat, "o_lat", torch.float32),
        _dev(lse, "lse", torch.float32) if lse is not None else None, _stream(stream))
    _check(st, "mla_decode_paged_noalloc")
    return o_lat, lse


def mla_absorb_output(o_lat, w_uv, w_o, *, out=None, stream=None):
    """out = W^O concat_h(W^UV_h o_lat[:, h])  -> [N, d] float32."""
    N, H, d_c = o_lat.shape
    HD, d_c2 = w_uv.shape
    d, HD2 = w_o.shape
    if d_c2 != d_c or HD2 != HD or HD % H:
        raise ValueError("shape mismatch")
    if w_uv.dtype != w_o.dtype:
        raise TypeError("w_uv and w_o must share a dtype")
    if out is None:
        out = torch.empty((N, d), device=o_lat.device, dtype=torch.float32)
    st = lib().mla_absorb_output(
        _dev(o_lat, "o_lat", torch.float32), _dev(w_uv, "w_uv"), _dev(w_o, "w_o"),
        _dtype_code(w_uv), N, H, HD // H, d_c, d, _dev(out, "out", torch.float32),
        _stream(stream))
    _check(st, "mla_absorb_output")
    return out


def mla_merge_output_weights(w_uv, w_o, H, *, out=None, stream=None):
    """W_m[j, h*d_c + c] = sum_v w_o[j, h*d_h + v] w_uv[h*d_h + v, c]  -> [d, H*d_c] bf16."""
    HD, d_c = w_uv.shape
    d, HD2 = w_o.shape
    if HD2 != HD or HD % H:
        raise ValueError("shape mismatch")
    if w_uv.dtype != w_o.dtype:
        raise TypeError("w_uv and w_o must share a dtype")
    if out is None:
        out = torch.empty((d, H * d_c), device=w_o.device, dtype=torch.bfloat16)
    st = lib().mla_merge_output_weights(_dev(w_uv, "w_uv"), _dev(w_o, "w_o"), _dtype_code(w_uv), H,
                                        HD // H, d_c, d, _dev(out, "w_merged", torch.bfloat16),
                                        _stream(stream))
    _check(st, "mla_merge_output_weights")
    return out


def mla_absorb_output_merged_workspace_size(N, H, d_c, d):
    return int(lib().mla_absorb_output_merged_workspace_size(N, H, d_c, d))


def mla_absorb_output_merged(o_lat, w_merged, *, workspace=None, out=None, stream=None):
    """out[n, j] = sum_{h,c} w_merged[j, h*d_c + c] o_lat[n, h, c]  -> [N, d] float32."""
    N, H, d_c = o_lat.shape
    d, K = w_merged.shape
    if K != H * d_c:
        raise ValueError("shape mismatch")
    need = mla_absorb_output_merged_workspace_size(N, H, d_c, d) if N > 0 else 0
    if workspace is None and N > 0:
        workspace = torch.empty(need, device=o_lat.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty((N, d), device=o_lat.device, dtype=torch.float32)
    st = lib().mla_absorb_output_merged(
        _dev(o_lat, "o_lat", torch.float32), _dev(w_merged, "w_merged"), _dtype_code(w_merged), N, H, d_c, d,
        _dev(workspace, "workspace") if workspace is not None else None,
        workspace.numel() * workspace.element_size() if workspace is not None else 0,
        _dev(out, "out", torch.float32), _stream(stream))
    _check(st, "mla_absorb_output_merged")
    return out


def mla_decode_split_plan(seqlens, T_q, max_blocks_per_seq, num_workers, item_cost=0):
    """Host helper: (first_worker, last_worker, total_pages) per sequence."""
    import numpy as np
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    B = sl.shape[0]
    first = np.empty(B, dtype=np.int32)
    last = np.empty(B, dtype=np.int32)
    total = ctypes.c_int64(0)
    st = lib().mla_decode_split_plan(sl.ctypes.data, B, T_q, max_blocks_per_seq, num_workers,
                                     item_cost, first.ctypes.data, last.ctypes.data,
                                     ctypes.addressof(total))
    _check(st, "mla_decode_split_plan")
    return first, last, int(total.value)


def mla_decode_item_cost(T_q, H, d_c, d_r, dtype=torch.bfloat16) -> int:
    """The split partition's per-item cost (pages) mla_decode_paged uses for a shape."""
    code = MLA_BF16 if dtype == torch.bfloat16 else MLA_F32
    return int(lib().mla_decode_item_cost(T_q, H, d_c, d_r, code))


def alloc_step_workspace(B, T_q, H, d_c, d_r, dtype=torch.bfloat16, device="cuda"):
    code = MLA_BF16 if dtype == torch.bfloat16 else MLA_F32
    n = int(lib().mla_decode_step_workspace_size(B, T_q, H, d_c, d_r, code))
    if n == 0:
        raise ValueError("invalid decode dims")
    return torch.empty(n, dtype=torch.uint8, device=device)


def mla_decode_step(q_nope, q_rope, w_uk, c_new, k_rope_new, kv_cache, block_table, seqlens, *,
                    softmax_scale, causal=False, rope_base=10000.0, workspace=None, o_lat=None,
                    lse=None, want_lse=True, stream=None):
    """One decode step: absorb q_nope/q_rope [B*T_q, H, .] into q_lat, append the new
    tokens' rows [c_new ; RoPE(k_rope_new)] at positions seqlens[b] - T_q + t, attend.
    Returns (o_lat [B, T_q, H, d_c] float32, lse [B, T_q, H] float32 or None)."""
    N, H, d_h = q_nope.shape
    d_r = q_rope.shape[2]
    num_blocks, page, D = kv_cache.shape
    d_c = D - d_r
    B = block_table.shape[0]
    if N % B or w_uk.shape != (H * d_h, d_c) or c_new.shape != (N, d_c) or \
            k_rope_new.shape != (N, d_r) or seqlens.shape != (B,):
        raise ValueError("shape mismatch")
    T_q = N // B
    if any(t.dtype != kv_cache.dtype for t in (q_nope, q_rope, w_uk, c_new, k_rope_new)):
        raise TypeError("all step inputs share the cache dtype")
    if workspace is None:
        workspace = alloc_step_workspace(B, T_q, H, d_c, d_r, kv_cache.dtype, kv_cache.device)
    if o_lat is None:
        o_lat = torch.empty((B, T_q, H, d_c), dtype=torch.float32, device=kv_cache.device)
    if lse is None and want_lse:
        lse = torch.empty((B, T_q, H), dtype=torch.float32, device=kv_cache.device)
    st = lib().mla_decode_step(
        _dev(q_nope, "q_nope"), _dev(q_rope, "q_rope"), _dev(w_uk, "w_uk"), d_h,
        _dev(c_new, "c_new"), _dev(k_rope_new, "k_rope_new"), _dev(kv_cache, "kv_cache"),
        _dtype_code(kv_cache), _dev(block_table, "block_table", torch.int32),
        _dev(seqlens, "seqlens", torch.int32), B, T_q, H, d_c, d_r, page, block_table.shape[1],
        num_blocks, float(softmax_scale), int(bool(causal)), float(rope_base),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(o_lat, "o_lat", torch.float32), _dev(lse, "lse", torch.float32) if lse is not None else None,
        _stream(stream))
    _check(st, "mla_decode_step")
    return o_lat, lse


def mla_decode_row_groups(T_q, H, d_c, d_r, dtype=torch.bfloat16) -> int:
    """How many row groups (work items over the same pages) a sequence's query rows form."""
    code = MLA_BF16 if dtype == torch.bfloat16 else MLA_F32
    return int(lib().mla_decode_row_groups(T_q, H, d_c, d_r, code))


def mla_decode_num_workers(B, T_q, H, d_c, d_r, dtype=torch.bfloat16) -> int:
    code = MLA_BF16 if dtype == torch.bfloat16 else MLA_F32
    return int(lib().mla_decode_num_workers(B, T_q, H, d_c, d_r, code))


# --------------------------------------------------------------------------
# prefill over rebuilt per-head keys and values
# --------------------------------------------------------------------------

def mla_prefill_kv_rows(max_blocks_per_seq) -> int:
    """Rows per sequence R of the rebuilt K/V buffers (64 * max_blocks rounded up to 128)."""
    return int(lib().mla_prefill_kv_rows(int(max_blocks_per_seq)))


def mla_prefill_use_rebuild(T_q, L, H, d_c=512, d_r=64, d_h=128, dtype=torch.bfloat16) -> int:
    """1 if a chunk of T_q tokens over L rows is expected to run faster on the
    rebuilt-key prefill path than on the absorbed decode, 0 if not, -1 if invalid."""
    code = MLA_BF16 if dtype == torch.bfloat16 else MLA_F32
    return int(lib().mla_prefill_use_rebuild(T_q, L, H, d_c, d_r, d_h, code))


def mla_prefill_kv(kv_cache, block_table, seqlens, w_uk, w_uv, *, H, out=None, stream=None, T_new=0):
    """Rebuild k_nope = W^UK_h c_s, v = W^UV_h c_s ([B, H, R, d_h] bf16) and copy
    k_rope = R_s k^R_s ([B, R, d_r]) for every cached row, or with T_new > 0
    only for the last T_new rows of each sequence into the caller's buffers
    `out` (mla_prefill_kv_chunk).  Returns (k_nope, v, k_rope)."""
    if T_new and out is None:
        raise ValueError("a chunk's rebuild writes into the buffers of the earlier chunks: pass out=")
    num_blocks, page, D = kv_cache.shape
    B, max_blocks = block_table.shape
    HD, d_c = w_uk.shape
    if HD % H or w_uv.shape != w_uk.shape or seqlens.shape != (B,):
        raise ValueError("shape mismatch")
    d_h, d_r = HD // H, D - d_c
    R = mla_prefill_kv_rows(max_blocks)
    if out is None:
        dev = kv_cache.device
        out = (torch.empty((B, H, R, d_h), device=dev, dtype=kv_cache.dtype),
               torch.empty((B, H, R, d_h), device=dev, dtype=kv_cache.dtype),
               torch.empty((B, R, d_r), device=dev, dtype=kv_cache.dtype))
    k_nope, v, k_rope = out
    st = lib().mla_prefill_kv_chunk(
        _dev(kv_cache, "kv_cache"), _dtype_code(kv_cache), _dev(block_table, "block_table", torch.int32),
        _dev(seqlens, "seqlens", torch.int32), B, d_c, d_r, page, max_blocks, num_blocks,
        _dev(w_uk, "w_uk", kv_cache.dtype), _dev(w_uv, "w_uv", kv_cache.dtype), H, d_h, int(T_new),
        _dev(k_nope, "k_nope", kv_cache.dtype), _dev(v, "v", kv_cache.dtype),
        _dev(k_rope, "k_rope", kv_cache.dtype), _stream(stream))
    _check(st, "mla_prefill_kv_chunk" if T_new else "mla_prefill_kv")
    return k_nope, v, k_rope


def mla_prefill_attention(q_nope, q_rope, k_nope, v, k_rope, seqlens, *, max_blocks_per_seq,
                          softmax_scale, rope_base=10000.0, o=None, lse=None, want_lse=True,
                          stream=None):
    """Causal attention of q [B, T_q, H, d_h (+ d_r unrotated)] over the rebuilt
    keys and values.  Returns (o [B, T_q, H, d_h] fp32, lse [B, T_q, H] or None)."""
    B, T_q, H, d_h = q_nope.shape
    d_r = q_rope.shape[3]
    if q_rope.shape[:3] != (B, T_q, H) or seqlens.shape != (B,):
        raise ValueError("shape mismatch")
    R = mla_prefill_kv_rows(max_blocks_per_seq)
    if k_nope.shape != (B, H, R, d_h) or v.shape != (B, H, R, d_h) or k_rope.shape != (B, R, d_r):
        raise ValueError("K/V buffers must be [B, H, R, d_h] and [B, R, d_r]")
    dev = q_nope.device
    if o is None:
        o = torch.empty((B, T_q, H, d_h), device=dev, dtype=torch.float32)
    if lse is None and want_lse:
        lse = torch.empty((B, T_q, H), device=dev, dtype=torch.float32)
    dt = q_nope.dtype
    st = lib().mla_prefill_attention(
        _dev(q_nope, "q_nope"), _dev(q_rope, "q_rope", dt), _dtype_code(q_nope),
        _dev(k_nope, "k_nope", dt), _dev(v, "v", dt), _dev(k_rope, "k_rope", dt),
        _dev(seqlens, "seqlens", torch.int32), B, T_q, H, d_h, d_r, int(max_blocks_per_seq),
        float(rope_base), float(softmax_scale), _dev(o, "o", torch.float32),
        _dev(lse, "lse", torch.float32) if lse is not None else None, _stream(stream))
    _check(st, "mla_prefill_attention")
    return o, lse


def mla_check_status(stream=None) -> int:
    """Wait for the stream and return (and clear) the device error status."""
    return int(lib().mla_check_status(_stream(stream)))


def mla_test_set_wait_fault(skip_load: int, wait_us: int = 1000) -> None:
    """Test hook: make tensor-core decode launches skip the load of page
    `skip_load` of split worker 0 with bounded waits of `wait_us` (0 turns
    the hook off); see include/mla.h."""
    _check(lib().mla_test_set_wait_fault(int(skip_load), int(wait_us)), "mla_test_set_wait_fault")


def mla_test_force_splits(num_workers: int) -> None:
    """Test knob: cap the decode split workers at num_workers (0: default);
    see include/mla.h."""
    _check(lib().mla_test_force_splits(int(num_workers)), "mla_test_force_splits")


def mla_status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()
