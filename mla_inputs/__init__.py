"""Seeded synthetic inputs for MLA latent-cache decode.

This module is the one piece of code that both the CUDA path and the oracle
consume.  It draws random numbers, rounds them to the storage type and lays
them out; it holds none of the method's arithmetic (no projection, rotation,
score, softmax or value sum).

Workloads follow the shapes of the multi-head latent attention pages
(DeepSeek-V2 scale: n_h = 128 heads, latent d_c = 512, decoupled rotary key
d^R_h = 64, so a cached row has 576 numbers; "Multi-head latent attention
(MLA)", ai-knowledge-tree, section 2).  The pages use no public dataset: all
values are i.i.d. normal draws from numpy's PCG64 generator, in a fixed
documented order.

Draw order for a decode workload (one ``default_rng(seed)``):
  1. sequence lengths (only for ragged workloads: ``integers(lo, hi, B,
     endpoint=True)``),
  2. the block permutation (``permutation(num_blocks)``; sequence b takes the
     next ceil(L_b / 64) ids in order),
  3. the latent query q [B, T_q, H, D] (``standard_normal``, float32),
  4. the cache rows of all sequences, concatenated in token order
     [sum L_b, D] (``standard_normal``, float32),
  5. for the outlier workload, a per-token mask ``random(sum L_b) < frac``;
     masked rows are multiplied by ``outlier_scale`` (a power of two, so the
     order of scaling and rounding does not matter).
Values are then rounded to bfloat16 with round-to-nearest-even, once.  Pool
blocks that hold no sequence data, and the rows of a last block past the
sequence end, are filled with NaN so that any read of them shows up.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE = 64                       # tokens per cache block
BF16_NAN = np.uint16(0x7FC0)    # quiet NaN in bfloat16


# --------------------------------------------------------------------------
# storage-type conversion (input formatting, not method arithmetic)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns.  Inputs are finite (normal draws)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    """Shape of one paged latent-cache decode workload."""
    name: str
    seed: int
    B: int
    H: int
    T_q: int = 1
    d_c: int = 512
    d_r: int = 64
    seqlen: Optional[int] = None          # every sequence this long, or
    seqlen_range: Optional[tuple] = None  # (lo, hi) inclusive, drawn per sequence
    seqlens: Optional[tuple] = None       # explicit lengths (small test cases)
    num_blocks: Optional[int] = None      # pool size; default = blocks needed
    causal: bool = False
    outlier_frac: float = 0.0
    outlier_scale: float = 8.0
    softmax_scale: float = 1.0 / math.sqrt(192.0)

    @property
    def D(self) -> int:
        return self.d_c + self.d_r


@dataclasses.dataclass(frozen=True)
class FullModelSpec:
    """Tiny full-layer workload: projections, cache, absorbed decode, output."""
    name: str
    seed: int
    d: int
    H: int
    d_h: int
    d_c: int
    d_r: int
    n_cached: int          # tokens already in the cache
    n_query: int = 1       # new tokens (appended, then attending)
    rope_base: float = 10000.0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_h + self.d_r)

    @property
    def n_tokens(self) -> int:
        return self.n_cached + self.n_query


# The five workloads the pages' shapes call for.  Scale 1/sqrt(192) is the
# V2-scale head (d_h = 128 plus d^R_h = 64); the workloads that do not state
# a scale reuse it.
TINY_FULL_MODEL = FullModelSpec("tiny_full_model_fp32", seed=0, d=256, H=8,
                                d_h=32, d_c=64, d_r=16, n_cached=128)
V2_DECODE = DecodeSpec("v2_decode_b32_l4096", seed=1, B=32, H=128, seqlen=4096)
RAGGED_SERVING = DecodeSpec("ragged_b128_l512_16384", seed=2, B=128, H=128,
                            seqlen_range=(512, 16384), num_blocks=40000)
LONG_CONTEXT = DecodeSpec("long_b4_l131072", seed=3, B=4, H=128,
                          seqlen=131072, outlier_frac=0.01)
FEW_HEAD_MTP = DecodeSpec("few_head_b64_h16_tq2", seed=4, B=64, H=16, T_q=2,
                          seqlen_range=(2048, 8192), causal=True)

DECODE_WORKLOADS = {s.name: s for s in (V2_DECODE, RAGGED_SERVING,
                                        LONG_CONTEXT, FEW_HEAD_MTP)}


# --------------------------------------------------------------------------
# decode inputs
# --------------------------------------------------------------------------

@dataclasses.dataclass
class DecodeInputs:
    spec: DecodeSpec
    seqlens: np.ndarray        # int32 [B]
    offsets: np.ndarray        # int64 [B+1], row offsets into cache_bits
    block_table: np.ndarray    # int32 [B, max_blocks]; unused entries = -1
    q_bits: np.ndarray         # uint16 [B, T_q, H, D]
    cache_bits: np.ndarray     # uint16 [sum L_b, D]  logical rows, token order
    pool_bits: np.ndarray      # uint16 [num_blocks, PAGE, D]  paged copy

    @property
    def num_blocks(self) -> int:
        return self.pool_bits.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    def seq_rows(self, b: int) -> np.ndarray:
        """bfloat16 bits of sequence b's cache rows [L_b, D]."""
        return self.cache_bits[self.offsets[b]:self.offsets[b + 1]]


def draw_seqlens(rng: np.random.Generator, spec: DecodeSpec) -> np.ndarray:
    if spec.seqlens is not None:
        return np.asarray(spec.seqlens, dtype=np.int32)
    if spec.seqlen is not None:
        return np.full(spec.B, spec.seqlen, dtype=np.int32)
    lo, hi = spec.seqlen_range
    return rng.integers(lo, hi, size=spec.B, endpoint=True).astype(np.int32)


def make_decode_inputs(spec: DecodeSpec, build_pool: bool = True) -> DecodeInputs:
    rng = np.random.default_rng(spec.seed)
    D = spec.D
    seqlens = draw_seqlens(rng, spec)                                  # 1
    if np.any(seqlens < spec.T_q):
        raise ValueError("every sequence must hold at least T_q rows")
    blocks_needed = (seqlens.astype(np.int64) + PAGE - 1) // PAGE
    total_blocks = int(blocks_needed.sum())
    num_blocks = spec.num_blocks if spec.num_blocks is not None else total_blocks
    if num_blocks < total_blocks:
        raise ValueError("pool too small for the drawn sequence lengths")
    perm = rng.permutation(num_blocks).astype(np.int32)               # 2
    max_blocks = int(blocks_needed.max())
    block_table = np.full((spec.B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(spec.B):
        nb = int(blocks_needed[b])
        block_table[b, :nb] = perm[pos:pos + nb]
        pos += nb

    q = rng.standard_normal((spec.B, spec.T_q, spec.H, D), dtype=np.float32)  # 3
    q_bits = f32_to_bf16_bits(q).reshape(q.shape)
    del q

    offsets = np.zeros(spec.B + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(seqlens.astype(np.int64))
    n_rows = int(offsets[-1])
    # draw and round in slabs to bound host memory for the 1.1M-row workload
    cache_bits = np.empty((n_rows, D), dtype=np.uint16)
    slab = 1 << 18
    for r0 in range(0, n_rows, slab):                                 # 4
        r1 = min(n_rows, r0 + slab)
        x = rng.standard_normal((r1 - r0, D), dtype=np.float32)
        cache_bits[r0:r1] = f32_to_bf16_bits(x).reshape(x.shape)
    if spec.outlier_frac > 0.0:                                       # 5
        mask = rng.random(n_rows) < spec.outlier_frac
        idx = np.nonzero(mask)[0]
        vals = bf16_bits_to_f32(cache_bits[idx]) * np.float32(spec.outlier_scale)
        cache_bits[idx] = f32_to_bf16_bits(vals).reshape(vals.shape)

    pool_bits = np.empty((0, PAGE, D), dtype=np.uint16)
    if build_pool:
        pool_bits = np.full((num_blocks, PAGE, D), BF16_NAN, dtype=np.uint16)
        for b in range(spec.B):
            rows = cache_bits[offsets[b]:offsets[b + 1]]
            L = rows.shape[0]
            for j in range(int(blocks_needed[b])):
                n = min(PAGE, L - j * PAGE)
                pool_bits[block_table[b, j], :n] = rows[j * PAGE:j * PAGE + n]
    return DecodeInputs(spec, seqlens, offsets, block_table, q_bits,
                        cache_bits, pool_bits)


# --------------------------------------------------------------------------
# full-model inputs (fp32)
# --------------------------------------------------------------------------

@dataclasses.dataclass
class FullModelInputs:
    spec: FullModelSpec
    h: np.ndarray      # float32 [n_tokens, d]      token representations
    W_dkv: np.ndarray  # float32 [d_c, d]           latent down-projection
    W_kr: np.ndarray   # float32 [d_r, d]           decoupled rotary key
    W_q: np.ndarray    # float32 [H*d_h, d]         content query
    W_qr: np.ndarray   # float32 [H*d_r, d]         rotary query
    W_uk: np.ndarray   # float32 [H*d_h, d_c]       key up-projection
    W_uv: np.ndarray   # float32 [H*d_h, d_c]       value up-projection
    W_o: np.ndarray    # float32 [d, H*d_h]         output projection


def make_full_model_inputs(spec: FullModelSpec) -> FullModelInputs:
    """h ~ N(0,1); every weight ~ N(0, 1/fan_in), fan_in = its column count.

    Drawn in float64 in the order h, W_dkv, W_kr, W_q, W_qr, W_uk, W_uv, W_o,
    then stored as float32 (the float32 values are the inputs)."""
    rng = np.random.default_rng(spec.seed)
    H, d, d_h, d_c, d_r = spec.H, spec.d, spec.d_h, spec.d_c, spec.d_r

    def w(rows, cols):
        return (rng.standard_normal((rows, cols)) / math.sqrt(cols)).astype(np.float32)

    h = rng.standard_normal((spec.n_tokens, d)).astype(np.float32)
    return FullModelInputs(spec, h,
                           W_dkv=w(d_c, d), W_kr=w(d_r, d), W_q=w(H * d_h, d),
                           W_qr=w(H * d_r, d), W_uk=w(H * d_h, d_c),
                           W_uv=w(H * d_h, d_c), W_o=w(d, H * d_h))


def shuffled_block_table(rng: np.random.Generator, n_tokens: int, num_blocks: int):
    """One sequence of n_tokens rows on a shuffled pool of num_blocks blocks."""
    nb = (n_tokens + PAGE - 1) // PAGE
    if nb > num_blocks:
        raise ValueError("pool too small")
    perm = rng.permutation(num_blocks).astype(np.int32)
    return perm[:nb].reshape(1, nb).copy()


# --------------------------------------------------------------------------
# prefill inputs (a chunk of T_q new tokens per sequence over the paged cache)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class PrefillSpec:
    """Prefill over per-head keys and values rebuilt from the latent cache."""
    name: str
    seed: int
    B: int
    H: int
    T_q: int
    seqlen: Optional[int] = None
    seqlens: Optional[tuple] = None
    d_h: int = 128
    d_c: int = 512
    d_r: int = 64
    rope_base: float = 10000.0
    softmax_scale: float = 1.0 / math.sqrt(192.0)


# DeepSeek-V2-scale prefill of one 4096-token prompt
V2_PREFILL = PrefillSpec("prefill_b1_t4096_h128", seed=5, B=1, H=128, T_q=4096, seqlen=4096)
PREFILL_WORKLOADS = {V2_PREFILL.name: V2_PREFILL}


def prefill_kv_rows(max_blocks: int) -> int:
    """Rows per sequence of the rebuilt K/V buffers: 64 * max_blocks rounded up to 128."""
    return (max_blocks * PAGE + 127) // 128 * 128


@dataclasses.dataclass
class PrefillInputs:
    spec: PrefillSpec
    cache: DecodeInputs          # seqlens, offsets, block_table, cache_bits, pool_bits
    q_nope_bits: np.ndarray      # uint16 [B, T_q, H, d_h]
    q_rope_bits: np.ndarray      # uint16 [B, T_q, H, d_r]  (not rotated)
    w_uk_bits: np.ndarray        # uint16 [H * d_h, d_c]
    w_uv_bits: np.ndarray        # uint16 [H * d_h, d_c]
    # standalone key/value buffers for the attention call alone (with_kv=True):
    # [B, H, R, d_h], [B, H, R, d_h], [B, R, d_r]; rows >= L_b are zero
    k_nope_bits: Optional[np.ndarray] = None
    v_bits: Optional[np.ndarray] = None
    k_rope_bits: Optional[np.ndarray] = None


def make_prefill_inputs(spec: PrefillSpec, with_kv: bool = False) -> PrefillInputs:
    """The cache comes from make_decode_inputs with one head (draws 1, 2, 4 of
    that recipe with the spec's seed; its one-head query is unused).  Then, from
    default_rng(seed + 7919): q_nope, q_rope ~ N(0, 1); W^UK, W^UV ~
    N(0, 1/d_c); and with with_kv the standalone buffers k_nope, v, k_rope ~
    N(0, 1), in that order, all float32 rounded once to bfloat16."""
    cache = make_decode_inputs(DecodeSpec(spec.name, spec.seed, spec.B, 1, T_q=spec.T_q,
                                          d_c=spec.d_c, d_r=spec.d_r, seqlen=spec.seqlen,
                                          seqlens=spec.seqlens))
    rng = np.random.default_rng(spec.seed + 7919)
    B, T, H = spec.B, spec.T_q, spec.H

    def draw(shape, scale=1.0):
        x = rng.standard_normal(shape, dtype=np.float32)
        if scale != 1.0:
            x = x * np.float32(scale)
        return f32_to_bf16_bits(x).reshape(shape)

    q_nope = draw((B, T, H, spec.d_h))
    q_rope = draw((B, T, H, spec.d_r))
    w_uk = draw((H * spec.d_h, spec.d_c), 1.0 / math.sqrt(spec.d_c))
    w_uv = draw((H * spec.d_h, spec.d_c), 1.0 / math.sqrt(spec.d_c))
    inp = PrefillInputs(spec, cache, q_nope, q_rope, w_uk, w_uv)
    if with_kv:
        R = prefill_kv_rows(cache.max_blocks)
        k = draw((B, H, R, spec.d_h))
        v = draw((B, H, R, spec.d_h))
        kr = draw((B, R, spec.d_r))
        for b in range(B):
            L = int(cache.seqlens[b])
            k[b, :, L:] = 0
            v[b, :, L:] = 0
            kr[b, L:] = 0
        inp.k_nope_bits, inp.v_bits, inp.k_rope_bits = k, v, kr
    return inp


# --------------------------------------------------------------------------
# output projection inputs (the attended latent and the value / output weights)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class OutProjSpec:
    """W^UV then W^O (or the two merged) applied to N attended latents."""
    name: str
    seed: int
    N: int
    H: int = 128
    d_h: int = 128
    d_c: int = 512
    d: int = 5120


# one decode step of the ragged serving batch (128 sequences x 1 token) at
# the pages' model width d = 5120
OUT_PROJ = OutProjSpec("out_proj_n128_h128_d5120", seed=9, N=128)
OUT_PROJ_WORKLOADS = {OUT_PROJ.name: OUT_PROJ}


@dataclasses.dataclass
class OutProjInputs:
    spec: OutProjSpec
    o_lat: np.ndarray           # float32 [N, H, d_c]
    w_uv_bits: np.ndarray       # uint16 [H * d_h, d_c]
    w_o_bits: np.ndarray        # uint16 [d, H * d_h]


def make_out_proj_inputs(spec: OutProjSpec) -> OutProjInputs:
    """From default_rng(seed): o_lat ~ N(0, 1) float32; W^UV ~ N(0, 1/d_c) and
    W^O ~ N(0, 1/(H d_h)) rounded once to bfloat16, in that order (unit-size
    numbers through both projections)."""
    rng = np.random.default_rng(spec.seed)
    o_lat = rng.standard_normal((spec.N, spec.H, spec.d_c), dtype=np.float32)
    w_uv = rng.standard_normal((spec.H * spec.d_h, spec.d_c), dtype=np.float32) * np.float32(1.0 / math.sqrt(spec.d_c))
    w_o = rng.standard_normal((spec.d, spec.H * spec.d_h), dtype=np.float32) * np.float32(
        1.0 / math.sqrt(spec.H * spec.d_h))
    return OutProjInputs(spec, o_lat, f32_to_bf16_bits(w_uv).reshape(w_uv.shape),
                         f32_to_bf16_bits(w_o).reshape(w_o.shape))
