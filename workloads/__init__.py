"""Seeded synthetic inputs for the TND attention-gradient workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (through ``bench.py`` and the GPU
tests) and the fp64 oracle (through the tests) take their inputs from here, so
the two sides see bit-identical values.

Workloads (shapes follow the TND cases of the Ascend FlashAttention grad pages,
"aclnnFlashAttentionUnpaddingScoreGrad" constraints section: T total tokens,
N heads, D head dim, per-sequence lengths given as cumulative offsets):

=====================  =====================================================
name                   shape
=====================  =====================================================
tiny_varlen_fp16       fp16, seqlens q=kv=[37,64], Nq=Nkv=2, D=64, no mask
causal_varlen_bf16     bf16, 8 seqs of U[256,2048], Nq=Nkv=16, D=128, causal
gqa_causal_bf16        bf16, seqs [4096,8192,8192,12288], Nq=32, Nkv=8, causal
window_dropout_bf16    bf16, 8x8192, Nq=16, Nkv=4, band pre=1024 next=0,
                       keepProb 0.9 with a Bernoulli(0.9) packed keep-bitmask
long_causal_sink_bf16  bf16, 1x32768, Nq=Nkv=8, causal, per-head sink ~ N(0,1)
=====================  =====================================================

Recipe: every tensor element is an independent N(0,1) draw from numpy's PCG64
generator seeded by ``SeedSequence([seed, stream_id])``; the fp64 draw is
rounded to fp32 (round-to-nearest-even) and then to the 16-bit dtype (RNE).
The dropout keep-bits are Bernoulli(p_keep) draws (a uniform 16-bit integer
compared against round(p_keep * 65536)), packed 8 bits per byte, least
significant bit first, over the flattened (sequence, q-head, q-row, kv-row)
index.  Sequence lengths of the varlen case are uniform integers in
[256, 2048].

Attention-mask matrices (sparseMode 0 / 1 cases): uint8 [S1Max, S2Max], each
element 1 (masked) with probability ``amask_density`` (uniform 16-bit integer
against round(density * 65536)); every row i with i % 97 == 5 is fully
masked, so rows that keep no key occur.  Prefix values (sparseMode 6) are
given with the workload.

pse (positional bias), stored as [B or 1, Nq, 1024, S2Max], the last 1024
rows of each sequence's bias: "random" draws every stored element N(0, 0.25);
"alibi" stores slope_h * (j - i) with slope_h = 2^-(4 + h) (zero beyond the
sequence's columns); both are rounded to the dtype like the other tensors.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

# stream ids of the independent tensors drawn for one workload
_STREAM = {"seqlens": 1, "q": 2, "k": 3, "v": 4, "dy": 5, "sink": 6, "mask": 7, "amask": 8, "pse": 9, "slopes": 10}

BASE_SEED = 20261202


@dataclasses.dataclass
class Workload:
    """Static description of one synthetic problem (no tensors)."""

    name: str
    dtype: str                 # "f16" | "bf16" | "f32"
    seqlens_q: List[int]
    seqlens_kv: List[int]
    nq: int
    nkv: int
    d: int
    scale: float
    keep_prob: float = 1.0
    pre_tokens: int = 2147483647
    next_tokens: int = 2147483647
    sparse_mode: int = 0
    has_sink: bool = False
    seed: int = BASE_SEED
    amask_density: float = 0.0             # > 0: an attention-mask matrix is drawn
    prefix: Optional[List[int]] = None     # prefixOptional (sparseMode 6)
    pse_kind: str = ""                     # "", "random" or "alibi" (stores), "slopes" (pseType 2 / 3)
    pse_batch: int = 1                     # 1 (shared) or B
    pse_type: int = 1                      # pseType 0 / 1
    value_d: int = 0                       # head dim of value / dy / output (0: d)

    @property
    def dv(self) -> int:
        return self.value_d or self.d

    @property
    def batch(self) -> int:
        return len(self.seqlens_q)

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_q)]).astype(np.int64)

    @property
    def cu_kv(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_kv)]).astype(np.int64)

    @property
    def tq(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def tkv(self) -> int:
        return int(sum(self.seqlens_kv))

    def mask_bits(self) -> int:
        """Number of keep-bits in the packed dropout mask."""
        return int(sum(self.nq * sq * skv for sq, skv in zip(self.seqlens_q, self.seqlens_kv)))

    def describe(self) -> Dict:
        return {
            "workload": self.name, "dtype": self.dtype, "B": self.batch,
            "seqlens_q": list(self.seqlens_q) if self.batch <= 16 else f"{self.batch} seqs",
            "T": self.tq, "Nq": self.nq, "Nkv": self.nkv, "D": self.d,
            "scale": self.scale, "keep_prob": self.keep_prob,
            "pre_tokens": self.pre_tokens, "next_tokens": self.next_tokens,
            "sparse_mode": self.sparse_mode, "sink": self.has_sink, "seed": self.seed,
            **({"atten_mask_density": self.amask_density} if self.amask_density > 0 else {}),
            **({"prefix": list(self.prefix)} if self.prefix is not None else {}),
        }


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAM[stream]])))


def varlen_lengths(seed: int, count: int, lo: int, hi: int) -> List[int]:
    """``count`` integers uniform in [lo, hi] (inclusive)."""
    return [int(x) for x in _rng(seed, "seqlens").integers(lo, hi + 1, size=count)]


def workload(name: str, seed: Optional[int] = None) -> Workload:
    """The named workload; ``seed`` defaults to BASE_SEED + its index."""
    index = WORKLOAD_NAMES.index(name)
    s = BASE_SEED + index if seed is None else seed
    if name == "tiny_varlen_fp16":
        return Workload(name, "f16", [37, 64], [37, 64], 2, 2, 64, 1.0 / math.sqrt(64), seed=s)
    if name == "causal_varlen_bf16":
        lens = varlen_lengths(s, 8, 256, 2048)
        return Workload(name, "bf16", lens, list(lens), 16, 16, 128, 1.0 / math.sqrt(128),
                        sparse_mode=3, seed=s)
    if name == "gqa_causal_bf16":
        lens = [4096, 8192, 8192, 12288]
        return Workload(name, "bf16", lens, list(lens), 32, 8, 128, 1.0 / math.sqrt(128),
                        sparse_mode=3, seed=s)
    if name == "window_dropout_bf16":
        lens = [8192] * 8
        return Workload(name, "bf16", lens, list(lens), 16, 4, 128, 1.0 / math.sqrt(128),
                        keep_prob=0.9, pre_tokens=1024, next_tokens=0, sparse_mode=4, seed=s)
    if name == "long_causal_sink_bf16":
        return Workload(name, "bf16", [32768], [32768], 8, 8, 128, 1.0 / math.sqrt(128),
                        sparse_mode=3, has_sink=True, seed=s)
    raise KeyError(name)


WORKLOAD_NAMES = [
    "tiny_varlen_fp16",
    "causal_varlen_bf16",
    "gqa_causal_bf16",
    "window_dropout_bf16",
    "long_causal_sink_bf16",
]


# ----------------------------------------------------------------------------
# rounding of fp64 draws to the storage dtype
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round-to-nearest-even); returns the uint16 patterns."""
    u = x32.astype(np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    rounded = u + np.uint32(0x7FFF) + lsb
    nan = np.isnan(x32)
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_to_dtype(x64: np.ndarray, dtype: str):
    """Round fp64 values to ``dtype``.

    Returns ``(stored, exact64)``: the storage array (uint16 bit patterns for
    bf16, float16 for f16, float32 for f32) and the exact fp64 value of every
    stored element.
    """
    x32 = x64.astype(np.float32)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x32)
        return bits, bf16_bits_to_f64(bits)
    if dtype == "f16":
        h = x32.astype(np.float16)
        return h, h.astype(np.float64)
    if dtype == "f32":
        return x32, x32.astype(np.float64)
    raise ValueError(dtype)


def normal(seed: int, stream: str, shape, dtype: str):
    """N(0,1) tensor rounded to ``dtype``: ``(stored, exact64)``."""
    x = _rng(seed, stream).standard_normal(size=shape, dtype=np.float64)
    return round_to_dtype(x, dtype)


def dropout_mask(seed: int, nbits: int, p_keep: float, chunk_bits: int = 1 << 26) -> np.ndarray:
    """Packed Bernoulli(p_keep) keep-bits, little-endian bit order within a byte."""
    nbytes = (nbits + 7) // 8
    out = np.empty(nbytes, dtype=np.uint8)
    thresh = np.uint16(min(65535, int(round(p_keep * 65536.0))))
    rng = _rng(seed, "mask")
    chunk_bits -= chunk_bits % 8
    done = 0
    while done < nbits:
        n = min(chunk_bits, nbits - done)
        u = rng.integers(0, 65536, size=n, dtype=np.uint16)
        keep = u < thresh if p_keep < 1.0 else np.ones(n, dtype=bool)
        packed = np.packbits(keep, bitorder="little")
        out[done // 8: done // 8 + packed.size] = packed
        done += n
    return out


@dataclasses.dataclass
class Inputs:
    """Host-side tensors of one workload (storage form and exact fp64 form)."""

    wl: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dy: np.ndarray
    q64: np.ndarray
    k64: np.ndarray
    v64: np.ndarray
    dy64: np.ndarray
    sink: Optional[np.ndarray]          # float32 [Nq] or None
    mask: Optional[np.ndarray]          # uint8 packed keep-bits or None
    amask: Optional[np.ndarray] = None  # uint8 [S1Max, S2Max] attention-mask matrix (nonzero masks) or None
    pse: Optional[np.ndarray] = None    # [pse_batch, Nq, 1024, S2Max] in the storage dtype, or None
    pse64: Optional[np.ndarray] = None  # its exact fp64 values


def make_inputs(wl: Workload, with_fp64: bool = True) -> Inputs:
    """Draw Q, K, V, dY (and sink / dropout mask when the workload uses them)."""
    q, q64 = normal(wl.seed, "q", (wl.tq, wl.nq, wl.d), wl.dtype)
    k, k64 = normal(wl.seed, "k", (wl.tkv, wl.nkv, wl.d), wl.dtype)
    v, v64 = normal(wl.seed, "v", (wl.tkv, wl.nkv, wl.dv), wl.dtype)
    dy, dy64 = normal(wl.seed, "dy", (wl.tq, wl.nq, wl.dv), wl.dtype)
    sink = None
    if wl.has_sink:
        sink = _rng(wl.seed, "sink").standard_normal(size=wl.nq, dtype=np.float64).astype(np.float32)
    mask = None
    if wl.keep_prob < 1.0:
        mask = dropout_mask(wl.seed, wl.mask_bits(), wl.keep_prob)
    amask = None
    if wl.amask_density > 0:
        amask = atten_mask_matrix(wl.seed, max(wl.seqlens_q), max(wl.seqlens_kv), wl.amask_density)
    pse = pse64 = None
    if wl.pse_kind == "slopes":
        pse, pse64 = pse_slopes(wl)
    elif wl.pse_kind:
        pse, pse64 = pse_store(wl)
    if not with_fp64:
        q64 = k64 = v64 = dy64 = None
    return Inputs(wl, q, k, v, dy, q64, k64, v64, dy64, sink, mask, amask, pse, pse64)


def pse_store(wl: Workload):
    """[pse_batch, Nq, 1024, S2Max] pse store ("random" or "alibi"), rounded to the dtype."""
    s2 = max(wl.seqlens_kv)
    shape = (wl.pse_batch, wl.nq, 1024, s2)
    if wl.pse_kind == "random":
        x = 0.5 * _rng(wl.seed, "pse").standard_normal(size=shape, dtype=np.float64)
    else:
        x = np.zeros(shape)
        slopes = 2.0 ** -(4.0 + np.arange(wl.nq))
        for b in range(wl.pse_batch):
            sq = wl.seqlens_q[b]
            rows = np.arange(1024) + (sq - 1024)          # the sequence row each stored row holds
            cols = np.arange(s2)
            x[b] = slopes[:, None, None] * (cols[None, None, :] - rows[None, :, None])
    return round_to_dtype(x, wl.dtype)


def pse_slopes(wl: Workload):
    """fp32 slopes of a generated pse: [pse_batch, Nq], or [Nq] when pse_batch is 1; the
    usual alibi geometric slopes 2^-(8 (h + 1) / Nq) with a per-sequence jitter."""
    base = 2.0 ** (-8.0 * (np.arange(wl.nq) + 1) / wl.nq)
    jit = 1.0 + 0.25 * _rng(wl.seed, "slopes").random(size=(wl.pse_batch, wl.nq))
    x = (base[None, :] * jit).astype(np.float32)
    if wl.pse_batch == 1:
        x = x[0]
    return x, x.astype(np.float64)


def atten_mask_matrix(seed: int, rows: int, cols: int, density: float) -> np.ndarray:
    """uint8 [rows, cols]: 1 (masked) with probability ``density``; rows i with
    i % 97 == 5 fully masked."""
    thresh = np.uint16(min(65535, int(round(density * 65536.0))))
    u = _rng(seed, "amask").integers(0, 65536, size=(rows, cols), dtype=np.uint16)
    out = (u < thresh).astype(np.uint8)
    out[5::97, :] = 1
    return out


def custom(name: str, dtype: str, seqlens_q, seqlens_kv, nq: int, nkv: int, d: int, *,
           scale: Optional[float] = None, keep_prob: float = 1.0, pre_tokens: int = 2147483647,
           next_tokens: int = 2147483647, sparse_mode: int = 0, has_sink: bool = False,
           seed: int = BASE_SEED, amask_density: float = 0.0, prefix=None, pse_kind: str = "",
           pse_batch: int = 1, pse_type: int = 1, dv: int = 0) -> Workload:
    """A workload with explicit shapes (used for edge cases and small parity runs)."""
    return Workload(name, dtype, list(seqlens_q), list(seqlens_kv), nq, nkv, d,
                    1.0 / math.sqrt(d) if scale is None else scale, keep_prob, pre_tokens,
                    next_tokens, sparse_mode, has_sink, seed, amask_density,
                    None if prefix is None else list(prefix), pse_kind, pse_batch, pse_type, dv)
