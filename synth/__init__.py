"""Seeded synthetic inputs for the routed MoE FFN layer.

This module is shared by the fp64 oracle (``oracle/``), the tests and the
benchmark. It holds none of the layer's arithmetic: it only draws random
numbers and writes them at the byte offsets of the four block formats, and it
draws activations and router logits. The GPU copy of the weight filler
(``synth/csrc/synth_fill.cu``) implements the same counter-based generator from
the same definition; ``tests/test_synth.py`` checks that both write identical
bytes.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014). The i-th output (i = 0, 1, ...) of the
sequence seeded with ``key`` is ``mix64(key + (i + 1) * GAMMA)``, so any draw is
computed from its index alone. A (seed, stream) pair selects the key:
``key = mix64(mix64(seed) + stream * GAMMA)``.

Recipe (all values little-endian):

* Weight block ``b`` of a matrix (blocks numbered row-major, ``row * nb + j``)
  uses draws ``32*b + 0 .. 32*b + 31`` of the matrix's stream.
* ``u24(r) = float32(r >> 40) * 2**-24`` is a uniform in [0, 1), exact in fp32.
* An fp16 scale drawn from U[lo, lo + span) is ``f16_rne(lo + span * u24(r))``
  with one fp32 multiply and one fp32 add, each rounded to nearest even (no
  fused multiply-add), then rounded to fp16 to nearest even.
* ``ubelow(x, n) = (x * n) >> bits(x)`` maps a uniform ``bits``-bit integer to
  {0..n-1} (multiply-shift; the bias is below 2**-16 and immaterial here).
* Q8_0 (34 B):  d = f16(0.002 + 0.018 u24(r0));  q_i (i < 32) =
  ubelow(16-bit chunk i%4 of r_{1+i//4}, 255) - 127, i.e. U{-127..127}.
* Q4_K (144 B): d = f16(0.0005 + 0.0045 u24(r0)), dmin likewise from r1; the
  12 scale bytes and 128 code bytes are the bytes of r2, r3, ... in order, so
  every 6-bit scale/min and every 4-bit code is uniform.
* Q6_K (210 B): ql (128 B) and qh (64 B) are the bytes of r0..r23 in order
  (6-bit codes uniform on 0..63); scale i (int8) = ubelow(16-bit chunk i%4 of
  r_{24+i//4}, 255) - 127; d = f16(1e-4 + 9e-4 u24(r28)).
* MXFP4 (17 B): e = 124 + ubelow(low 32 bits of r0, 3); the 16 code bytes are
  the bytes of r1, r2.
* IQ4_NL (18 B): d = f16(0.002 + 0.018 u24(r0)); the 16 code bytes are the
  bytes of r1, r2.
* IQ4_XS (136 B): d = f16(2e-4 + 1e-3 u24(r0)); bytes 2..7 (high scale bits
  and low scale nibbles) are bytes 0..5 of r1; the 128 code bytes are the
  bytes of r2..r17.
* IQ3_XXS (98 B): d = f16(0.001 + 0.009 u24(r0)); the 64 grid-index bytes
  are the bytes of r1..r8; the 32 scale/sign bytes are the bytes of r9..r12.
  The layer's grid (256 entries of four magnitude bytes) is drawn once from
  stream GRID of seed 0: byte j of entry i is ``IQ3_MAGNITUDES[ubelow(16-bit
  chunk j of draw i, 8)]``.
* T5_G128 (28 B): s = f16(0.25 + 0.75 u24(r0)); code byte i < 25 =
  ubelow(16-bit chunk i%4 of r_{1+i//4}, 243) (five uniform base-3 digits),
  code byte 25 = ubelow(chunk 1 of r7, 27) (three digits, the unused two 0).
* Row padding bytes (``row_stride`` beyond the row's blocks) are zero.
* Normals: Box-Muller in fp64 on draws (2i, 2i+1):
  ``sqrt(-2 ln u1) cos(2 pi u2)`` with ``u1 = ((r >> 11) + 1) 2**-53``,
  ``u2 = (r' >> 11) 2**-53``; rounded to fp32 (nearest even), and for bf16
  activations further to bf16 (nearest even).
* Router logits: ``fp32(z + b[rank(e)])`` where ``b_r = -1.5 ln(1 + r/512)``
  is the Zipf-shaped (shifted power law in rank) bias and ``rank`` inverts the
  permutation ``perm = argsort(draws of the PERM stream)`` (stable), so that
  hot experts are not contiguous ids. The tiny layer uses no bias.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# Format tags (the same numeric values as the C ABI's moe_format enum).
Q8_0, Q4_K, Q6_K, MXFP4, IQ4_NL, IQ4_XS, IQ3_XXS, T5_G128 = 1, 2, 3, 4, 5, 6, 7, 8
FORMAT_NAMES = {Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", MXFP4: "MXFP4", IQ4_NL: "IQ4_NL", IQ4_XS: "IQ4_XS",
                IQ3_XXS: "IQ3_XXS", T5_G128: "T5_G128"}
BLOCK_ELEMS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, MXFP4: 32, IQ4_NL: 32, IQ4_XS: 256, IQ3_XXS: 256, T5_G128: 128}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, MXFP4: 17, IQ4_NL: 18, IQ4_XS: 136, IQ3_XXS: 98, T5_G128: 28}
# the magnitudes the synthetic IQ3_XXS grid draws from
IQ3_MAGNITUDES = np.array([4, 12, 20, 28, 36, 44, 52, 62], dtype=np.int64)

GAMMA = 0x9E3779B97F4A7C15
_MASK64 = (1 << 64) - 1

STREAM_X = 1
STREAM_LOGITS = 2
STREAM_PERM = 3
STREAM_GRID = 4
STREAM_WEIGHTS = 16          # + 3 * expert + matrix (0 gate, 1 up, 2 down)
DRAWS_PER_BLOCK = 32

GATE, UP, DOWN = 0, 1, 2


# --------------------------------------------------------------------------
# SplitMix64
# --------------------------------------------------------------------------
def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> int:
    """Key of stream ``stream`` under ``seed`` (both non-negative ints)."""
    return _mix64_int(_mix64_int(seed) + stream * GAMMA)


def draws(key: int, idx: np.ndarray) -> np.ndarray:
    """uint64 draws number ``idx`` (any int array) of the sequence ``key``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + (idx + np.uint64(1)) * np.uint64(GAMMA))


def _u24(r: np.ndarray) -> np.ndarray:
    return (r >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)


def _f16_uniform(r: np.ndarray, lo: float, span: float) -> np.ndarray:
    # one fp32 multiply, one fp32 add (numpy float32 ops round to nearest even)
    v = np.float32(lo) + np.float32(span) * _u24(r)
    return v.astype(np.float32).astype(np.float16)


def _ubelow16(chunk: np.ndarray, n: int) -> np.ndarray:
    return ((chunk.astype(np.uint64) * np.uint64(n)) >> np.uint64(16)).astype(np.int64)


def _chunks16(r: np.ndarray) -> np.ndarray:
    """[..., m] uint64 -> [..., 4m] 16-bit chunks (chunk c of r_j at 4j+c)."""
    c = np.stack([(r >> np.uint64(16 * i)) & np.uint64(0xFFFF) for i in range(4)], axis=-1)
    return c.reshape(*r.shape[:-1], r.shape[-1] * 4)


def _bytes_of(r: np.ndarray) -> np.ndarray:
    """[..., m] uint64 -> [..., 8m] uint8, little-endian bytes in order."""
    return np.ascontiguousarray(r.astype("<u8")).view(np.uint8).reshape(*r.shape[:-1], r.shape[-1] * 8)


# --------------------------------------------------------------------------
# weight matrices
# --------------------------------------------------------------------------
@dataclass
class MatrixBytes:
    """A block-quantized matrix: ``rows`` rows of ``cols`` weights, blocks
    along the columns; row ``r`` occupies ``data[r*stride : r*stride + nb*bb]``."""
    fmt: int
    rows: int
    cols: int
    stride: int
    data: np.ndarray  # uint8 [rows * stride]
    grid: Optional[np.ndarray] = None   # IQ3_XXS: the 256-entry grid (uint32)

    @property
    def nbytes_unpadded(self) -> int:
        return self.rows * (self.cols // BLOCK_ELEMS[self.fmt]) * BLOCK_BYTES[self.fmt]


def row_bytes(fmt: int, cols: int) -> int:
    return (cols // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def padded_stride(fmt: int, cols: int, align: int = 16) -> int:
    rb = row_bytes(fmt, cols)
    return (rb + align - 1) // align * align


def gen_blocks(fmt: int, key: int, block_idx: np.ndarray) -> np.ndarray:
    """Bytes of the blocks numbered ``block_idx`` -> uint8 [n, BLOCK_BYTES]."""
    block_idx = np.asarray(block_idx, dtype=np.uint64).reshape(-1)
    j = np.arange(DRAWS_PER_BLOCK, dtype=np.uint64)
    r = draws(key, block_idx[:, None] * np.uint64(DRAWS_PER_BLOCK) + j[None, :])
    n = block_idx.shape[0]
    out = np.zeros((n, BLOCK_BYTES[fmt]), dtype=np.uint8)
    if fmt == Q8_0:
        out[:, 0:2] = _f16_uniform(r[:, 0], 0.002, 0.018).view(np.uint8).reshape(n, 2)
        q = _ubelow16(_chunks16(r[:, 1:9]), 255) - 127
        out[:, 2:34] = q.astype(np.int8).view(np.uint8)
    elif fmt == Q4_K:
        out[:, 0:2] = _f16_uniform(r[:, 0], 0.0005, 0.0045).view(np.uint8).reshape(n, 2)
        out[:, 2:4] = _f16_uniform(r[:, 1], 0.0005, 0.0045).view(np.uint8).reshape(n, 2)
        out[:, 4:144] = _bytes_of(r[:, 2:20])[:, :140]
    elif fmt == Q6_K:
        out[:, 0:192] = _bytes_of(r[:, 0:24])
        sc = _ubelow16(_chunks16(r[:, 24:28]), 255) - 127
        out[:, 192:208] = sc.astype(np.int8).view(np.uint8)
        out[:, 208:210] = _f16_uniform(r[:, 28], 1e-4, 9e-4).view(np.uint8).reshape(n, 2)
    elif fmt == MXFP4:
        lo32 = (r[:, 0] & np.uint64(0xFFFFFFFF)).astype(np.uint64)
        out[:, 0] = (124 + ((lo32 * np.uint64(3)) >> np.uint64(32))).astype(np.uint8)
        out[:, 1:17] = _bytes_of(r[:, 1:3])
    elif fmt == IQ4_NL:
        out[:, 0:2] = _f16_uniform(r[:, 0], 0.002, 0.018).view(np.uint8).reshape(n, 2)
        out[:, 2:18] = _bytes_of(r[:, 1:3])
    elif fmt == IQ4_XS:
        out[:, 0:2] = _f16_uniform(r[:, 0], 2e-4, 1e-3).view(np.uint8).reshape(n, 2)
        out[:, 2:8] = _bytes_of(r[:, 1:2])[:, 0:6]
        out[:, 8:136] = _bytes_of(r[:, 2:18])
    elif fmt == IQ3_XXS:
        out[:, 0:2] = _f16_uniform(r[:, 0], 0.001, 0.009).view(np.uint8).reshape(n, 2)
        out[:, 2:66] = _bytes_of(r[:, 1:9])
        out[:, 66:98] = _bytes_of(r[:, 9:13])
    elif fmt == T5_G128:
        out[:, 0:2] = _f16_uniform(r[:, 0], 0.25, 0.75).view(np.uint8).reshape(n, 2)
        ch = _chunks16(r[:, 1:8])
        out[:, 2:27] = _ubelow16(ch[:, 0:25], 243)
        out[:, 27] = _ubelow16(ch[:, 25], 27)
    else:
        raise ValueError(f"unknown format {fmt}")
    return out


def gen_matrix(fmt: int, rows: int, cols: int, key: int, stride: Optional[int] = None) -> MatrixBytes:
    be, bb = BLOCK_ELEMS[fmt], BLOCK_BYTES[fmt]
    if cols % be:
        raise ValueError(f"{FORMAT_NAMES[fmt]} needs cols % {be} == 0, got {cols}")
    nb = cols // be
    if stride is None:
        stride = padded_stride(fmt, cols)
    blocks = gen_blocks(fmt, key, np.arange(rows * nb))
    data = np.zeros((rows, stride), dtype=np.uint8)
    data[:, : nb * bb] = blocks.reshape(rows, nb * bb)
    return MatrixBytes(fmt, rows, cols, stride, data.reshape(-1))


def iq3_grid() -> np.ndarray:
    """The synthetic IQ3_XXS grid (uint32 [256]), the same for every layer."""
    r = draws(stream_key(0, STREAM_GRID), np.arange(256))
    idx = _ubelow16(_chunks16(r[:, None]), 8).reshape(256, 4)
    mag = IQ3_MAGNITUDES[idx]
    return (mag[:, 0] | (mag[:, 1] << 8) | (mag[:, 2] << 16) | (mag[:, 3] << 24)).astype(np.uint32)


def weight_key(seed: int, expert: int, matrix: int) -> int:
    return stream_key(seed, STREAM_WEIGHTS + 3 * expert + matrix)


# --------------------------------------------------------------------------
# layer configurations
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class LayerConfig:
    name: str
    n_experts: int
    k: int
    hidden: int
    inter: int
    tokens: int
    tiers: str            # "q8_0" (all Q8_0), "q4k" (Q4_K gate/up + Q8_0 down), "mixed", "mixed_iq", "t5"
    zipf_bias: bool
    seed_base: int        # layer l uses seed seed_base + l (tiny: seed 0)
    n_shared: int = 0     # shared experts (Q8_0), entries n_experts .. n_experts + n_shared - 1

    @property
    def n_entries(self) -> int:
        """Routed plus shared experts: the length of the layer's expert table."""
        return self.n_experts + self.n_shared


CONFIGS: Dict[str, LayerConfig] = {
    "tiny": LayerConfig("tiny", 8, 2, 256, 128, 4, "q8_0", False, 0),
    "decode1": LayerConfig("decode1", 512, 10, 2048, 640, 1, "q4k", True, 2000),
    "decode16": LayerConfig("decode16", 512, 10, 2048, 640, 16, "q4k", True, 3000),
    "mtp6": LayerConfig("mtp6", 512, 10, 2048, 640, 6, "mixed", True, 4000),
    "prefill2048": LayerConfig("prefill2048", 512, 10, 2048, 640, 2048, "mixed", True, 5000),
    # the pages' own tier formats: Q6_K/Q8_0, IQ4_XS/IQ4_NL, IQ3_XXS/MXFP4
    "mtp6_iq": LayerConfig("mtp6_iq", 512, 10, 2048, 640, 6, "mixed_iq", True, 6000),
    "prefill2048_iq": LayerConfig("prefill2048_iq", 512, 10, 2048, 640, 2048, "mixed_iq", True, 7000),
    # one Q8_0 shared expert beside the routed ones
    "decode16_shared": LayerConfig("decode16_shared", 512, 10, 2048, 640, 16, "q4k", True, 8000, 1),
    "prefill512_shared": LayerConfig("prefill512_shared", 512, 10, 2048, 640, 512, "mixed", True, 9000, 1),
    # ternary experts (every matrix T5_G128)
    "decode16_t5": LayerConfig("decode16_t5", 512, 10, 2048, 640, 16, "t5", True, 10000),
    "prefill512_t5": LayerConfig("prefill512_t5", 512, 10, 2048, 640, 512, "t5", True, 11000),
}


def tier_bounds(n_experts: int) -> Tuple[int, int]:
    """Rank boundaries of the three tiers: top 25%, middle 55%, tail 20%.

    Ranks [0, a) are the top tier, [a, b) the middle tier, [b, E) the tail,
    with a = floor(0.25 E) and b = E - floor(0.20 E) (512 -> 128, 410)."""
    return n_experts * 25 // 100, n_experts - n_experts * 20 // 100


def permutation(seed: int, n_experts: int) -> np.ndarray:
    """perm[rank] = expert id (rank 0 is the hottest expert)."""
    r = draws(stream_key(seed, STREAM_PERM), np.arange(n_experts))
    return np.argsort(r, kind="stable").astype(np.int64)


def expert_formats(cfg: LayerConfig, seed: int) -> List[Tuple[int, int]]:
    """Per table entry: (gate/up format, down format); the shared experts,
    after the routed ones, are Q8_0."""
    return _routed_formats(cfg, seed) + [(Q8_0, Q8_0)] * cfg.n_shared


def _routed_formats(cfg: LayerConfig, seed: int) -> List[Tuple[int, int]]:
    E = cfg.n_experts
    if cfg.tiers == "q8_0":
        return [(Q8_0, Q8_0)] * E
    if cfg.tiers == "q4k":
        return [(Q4_K, Q8_0)] * E
    if cfg.tiers == "t5":
        return [(T5_G128, T5_G128)] * E
    if cfg.tiers in ("mixed", "mixed_iq"):
        iq = cfg.tiers == "mixed_iq"
        perm = permutation(seed, E)
        a, b = tier_bounds(E)
        fm: List[Tuple[int, int]] = [(0, 0)] * E
        for rank, e in enumerate(perm):
            if rank < a:
                fm[int(e)] = (Q6_K, Q8_0)
            elif rank < b:
                fm[int(e)] = (IQ4_XS, IQ4_NL) if iq else (Q4_K, Q8_0)
            else:
                fm[int(e)] = (IQ3_XXS, MXFP4) if iq else (MXFP4, MXFP4)
        return fm
    raise ValueError(cfg.tiers)


def layer_seed(cfg: LayerConfig, layer: int) -> int:
    return cfg.seed_base + layer


def expert_matrices(cfg: LayerConfig, seed: int, expert: int,
                    fmts: Optional[Tuple[int, int]] = None) -> Dict[str, MatrixBytes]:
    if fmts is None:
        fmts = expert_formats(cfg, seed)[expert]
    gu, dn = fmts
    H, I = cfg.hidden, cfg.inter
    m = {
        "gate": gen_matrix(gu, I, H, weight_key(seed, expert, GATE)),
        "up": gen_matrix(gu, I, H, weight_key(seed, expert, UP)),
        "down": gen_matrix(dn, H, I, weight_key(seed, expert, DOWN)),
    }
    for v in m.values():
        if v.fmt == IQ3_XXS:
            v.grid = iq3_grid()
    return m


# --------------------------------------------------------------------------
# activations and logits
# --------------------------------------------------------------------------
def normals(key: int, n: int, start: int = 0) -> np.ndarray:
    i = np.arange(start, start + n, dtype=np.uint64)
    r1 = draws(key, 2 * i)
    r2 = draws(key, 2 * i + np.uint64(1))
    u1 = ((r1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (r2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def gen_x_bf16(seed: int, T: int, H: int) -> np.ndarray:
    """Activations as bf16 bit patterns, uint16 [T, H]."""
    z = normals(stream_key(seed, STREAM_X), T * H).astype(np.float32)
    return f32_to_bf16_bits(z).reshape(T, H)


def zipf_bias(n_experts: int) -> np.ndarray:
    r = np.arange(n_experts, dtype=np.float64)
    return -1.5 * np.log1p(r / 512.0)


def gen_logits(seed: int, T: int, E: int, biased: bool) -> np.ndarray:
    z = normals(stream_key(seed, STREAM_LOGITS), T * E).reshape(T, E)
    if biased:
        perm = permutation(seed, E)
        rank = np.empty(E, dtype=np.int64)
        rank[perm] = np.arange(E)
        z = z + zipf_bias(E)[rank][None, :]
    return z.astype(np.float32)


@dataclass
class SynthLayer:
    cfg: LayerConfig
    seed: int
    fmts: List[Tuple[int, int]]
    x_bf16: np.ndarray          # uint16 [T, H]
    logits: np.ndarray          # float32 [T, E]
    experts: List[Dict[str, MatrixBytes]]   # may be empty when weights are made on the GPU


def make_layer(cfg: LayerConfig, layer: int = 0, with_weights: bool = True,
               tokens: Optional[int] = None) -> SynthLayer:
    seed = layer_seed(cfg, layer)
    T = cfg.tokens if tokens is None else tokens
    fmts = expert_formats(cfg, seed)
    x = gen_x_bf16(seed, T, cfg.hidden)
    logits = gen_logits(seed, T, cfg.n_experts, cfg.zipf_bias)
    experts = [expert_matrices(cfg, seed, e, fmts[e]) for e in range(cfg.n_entries)] if with_weights else []
    return SynthLayer(cfg, seed, fmts, x, logits, experts)


class LazyExperts:
    """Indexable of a layer's experts that generates (and keeps) an expert's
    matrices on first access; ``len`` is the table length (routed + shared)."""

    def __init__(self, cfg: LayerConfig, seed: int, fmts: Optional[List[Tuple[int, int]]] = None):
        self.cfg, self.seed = cfg, seed
        self.fmts = fmts if fmts is not None else expert_formats(cfg, seed)
        self._cache: Dict[int, Dict[str, MatrixBytes]] = {}

    def __len__(self) -> int:
        return self.cfg.n_entries

    def __getitem__(self, e: int) -> Dict[str, MatrixBytes]:
        e = int(e)
        if e not in self._cache:
            self._cache[e] = expert_matrices(self.cfg, self.seed, e, self.fmts[e])
        return self._cache[e]

    def gate_formats(self) -> List[int]:
        return [f[0] for f in self.fmts]

    def release(self, e: int) -> None:
        """Forget expert e's generated bytes (it is regenerated on next access)."""
        self._cache.pop(int(e), None)

    def __getstate__(self):
        # pickled without the generated bytes (they are regenerated on access)
        d = dict(self.__dict__)
        d["_cache"] = {}
        return d


def expert_bytes(fmts: Tuple[int, int], hidden: int, inter: int) -> int:
    """Unpadded quantized bytes of one expert (gate + up + down)."""
    gu, dn = fmts
    return 2 * inter * row_bytes(gu, hidden) + hidden * row_bytes(dn, inter)
