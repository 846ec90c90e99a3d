"""Seeded synthetic inputs for the TT-linear layer.

This module only draws random numbers; it holds none of the layer's
arithmetic.  Both the CUDA path (through the tests and the benchmark) and the
CPU oracle take their inputs from here, so that the two sides see the same
values.

The workloads mirror the transformer layers of the CoMERA project page
("Results": six-encoder transformer, sequence length 128, every linear layer
tensorised starting from rank 30; the rank table "Internal tensor-train ranks
of each layer in one encoder block").  The ranks below are the capped ranks
that table prints (12/16 at the chain ends, 30 inside) and are written out as
numbers, not computed here.

Draw order for one layer: cores G_1..G_2d, diagonals D_1..D_{2d-1}, x, dy,
all from one numpy PCG64 stream seeded with ``seed``.  "N(0, s)" means
standard deviation s.  Activations drawn for a bf16 workload are rounded to
the nearest bf16 value (round to nearest even) once, here, so both sides read
identical numbers.  Activations of an e4m3 workload are rounded the same way
to the nearest OCP FP8 E4M3 ("e4m3fn") value, saturating at +-448; the device
receives the one-byte codes of those values.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One TT linear layer: y (T x M) = x (T x N) W^T, W stored as 2d cores."""

    in_modes: Tuple[int, ...]   # n_1..n_d, N = prod
    out_modes: Tuple[int, ...]  # m_1..m_d, M = prod
    ranks: Tuple[int, ...]      # r_0..r_2d, r_0 = r_2d = 1

    @property
    def d(self) -> int:
        return len(self.in_modes)

    @property
    def N(self) -> int:
        return int(np.prod(self.in_modes))

    @property
    def M(self) -> int:
        return int(np.prod(self.out_modes))

    @property
    def modes(self) -> Tuple[int, ...]:
        return tuple(self.in_modes) + tuple(self.out_modes)

    def core_shapes(self) -> List[Tuple[int, int, int]]:
        s = self.modes
        r = self.ranks
        return [(r[k], s[k], r[k + 1]) for k in range(2 * self.d)]

    def diag_sizes(self) -> List[int]:
        return [self.ranks[k + 1] for k in range(2 * self.d - 1)]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: Tuple[LayerShape, ...]   # one layer, or (up, down) for the FFN pair
    tokens: int
    act: str                         # "f32", "bf16" or "e4m3" (x, dy; y and dx bf16)
    core_std: float
    x_std: float
    dy_std: float
    diag: str                        # "ones", "uniform", "pruned_half"
    ffn: bool = False
    description: str = ""


_L768_768 = LayerShape((12, 8, 8), (8, 8, 12), (1, 12, 30, 30, 30, 12, 1))
_L768_3072 = LayerShape((12, 8, 8), (12, 16, 16), (1, 12, 30, 30, 30, 16, 1))
_L3072_768 = LayerShape((16, 16, 12), (8, 8, 12), (1, 16, 30, 30, 30, 12, 1))
_L1024_4096 = LayerShape((8, 8, 16), (16, 16, 16), (1, 8, 64, 64, 64, 16, 1))
_L64_64 = LayerShape((4, 4, 4), (4, 4, 4), (1, 4, 8, 8, 8, 4, 1))

WORKLOADS = {
    "tiny64_f32": Workload(
        "tiny64_f32", (_L64_64,), 16, "f32", 0.1, 0.1, 1.0, "ones",
        description="TT linear 64x64, modes (4,4,4)x(4,4,4), ranks 8, D=1, 16 tokens, fp32"),
    "tt768_bf16": Workload(
        "tt768_bf16", (_L768_768,), 16384, "bf16", 0.05, 1.0, 1.0, "uniform",
        description="TT linear 768x768, modes (12,8,8)x(8,8,12), ranks 30, "
                    "D~U(0.5,1.5), 16384 tokens (128 seq x 128 batch), bf16 x/dy"),
    "ffn768_3072_bf16": Workload(
        "ffn768_3072_bf16", (_L768_3072, _L3072_768), 16384, "bf16", 0.05, 1.0, 1.0,
        "uniform", ffn=True,
        description="TT FFN 768->3072->768 with exact GELU, ranks 30, 16384 tokens, bf16"),
    "pruned768_3072_bf16": Workload(
        "pruned768_3072_bf16", (_L768_3072,), 16384, "bf16", 0.05, 1.0, 1.0,
        "pruned_half",
        description="TT linear 768->3072, ranks 30, half of every D_k exactly zero, "
                    "16384 tokens, bf16"),
    "pruned768_768_bf16": Workload(
        "pruned768_768_bf16", (_L768_768,), 16384, "bf16", 0.05, 1.0, 1.0,
        "pruned_half",
        description="TT linear 768x768, ranks 30, half of every D_k exactly zero, "
                    "16384 tokens, bf16"),
    "tt768_e4m3": Workload(
        "tt768_e4m3", (_L768_768,), 16384, "e4m3", 0.05, 1.0, 1.0, "uniform",
        description="TT linear 768x768, modes (12,8,8)x(8,8,12), ranks 30, "
                    "D~U(0.5,1.5), 16384 tokens, e4m3 x/dy, bf16 y/dx"),
    "tt1024_4096_e4m3": Workload(
        "tt1024_4096_e4m3", (_L1024_4096,), 32768, "e4m3", 0.03, 1.0, 1.0, "uniform",
        description="TT linear 1024->4096, modes (8,8,16)x(16,16,16), ranks 64, "
                    "32768 tokens, e4m3 x/dy, bf16 y/dx"),
    "tt1024_4096_bf16": Workload(
        "tt1024_4096_bf16", (_L1024_4096,), 32768, "bf16", 0.03, 1.0, 1.0, "uniform",
        description="TT linear 1024->4096, modes (8,8,16)x(16,16,16), ranks 64, "
                    "32768 tokens (64 x 512), bf16"),
}


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 value (ties to even).

    Returns float32 values that are exactly representable in bfloat16.
    Non-finite inputs are not expected from the generators here.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


E4M3_MAX = 448.0


def round_e4m3(a: np.ndarray) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (ties to even), saturating at +-448.

    E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities; the largest finite value is 1.75 * 2^8 = 448, the
    smallest normal 2^-6, the subnormal step 2^-9.  Returns float32 values
    exactly representable in E4M3.
    """
    v = np.asarray(a, dtype=np.float64)
    m = np.minimum(np.abs(v), E4M3_MAX)
    _, ex = np.frexp(np.maximum(m, 2.0 ** -6))
    step = np.ldexp(1.0, ex - 1 - 3)          # 2^(e - 3), e = floor(log2 m) >= -6
    r = np.round(m / step) * step               # numpy rounds halves to even
    return (np.sign(v) * r).astype(np.float32)


def e4m3_bytes(a: np.ndarray) -> np.ndarray:
    """One-byte E4M3 codes of values that are already E4M3-representable."""
    v = np.asarray(a, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint16) << 7
    m = np.abs(v)
    _, ex = np.frexp(np.maximum(m, 2.0 ** -6))
    e = ex - 1
    normal = m >= 2.0 ** -6
    field = np.where(normal, (e + 7) * 8 + (m / np.ldexp(1.0, e) - 1.0) * 8, m / 2.0 ** -9)
    code = np.rint(field).astype(np.uint16)
    assert np.all(np.abs(field - code) == 0), "value not representable in E4M3"
    return (sign | code).astype(np.uint8)


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """float32 values of one-byte E4M3 codes (NaN codes 0x7F / 0xFF included)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    mt = c & 7
    mag = np.where(E == 0, mt * 2.0 ** -9, np.ldexp(1.0 + mt / 8.0, E - 7))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return (s * mag).astype(np.float32)


@dataclasses.dataclass
class LayerInputs:
    cores: List[np.ndarray]   # float32, shapes (r_{k-1}, s_k, r_k)
    diags: List[np.ndarray]   # float32, lengths r_k for the 2d-1 internal links


def draw_layer(rng: np.random.Generator, shape: LayerShape, core_std: float,
               diag: str) -> LayerInputs:
    cores = [(rng.standard_normal(cs) * core_std).astype(np.float32)
             for cs in shape.core_shapes()]
    diags = []
    for n in shape.diag_sizes():
        if diag == "ones":
            dv = np.ones(n, dtype=np.float32)
        elif diag == "uniform":
            dv = rng.uniform(0.5, 1.5, size=n).astype(np.float32)
        elif diag == "pruned_half":
            dv = rng.uniform(0.5, 1.5, size=n).astype(np.float32)
            dv[rng.permutation(n)[: n // 2]] = 0.0
        else:
            raise ValueError(diag)
        diags.append(dv)
    return LayerInputs(cores, diags)


@dataclasses.dataclass
class WorkloadInputs:
    layers: List[LayerInputs]
    x: np.ndarray    # (T, N_first) float32 (bf16-representable for bf16 workloads)
    dy: np.ndarray   # (T, M_last)


def draw(w: Workload, seed: int = 0, tokens: Optional[int] = None) -> WorkloadInputs:
    """All inputs of one workload from one seeded stream (see module doc)."""
    T = w.tokens if tokens is None else int(tokens)
    rng = np.random.Generator(np.random.PCG64(seed))
    layers = [draw_layer(rng, s, w.core_std, w.diag) for s in w.layers]
    x = (rng.standard_normal((T, w.layers[0].N)) * w.x_std).astype(np.float32)
    dy = (rng.standard_normal((T, w.layers[-1].M)) * w.dy_std).astype(np.float32)
    if w.act == "bf16":
        x = round_bf16(x)
        dy = round_bf16(dy)
    elif w.act == "e4m3":
        x = round_e4m3(x)
        dy = round_e4m3(dy)
    return WorkloadInputs(layers, x, dy)


# ---------------------------------------------------------------------------
# The TT layers of one transformer encoder block (the project page's
# six-encoder model, "Results": the attention projections Q, K, V, O at
# 768 x 768 and the feed-forward pair 768 -> 3072 -> 768, every one a
# rank-30 TT as in the rank table "Internal tensor-train ranks of each layer
# in one encoder block").  Q, K and V read the same input x; O reads the
# attention output and the FFN pair the block's middle activations, for which
# independent synthetic tensors stand in (the attention itself is not a TT
# layer).  Distributions as "tt768_bf16": cores N(0, 0.05), D ~ U(0.5, 1.5),
# activations and upstream gradients bf16 N(0, 1).

ENCODER_LAYERS = {"q": _L768_768, "k": _L768_768, "v": _L768_768, "o": _L768_768,
                  "up": _L768_3072, "down": _L3072_768}


@dataclasses.dataclass
class EncoderInputs:
    layers: dict        # name -> LayerInputs ("q", "k", "v", "o", "up", "down")
    x: np.ndarray       # (T, 768): input of Q, K and V
    xo: np.ndarray      # (T, 768): input of O (stands in for the attention output)
    xf: np.ndarray      # (T, 768): input of the FFN pair
    dy: dict            # "q", "k", "v", "o", "ffn" -> (T, 768) upstream gradients


def draw_encoder(tokens: int = 16384, seed: int = 0) -> EncoderInputs:
    """The block's inputs, from one seeded stream: the layers' cores and
    diagonals in the order q, k, v, o, up, down, then x, xo, xf, then the
    upstream gradients of q, k, v, o and the FFN pair."""
    rng = np.random.Generator(np.random.PCG64(seed))
    layers = {nm: draw_layer(rng, sh, 0.05, "uniform") for nm, sh in ENCODER_LAYERS.items()}

    def act(n):
        return round_bf16(rng.standard_normal((tokens, n)).astype(np.float32))
    x, xo, xf = act(768), act(768), act(768)
    dy = {nm: act(768) for nm in ("q", "k", "v", "o", "ffn")}
    return EncoderInputs(layers, x, xo, xf, dy)


def random_shape(rng: np.random.Generator, d: int, max_mode: int = 4,
                 max_rank: int = 4) -> LayerShape:
    """A small random TT shape for sweep tests (ranks not capped: any r >= 1 is a TT)."""
    nm = tuple(int(v) for v in rng.integers(1, max_mode + 1, size=d))
    mm = tuple(int(v) for v in rng.integers(1, max_mode + 1, size=d))
    inner = [int(v) for v in rng.integers(1, max_rank + 1, size=2 * d - 1)]
    return LayerShape(nm, mm, tuple([1] + inner + [1]))


def pack(cores: Sequence[np.ndarray], diags: Sequence[np.ndarray]) -> np.ndarray:
    """Concatenate cores (row-major) then diagonals into one float32 vector.

    This is the packed parameter layout the library reads: G_1..G_2d each
    (r_{k-1}, s_k, r_k) row-major, then D_1..D_{2d-1}.
    """
    parts = [np.ascontiguousarray(c, dtype=np.float32).ravel() for c in cores]
    parts += [np.ascontiguousarray(dv, dtype=np.float32).ravel() for dv in diags]
    return np.concatenate(parts) if parts else np.zeros(0, np.float32)


def unpack(shape: LayerShape, flat: np.ndarray):
    """Inverse of :func:`pack` for one layer shape."""
    cores, diags, off = [], [], 0
    for cs in shape.core_shapes():
        n = int(np.prod(cs))
        cores.append(np.asarray(flat[off:off + n]).reshape(cs))
        off += n
    for n in shape.diag_sizes():
        diags.append(np.asarray(flat[off:off + n]).copy())
        off += n
    assert off == flat.size, (off, flat.size)
    return cores, diags


# ---------------------------------------------------------------------------
# TT-matrix (TTM) embedding tables: E (V x Dm), V = prod m_k rows (the
# vocabulary), Dm = prod n_k columns; cores F_k of shape (r_{k-1}, m_k, n_k,
# r_k), r_0 = r_d = 1, with a diagonal on every internal link as for the TT
# layers.  Packed like the TT layers: F_1..F_d row-major, then D_1..D_{d-1}.


@dataclasses.dataclass(frozen=True)
class TtmShape:
    row_modes: Tuple[int, ...]   # m_1..m_d, V = prod
    col_modes: Tuple[int, ...]   # n_1..n_d, Dm = prod
    ranks: Tuple[int, ...]       # r_0..r_d, r_0 = r_d = 1

    @property
    def d(self) -> int:
        return len(self.row_modes)

    @property
    def V(self) -> int:
        return int(np.prod(self.row_modes))

    @property
    def Dm(self) -> int:
        return int(np.prod(self.col_modes))

    def core_shapes(self):
        return [(self.ranks[k], self.row_modes[k], self.col_modes[k], self.ranks[k + 1])
                for k in range(self.d)]

    def diag_sizes(self):
        return [self.ranks[k] for k in range(1, self.d)]


@dataclasses.dataclass(frozen=True)
class TtmWorkload:
    name: str
    shape: TtmShape
    batch: int        # indices looked up per step
    vocab: int        # indices are drawn from [0, vocab) (vocab <= V)
    zipf_s: float     # P(rank k) proportional to 1 / (k + 1)^s
    core_std: float
    description: str = ""


_TTM_BERT = TtmShape((32, 32, 32), (8, 8, 12), (1, 30, 30, 1))

TTM_WORKLOADS = {
    f"ttm_emb_{b // 1000}k": TtmWorkload(
        f"ttm_emb_{b // 1000}k", _TTM_BERT, b, 30522, 1.0, 0.2,
        description=f"TTM embedding 30522(->32768 as (32,32,32)) x 768 as (8,8,12), "
                    f"ranks 30, D~U(0.5,1.5), {b} Zipf(1.0) indices, fp32")
    for b in (10000, 20000, 40000)
}


@dataclasses.dataclass
class TtmInputs:
    cores: List[np.ndarray]   # float32 (r_{k-1}, m_k, n_k, r_k)
    diags: List[np.ndarray]   # float32
    idx: np.ndarray           # (B,) int32 row indices
    dout: np.ndarray          # (B, Dm) float32 upstream gradient


def zipf_indices(rng: np.random.Generator, n: int, vocab: int, s: float) -> np.ndarray:
    """n indices in [0, vocab): frequency rank k has probability
    proportional to 1/(k+1)^s (inverse-CDF sampling), and a seeded
    permutation maps ranks to indices so frequent rows are spread out."""
    w = 1.0 / np.arange(1, vocab + 1, dtype=np.float64) ** s
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    perm = rng.permutation(vocab)
    ranks = np.searchsorted(cdf, rng.random(n), side="right")
    ranks = np.minimum(ranks, vocab - 1)
    return perm[ranks].astype(np.int32)


def draw_ttm(w: TtmWorkload, seed: int = 0, batch: Optional[int] = None) -> TtmInputs:
    """Draw order: cores, diagonals, index permutation and indices, dout."""
    B = w.batch if batch is None else int(batch)
    rng = np.random.Generator(np.random.PCG64(seed))
    cores = [(rng.standard_normal(cs) * w.core_std).astype(np.float32)
             for cs in w.shape.core_shapes()]
    diags = [rng.uniform(0.5, 1.5, n).astype(np.float32) for n in w.shape.diag_sizes()]
    idx = zipf_indices(rng, B, w.vocab, w.zipf_s)
    dout = rng.standard_normal((B, w.shape.Dm)).astype(np.float32)
    return TtmInputs(cores, diags, idx, dout)
