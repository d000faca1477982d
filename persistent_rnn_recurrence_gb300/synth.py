"""Seeded synthetic inputs for the vanilla ReLU RNN layer.

This module only draws random numbers and lays them out; it holds none of the
recurrence's arithmetic.  The CUDA path's tests, the benchmark and the CPU
oracle's tests all take their inputs from here, so both sides see identical
bytes.

Workload shapes follow the layer sizes, batch size, densities and step count
that the sparse persistent RNN summary page (atlas.scime.ai, "Measured effects
reported in the paper" table) measures on: layer sizes 1152-5760, batch 4,
densities 1-10 %, 256 timesteps.  Weight scales give the recurrent matrix a
spectral radius of about 0.9 (std = 0.9 / sqrt(fan-in of the row)), so the
recurrence neither dies out nor blows up over 256 steps.

Draw order, per problem, from ``numpy.random.default_rng(seed)``:
x, Wx, Wh (sparse: the column sets row by row, then the values), b, h0.
fp16 tensors are rounded to nearest-even by ``astype(np.float16)``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = ["Problem", "make_problem", "named_problem", "NAMED", "sweep_points",
           "sparse_k", "make_pruned_pair", "StackProblem", "make_stack_problem"]


@dataclasses.dataclass
class Problem:
    """One forward problem: h_t = ReLU(Wx x_t + Wh h_{t-1} + b), t < T."""
    name: str
    T: int
    B: int
    H: int
    I: int
    wdtype: str                      # "f32" or "f16": storage type of Wx and Wh
    x: np.ndarray                    # float32 [T, B, I]
    Wx: np.ndarray                   # wdtype [H, I]
    b: np.ndarray                    # float32 [H]
    h0: Optional[np.ndarray]         # float32 [B, H] or None (zeros)
    Wh: Optional[np.ndarray] = None  # wdtype [H, H] (dense problems)
    vals: Optional[np.ndarray] = None  # float16 [H, k] (sparse) or [nnz] (compressed rows)
    cols: Optional[np.ndarray] = None  # uint16 [H, k] ascending, distinct per row; or [nnz]
    seed: int = 0
    row_ptr: Optional[np.ndarray] = None  # int32 [H+1]: unbalanced compressed-row form

    @property
    def sparse(self) -> bool:
        return self.vals is not None

    @property
    def k(self) -> int:
        """Non-zeros per row (compressed rows: the longest row)."""
        if self.row_ptr is not None:
            return int(np.diff(self.row_ptr).max())
        return int(self.vals.shape[1]) if self.sparse else self.H

    @property
    def nnz(self) -> int:
        if self.row_ptr is not None:
            return int(self.vals.size)
        return self.H * self.k


def sparse_k(H: int, density: float) -> int:
    """Non-zeros per row of a row-balanced matrix: floor(density * H), >= 1."""
    return max(1, int(math.floor(density * H + 1e-9)))


def _np_dtype(wdtype: str):
    if wdtype == "f16":
        return np.float16
    if wdtype == "f32":
        return np.float32
    raise ValueError(f"unknown weight dtype {wdtype!r}")


def _row_balanced_cols(rng: np.random.Generator, H: int, k: int) -> np.ndarray:
    """k distinct uniformly random columns per row, each row sorted ascending."""
    cols = np.empty((H, k), dtype=np.uint16)
    for r in range(H):
        cols[r] = np.sort(rng.choice(H, size=k, replace=False)).astype(np.uint16)
    return cols


def make_problem(*, H: int, B: int, T: int, I: Optional[int] = None,
                 density: float = 1.0, k: Optional[int] = None,
                 wdtype: str = "f16", seed: int = 0,
                 wx_std: Optional[float] = None, wh_std: Optional[float] = None,
                 x_std: float = 1.0, b_range: float = 0.1,
                 h0_std: Optional[float] = None, name: str = "custom") -> Problem:
    """Draw one problem.  ``density < 1`` (or an explicit ``k``) makes Wh
    row-balanced sparse with fp16 values and uint16 column indices."""
    I = H if I is None else I
    if T < 0 or B < 0 or H <= 0 or I <= 0:
        raise ValueError("need T, B >= 0 and H, I > 0")
    sparse = k is not None or density < 1.0
    if sparse:
        k = sparse_k(H, density) if k is None else int(k)
        if not (0 < k <= H):
            raise ValueError("need 0 < k <= H")
        if H > 65536:
            raise ValueError("uint16 column indices need H <= 65536")
        if wdtype != "f16":
            raise ValueError("sparse weights are fp16 values + uint16 indices")
    fan_in = k if sparse else H
    wx_std = 0.9 / math.sqrt(H) if wx_std is None else wx_std
    wh_std = 0.9 / math.sqrt(fan_in) if wh_std is None else wh_std
    wt = _np_dtype(wdtype)

    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, x_std, size=(T, B, I)).astype(np.float32)
    Wx = rng.normal(0.0, wx_std, size=(H, I)).astype(wt)
    Wh = vals = cols = None
    if sparse:
        cols = _row_balanced_cols(rng, H, k)
        vals = rng.normal(0.0, wh_std, size=(H, k)).astype(np.float16)
    else:
        Wh = rng.normal(0.0, wh_std, size=(H, H)).astype(wt)
    b = rng.uniform(-b_range, b_range, size=(H,)).astype(np.float32)
    h0 = None
    if h0_std is not None:
        h0 = rng.normal(0.0, h0_std, size=(B, H)).astype(np.float32)
    return Problem(name=name, T=T, B=B, H=H, I=I, wdtype=wdtype, x=x, Wx=Wx,
                   b=b, h0=h0, Wh=Wh, vals=vals, cols=cols, seed=seed)


# The named workloads.  Seeds are 1000 + position in this table.
NAMED = {
    # dense fp32 weights, small: the case the oracle finishes in well under a second
    "dense_f32_h256_b4_t32": dict(H=256, B=4, T=32, wdtype="f32"),
    # dense fp16 weights, the ablation's layer size, h0 ~ N(0, 0.1)
    "dense_f16_h1152_b4_t256": dict(H=1152, B=4, T=256, wdtype="f16", h0_std=0.1),
    # sparse 10 %: 179 non-zeros per row; Wx ~ N(0, 1/sqrt(H))
    "sparse_f16_h1792_d10_b4_t256": dict(H=1792, B=4, T=256, k=179, wdtype="f16",
                                         wx_std=1.0 / math.sqrt(1792)),
    # large sparse, 1 % (57 per row) and 5 % (288 per row)
    "sparse_f16_h5760_d1_b4_t256": dict(H=5760, B=4, T=256, k=57, wdtype="f16",
                                        wx_std=1.0 / math.sqrt(5760)),
    "sparse_f16_h5760_d5_b4_t256": dict(H=5760, B=4, T=256, k=288, wdtype="f16",
                                        wx_std=1.0 / math.sqrt(5760)),
}
_SEEDS = {name: 1000 + i for i, name in enumerate(NAMED)}


def named_problem(name: str, *, T: Optional[int] = None,
                  B: Optional[int] = None) -> Problem:
    """One of the named workloads; ``T``/``B`` may shrink it (same seed)."""
    spec = dict(NAMED[name])
    if T is not None:
        spec["T"] = T
    if B is not None:
        spec["B"] = B
    return make_problem(name=name, seed=_SEEDS[name], **spec)


def sweep_points():
    """The persistent-vs-per-step sweep: H x B x density, T = 256, fp16.
    Yields (name, kwargs) in a fixed order; seed = 2000 + linear index."""
    i = 0
    for H in (1152, 2304, 4096):
        for B in (1, 4, 16, 32):
            for d in (1.0, 0.25, 0.10, 0.01):
                kw = dict(H=H, B=B, T=256, wdtype="f16", seed=2000 + i)
                if d < 1.0:
                    kw["k"] = sparse_k(H, d)
                name = f"sweep_h{H}_b{B}_d{int(round(d * 100))}"
                yield name, kw
                i += 1


def make_pruned_pair(*, H: int, B: int, T: int, density: float, seed: int,
                     row_sigma: float = 0.25, name: str = "pruned"):
    """The same layer pruned two ways, for the balanced-versus-unbalanced
    comparison: a dense score matrix Z[r][c] = s_r * N(0,1) with per-row
    scales s_r = exp(row_sigma * N(0,1)) (rows of a trained layer differ in
    magnitude), then
      * unbalanced: keep the floor(density*H*H) largest |Z| over the whole
        matrix (global magnitude pruning) -> rows of unequal length;
      * balanced: keep the k = floor(density*H) largest |Z| of every row.
    Kept positions get fresh values N(0, 0.9/sqrt(row length)) (fp16), so both
    recurrences stay stable.  x, Wx, b are shared.  Returns (unbalanced,
    balanced) Problems; the unbalanced one is in compressed-row form."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.0, size=(T, B, H)).astype(np.float32)
    Wx = rng.normal(0.0, 1.0 / math.sqrt(H), size=(H, H)).astype(np.float16)
    b = rng.uniform(-0.1, 0.1, size=(H,)).astype(np.float32)
    scale = np.exp(row_sigma * rng.standard_normal(H)).astype(np.float32)
    Z = np.abs(rng.standard_normal((H, H)).astype(np.float32)) * scale[:, None]
    k = sparse_k(H, density)
    keep = H * k
    thr = np.partition(Z.ravel(), Z.size - keep)[Z.size - keep]
    mask = Z >= thr
    lens = mask.sum(axis=1)
    row_ptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cols_u = np.nonzero(mask)[1].astype(np.uint16)            # row-major, ascending per row
    vals_u = np.concatenate([rng.normal(0.0, 0.9 / math.sqrt(max(n, 1)), size=n)
                             for n in lens]).astype(np.float16)
    top = np.argpartition(-Z, k - 1, axis=1)[:, :k]
    cols_b = np.sort(top, axis=1).astype(np.uint16)
    vals_b = rng.normal(0.0, 0.9 / math.sqrt(k), size=(H, k)).astype(np.float16)
    unb = Problem(name=name + "_unbalanced", T=T, B=B, H=H, I=H, wdtype="f16", x=x, Wx=Wx,
                  b=b, h0=None, vals=vals_u, cols=cols_u, seed=seed, row_ptr=row_ptr)
    bal = Problem(name=name + "_balanced", T=T, B=B, H=H, I=H, wdtype="f16", x=x, Wx=Wx,
                  b=b, h0=None, vals=vals_b, cols=cols_b, seed=seed)
    return unb, bal


@dataclasses.dataclass
class StackProblem:
    """L dense layers: layer 0 reads x [T,B,I], layer l > 0 reads layer l-1's
    output; every layer has H units.  layers[l] = (Wx [H, I_l], Wh [H, H],
    b [H]); h0 [L, B, H] or None (zeros)."""
    name: str
    T: int
    B: int
    H: int
    I: int
    L: int
    wdtype: str
    x: np.ndarray
    layers: list
    h0: Optional[np.ndarray]
    seed: int = 0


def make_stack_problem(*, L: int, H: int, B: int, T: int, I: Optional[int] = None,
                       wdtype: str = "f16", seed: int = 0, h0_std: Optional[float] = None,
                       name: str = "stack") -> StackProblem:
    """Draw order from ``default_rng(seed)``: x ~ N(0, 1); then per layer
    Wx ~ N(0, 0.9/sqrt(I_l)), Wh ~ N(0, 0.9/sqrt(H)), b ~ U(-0.1, 0.1);
    then h0 ~ N(0, h0_std) if asked."""
    I = H if I is None else I
    if L < 1 or T < 0 or B < 0 or H <= 0 or I <= 0:
        raise ValueError("need L >= 1, T, B >= 0 and H, I > 0")
    wt = _np_dtype(wdtype)
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 1.0, size=(T, B, I)).astype(np.float32)
    layers = []
    for l in range(L):
        il = I if l == 0 else H
        Wx = rng.normal(0.0, 0.9 / math.sqrt(il), size=(H, il)).astype(wt)
        Wh = rng.normal(0.0, 0.9 / math.sqrt(H), size=(H, H)).astype(wt)
        b = rng.uniform(-0.1, 0.1, size=(H,)).astype(np.float32)
        layers.append((Wx, Wh, b))
    h0 = None
    if h0_std is not None:
        h0 = rng.normal(0.0, h0_std, size=(L, B, H)).astype(np.float32)
    return StackProblem(name=name, T=T, B=B, H=H, I=I, L=L, wdtype=wdtype, x=x, layers=layers,
                        h0=h0, seed=seed)
