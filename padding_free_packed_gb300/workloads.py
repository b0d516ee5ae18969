"""Seeded synthetic inputs for packed-attention workloads.

This module holds no part of the attention arithmetic. It draws sequence lengths
and N(0, 1) tensors, and nothing else, so that the CUDA path and the fp64 oracle
receive byte-identical inputs while sharing no code.

The shapes and distributions stand in for the workloads the pages describe:

* ``tiny_fp32``        - 8 sequences, lengths uniform in [1, 32], 2 heads x 8
                         (the shape of the doctest in "Source code for
                         gigl.nn.packed_attention", section "Example").
* ``graph_fp32``       - 1024 sequences, lengths round(N(90, 40)) clipped to
                         [1, 256], 8 heads x 64, fp32 (the one-L4 graph
                         transformer of the same page, section "Results": about
                         90 real tokens out of 256, 8 heads, fp32 kernel).
* ``contrastive_bf16`` - 256 queries of 16..48 tokens plus 64 documents whose
                         lengths are lognormal (median 300, sigma 0.8) clipped to
                         [64, 8192], 12 heads x 64, bf16 (the contrastive
                         batches of "packed-encoders 0.1.0", section "Why
                         packing?": queries of about 30 tokens, documents of
                         hundreds to thousands).
* ``longdoc_bf16``     - 32 documents of 2048..8192 tokens, 16 heads x 64, bf16,
                         forward only (the indexing runs of the same README).
* ``train_bf16``       - the ``contrastive_bf16`` shapes with an upstream
                         gradient dO, forward plus backward.

The draw order is fixed: lengths, then q, k, v, then dO, all from one
``numpy.random.default_rng(seed)``. Values are drawn in float64 and cast to the
run dtype with torch (bf16 through fp32, round to nearest even).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_heads: int
    head_dim: int
    dtype: str  # "fp32" or "bf16"
    max_seq_len: int
    backward: bool
    description: str

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", 2, 8, "fp32", 32, False,
        "8 sequences, lengths uniform int [1,32], 2 heads x 8, fp32"),
    "graph_fp32": Workload(
        "graph_fp32", 8, 64, "fp32", 256, False,
        "1024 sequences, lengths round(N(90,40)) clipped to [1,256], 8 heads x 64, fp32"),
    "contrastive_bf16": Workload(
        "contrastive_bf16", 12, 64, "bf16", 8192, False,
        "256 queries U[16,48] + 64 documents lognormal(median 300, sigma 0.8) "
        "clipped to [64,8192], 12 heads x 64, bf16"),
    "longdoc_bf16": Workload(
        "longdoc_bf16", 16, 64, "bf16", 8192, False,
        "32 documents U[2048,8192], 16 heads x 64, bf16, forward only"),
    "train_bf16": Workload(
        "train_bf16", 12, 64, "bf16", 8192, True,
        "contrastive_bf16 shapes, forward + backward with dO ~ N(0,1)"),
}


def draw_lengths(name: str, rng: np.random.Generator) -> np.ndarray:
    """Sequence lengths (int32) for a named workload, drawn first from ``rng``."""
    if name == "tiny_fp32":
        lengths = rng.integers(1, 33, 8)
    elif name == "graph_fp32":
        lengths = np.clip(np.round(rng.normal(90.0, 40.0, 1024)), 1, 256)
    elif name in ("contrastive_bf16", "train_bf16"):
        queries = rng.integers(16, 49, 256)
        docs = np.clip(np.round(rng.lognormal(math.log(300.0), 0.8, 64)), 64, 8192)
        lengths = np.concatenate([queries, docs])
    elif name == "longdoc_bf16":
        lengths = rng.integers(2048, 8193, 32)
    else:
        raise KeyError(f"unknown workload {name!r}")
    return np.ascontiguousarray(lengths.astype(np.int32))


def _normal(rng: np.random.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    x = torch.from_numpy(rng.standard_normal(shape))
    if dtype == torch.bfloat16:
        return x.to(torch.float32).to(torch.bfloat16)
    return x.to(dtype)


@dataclasses.dataclass
class Inputs:
    workload: Workload
    lengths: np.ndarray          # int32 [B]
    q: torch.Tensor              # [N, H, d] in the run dtype (CPU)
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor | None    # [N, H, d] or None

    @property
    def num_tokens(self) -> int:
        return int(self.lengths.astype(np.int64).sum())

    @property
    def num_sequences(self) -> int:
        return int(self.lengths.shape[0])


def make_inputs(name: str, seed: int = 0, with_dout: bool | None = None) -> Inputs:
    """Draws lengths, q, k, v (and dO) for a named workload on the CPU."""
    wl = WORKLOADS[name]
    rng = np.random.default_rng(seed)
    lengths = draw_lengths(name, rng)
    n = int(lengths.astype(np.int64).sum())
    shape = (n, wl.num_heads, wl.head_dim)
    q = _normal(rng, shape, wl.torch_dtype)
    k = _normal(rng, shape, wl.torch_dtype)
    v = _normal(rng, shape, wl.torch_dtype)
    want_dout = wl.backward if with_dout is None else with_dout
    dout = _normal(rng, shape, wl.torch_dtype) if want_dout else None
    return Inputs(wl, lengths, q, k, v, dout)


def make_custom(lengths, num_heads: int, head_dim: int, dtype: torch.dtype,
                seed: int = 0, with_dout: bool = False) -> Inputs:
    """Same draw order as ``make_inputs`` for caller-chosen lengths and shapes."""
    lengths = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
    max_len = int(lengths.max()) if lengths.size else 1
    wl = Workload("custom", num_heads, head_dim,
                  "fp32" if dtype == torch.float32 else "bf16", max_len, with_dout,
                  "caller-chosen lengths")
    rng = np.random.default_rng(seed)
    n = int(lengths.astype(np.int64).sum())
    shape = (n, num_heads, head_dim)
    q = _normal(rng, shape, dtype)
    k = _normal(rng, shape, dtype)
    v = _normal(rng, shape, dtype)
    dout = _normal(rng, shape, dtype) if with_dout else None
    return Inputs(wl, lengths, q, k, v, dout)


def make_padded_inputs(name: str, seed: int = 0, max_sequences: int | None = None,
                       with_dout: bool = False) -> tuple:
    """Lengths plus q, k, v drawn directly as padded ``[B, S, H, d]`` grids.

    The lengths come from the same first draw as ``make_inputs`` (optionally
    only the first ``max_sequences`` of them); every grid row,
    pad rows included, then holds fresh N(0, 1) values drawn in float32 (pad rows
    are never meant to be read). These are the inputs of a padded-to-packed step.
    Returns (lengths, q, k, v), plus a dO grid drawn last when ``with_dout``.
    """
    wl = WORKLOADS[name]
    rng = np.random.default_rng(seed)
    lengths = draw_lengths(name, rng)
    if max_sequences is not None:
        lengths = np.ascontiguousarray(lengths[:max_sequences])
    shape = (int(lengths.shape[0]), wl.max_seq_len, wl.num_heads, wl.head_dim)
    grids = []
    for _ in range(4 if with_dout else 3):
        x = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32))
        grids.append(x.to(wl.torch_dtype) if wl.torch_dtype != torch.float32 else x)
    return (lengths, *grids)


def make_packed_row_inputs(name: str, row_len: int, seed: int = 0, with_dout: bool = False,
                           max_sequences: int | None = None) -> tuple:
    """The workload's documents packed in order into padded rows of ``row_len``
    tokens, as a packing collater lays them out: a document goes to the current
    row if it fits, else it starts a new row. Returns (document lengths, the
    indexed packing mask ``[R, row_len]`` int32 (document i of a row marked i,
    0 = padding), q, k, v grids ``[R, row_len, H, d]``, plus dO when
    ``with_dout``). Lengths are the workload's first draw; grid values are
    fresh N(0, 1) draws in float32, pad positions included."""
    wl = WORKLOADS[name]
    rng = np.random.default_rng(seed)
    lengths = draw_lengths(name, rng)
    if max_sequences is not None:
        lengths = np.ascontiguousarray(lengths[:max_sequences])
    if int(lengths.max()) > row_len:
        raise ValueError(f"a document of {int(lengths.max())} tokens does not fit a row of {row_len}")
    rows, fill = [[]], 0
    for length in lengths.tolist():
        if fill + length > row_len:
            rows.append([])
            fill = 0
        rows[-1].append(length)
        fill += length
    ids = np.zeros((len(rows), row_len), np.int32)
    for r, docs in enumerate(rows):
        n = sum(docs)
        ids[r, :n] = np.repeat(np.arange(1, len(docs) + 1), docs)
    shape = (len(rows), row_len, wl.num_heads, wl.head_dim)
    grids = []
    for _ in range(4 if with_dout else 3):
        x = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32))
        grids.append(x.to(wl.torch_dtype) if wl.torch_dtype != torch.float32 else x)
    return (lengths, ids, *grids)
