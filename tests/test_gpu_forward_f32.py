"""The fp32 forward on the tensor cores (head_dim 64, full attention) against
the fp64 oracle at the fp32 bar (max abs error <= 1e-4; page "Source code for
gigl.nn.packed_attention", _varlen_attention: the memory-efficient kernel runs
in fp32 "which inference needs for accuracy").

Every fp32 operand is split into bf16 hi and lo parts and each product taken
as hi*hi + hi*lo + lo*hi, so these tests also bound the error of that split:
ragged lengths around the 64/128/256-row item edges, every multi-head item
shape, many items per CTA, long sequences, and bitwise determinism.
"""

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import FP32_ATOL, check, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(lengths, heads, seed, scale=0.125, workspace=True):
    x = workloads.make_custom(lengths, heads, 64, torch.float32, seed=seed)
    s = int(max(lengths))
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    cu_d = torch.from_numpy(cu).to(DEV)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    ws = torch.empty(pe.attention_workspace_bytes(torch.float32, len(lengths), q.shape[0], heads,
                                                  64, s), dtype=torch.uint8, device=DEV)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, scale, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    return x, cu, s, (q, k, v, cu_d), out, lse


def _check_against_oracle(x, cu, s, out, lse, scale, what):
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, scale)
    check(out, ref, "fp32", what)
    assert float(np.abs(to64(lse) - ref_lse).max()) <= FP32_ATOL, f"{what}: lse"


def test_fp32_d64_runs_on_the_tensor_cores():
    assert pe.pe_attention_kernel(torch.float32, 64) == "tcgen05_f32_d64"


def test_pair_tile_edges():
    # Work items hit every case of the 256-row query pair: second tile empty,
    # partial, both full, a single row; plus a one-token sequence.
    lengths = [128, 129, 256, 257, 384, 385, 512, 1, 100, 640, 1000]
    x, cu, s, _, out, lse = _run(lengths, 5, seed=61)
    _check_against_oracle(x, cu, s, out, lse, 0.125, "f32 pair edges")


@pytest.mark.parametrize("heads", [1, 2, 3, 5, 7, 12])
def test_multi_head_items(heads):
    """Sequences of at most 128 tokens run one head per query tile, those of at
    most 64 tokens two heads per tile; an odd head count leaves a partial item."""
    rng = np.random.default_rng(80 + heads)
    lengths = np.concatenate([[1, 2, 63, 64, 65, 127, 128, 129, 130], rng.integers(1, 129, 50),
                              rng.integers(129, 300, 3)])
    rng.shuffle(lengths)
    x, cu, s, _, out, lse = _run(lengths, heads, seed=81 + heads)
    _check_against_oracle(x, cu, s, out, lse, 0.125, f"f32 multi-head, {heads} heads")


def test_many_items_per_cta():
    rng = np.random.default_rng(62)
    lengths = rng.integers(1, 700, 400).astype(np.int32)
    x, cu, s, _, out, lse = _run(lengths, 8, seed=63)
    _check_against_oracle(x, cu, s, out, lse, 0.125, "f32 many items")


def test_long_sequences():
    lengths = [4096, 3001, 2500, 1]
    x, cu, s, _, out, lse = _run(lengths, 2, seed=64)
    _check_against_oracle(x, cu, s, out, lse, 0.125, "f32 long sequences")


def test_graph_workload_matches_oracle_elementwise():
    """The graph-transformer workload (1024 sequences, ~90k tokens, 8 x 64)
    element by element against the oracle."""
    x = workloads.make_inputs("graph_fp32")
    wl = x.workload
    _, cu, _ = oracle.pack_sequences(x.lengths, wl.max_seq_len)
    cu_d = torch.from_numpy(cu).to(DEV)
    out, lse = pe.pe_packed_attention_fwd(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), cu_d,
                                          wl.max_seq_len, wl.scale, need_lse=True)
    _check_against_oracle(x, cu, wl.max_seq_len, out, lse, wl.scale, "graph workload")


def test_deterministic():
    lengths = [700, 3, 129, 64, 1500]
    _, _, s, (q, k, v, cu_d), out, lse = _run(lengths, 3, seed=65)
    out2, lse2 = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, 0.125, need_lse=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_other_scales():
    lengths = [300, 77, 1, 520]
    for scale in (0.05, 0.3):
        x, cu, s, _, out, lse = _run(lengths, 2, seed=66, scale=scale)
        _check_against_oracle(x, cu, s, out, lse, scale, f"f32 scale {scale}")
