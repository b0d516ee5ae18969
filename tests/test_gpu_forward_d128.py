"""The bf16 forward with head_dim 128 on the tensor cores against the fp64
oracle at the bf16 bar (max abs error <= 2e-2, per-row cosine >= 0.999; page
"Source code for gigl.nn.packed_attention", module docstring, "Constraints":
any head_dim that is a multiple of 8).

The kernel writes each tile's P over its own score columns (the two tiles'
scores and 128-wide outputs fill tensor memory), so these tests cover the
ordering that makes that safe: many blocks per item (long sequences), many
items per CTA, every multi-head item shape, and bitwise determinism.
"""

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCALE = 1.0 / np.sqrt(128)


def _run(lengths, heads, seed, scale=SCALE):
    x = workloads.make_custom(lengths, heads, 128, torch.bfloat16, seed=seed)
    s = int(max(lengths))
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    cu_d = torch.from_numpy(cu).to(DEV)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    ws = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, len(lengths), q.shape[0], heads,
                                                  128, s), dtype=torch.uint8, device=DEV)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, scale, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    return x, cu, s, (q, k, v, cu_d), out, lse


def _check(x, cu, s, out, lse, scale, what):
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, scale)
    check(out, ref, "bf16", what)
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3, f"{what}: lse"


def test_bf16_d128_runs_on_the_tensor_cores():
    assert pe.pe_attention_kernel(torch.bfloat16, 128) == "tcgen05_bf16_d128"
    assert pe.pe_attention_kernel(torch.bfloat16, 96) == "simt_ffma"


def test_pair_tile_edges():
    lengths = [128, 129, 256, 257, 384, 385, 512, 1, 100, 640, 1000]
    x, cu, s, _, out, lse = _run(lengths, 5, seed=91)
    _check(x, cu, s, out, lse, SCALE, "d128 pair edges")


@pytest.mark.parametrize("heads", [1, 2, 3, 5, 7, 12])
def test_multi_head_items(heads):
    rng = np.random.default_rng(100 + heads)
    lengths = np.concatenate([[1, 2, 63, 64, 65, 127, 128, 129, 130], rng.integers(1, 129, 50),
                              rng.integers(129, 300, 3)])
    rng.shuffle(lengths)
    x, cu, s, _, out, lse = _run(lengths, heads, seed=101 + heads)
    _check(x, cu, s, out, lse, SCALE, f"d128 multi-head, {heads} heads")


def test_many_items_per_cta():
    rng = np.random.default_rng(92)
    lengths = rng.integers(1, 700, 400).astype(np.int32)
    x, cu, s, _, out, lse = _run(lengths, 4, seed=93)
    _check(x, cu, s, out, lse, SCALE, "d128 many items")


def test_long_sequences():
    lengths = [4096, 3001, 2500, 1]
    x, cu, s, _, out, lse = _run(lengths, 2, seed=94)
    _check(x, cu, s, out, lse, SCALE, "d128 long sequences")


def test_deterministic():
    lengths = [700, 3, 129, 64, 1500]
    _, _, s, (q, k, v, cu_d), out, lse = _run(lengths, 3, seed=95)
    out2, lse2 = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, SCALE, need_lse=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_backward_through_the_d128_forward():
    """The backward (CUDA cores for head_dim 128) consumes this forward's output
    and log-sum-exp; the gradients match the oracle's."""
    lengths = [1, 63, 64, 65, 128, 129, 300, 2, 257]
    x = workloads.make_custom(lengths, 2, 128, torch.bfloat16, seed=96, with_dout=True)
    s = max(lengths)
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    cu_d = torch.from_numpy(cu).to(DEV)
    q, k, v, do = (t.to(DEV) for t in (x.q, x.k, x.v, x.dout))
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, SCALE, need_lse=True)
    dq, dk, dv = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu_d, s, SCALE)
    rq, rk, rv = oracle.attention_bwd(x.q, x.k, x.v, x.dout, cu, SCALE)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check(got, want, "bf16", f"d128 {name}")
