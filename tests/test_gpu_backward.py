"""Packed attention backward on the GPU against the oracle's analytic fp64
gradients (the training-step workload and small ragged cases)."""

import math

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check, check_grad, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(x, s, scale, first_token=False):
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    cu_d = torch.from_numpy(cu).to(DEV)
    q, k, v, do = (t.to(DEV) for t in (x.q, x.k, x.v, x.dout))
    if first_token:
        first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
        q, do = q[first].contiguous(), do[first].contiguous()
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, scale,
                                          query_is_first_token=first_token, need_lse=True)
    grads = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu_d, s, scale,
                                       query_is_first_token=first_token)
    return cu, (q, k, v, do), out, grads


def test_training_step_workload_matches_oracle():
    x = workloads.make_inputs("train_bf16")
    wl = x.workload
    cu, _, out, (dq, dk, dv) = _run(x, wl.max_seq_len, wl.scale)
    ref, _ = oracle.attention_fwd(x.q, x.k, x.v, cu, wl.max_seq_len, wl.scale)
    check(out, ref, "bf16", "train out")
    rq, rk, rv = oracle.attention_bwd(x.q, x.k, x.v, x.dout, cu, wl.scale)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check(got, want, "bf16", f"train {name}")


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.bfloat16, 64),
                                     (torch.float32, 8), (torch.float32, 32),
                                     (torch.bfloat16, 128)])
@pytest.mark.parametrize("first_token", [False, True])
def test_ragged_gradients(dtype, d, first_token):
    lengths = [1, 63, 64, 65, 128, 129, 300, 2, 257]
    x = workloads.make_custom(lengths, 2, d, dtype, seed=21, with_dout=True)
    s = max(lengths)
    scale = 1.0 / math.sqrt(d)
    cu, (q, k, v, do), out, (dq, dk, dv) = _run(x, s, scale, first_token)
    qq = q.cpu() if first_token else x.q
    dd = do.cpu() if first_token else x.dout
    rq, rk, rv = oracle.attention_bwd(qq, x.k, x.v, dd, cu, scale, first_token=first_token)
    tag = "fp32" if dtype == torch.float32 else "bf16"
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check(got, want, tag, f"{name} d={d} first_token={first_token}")


def test_backward_is_deterministic():
    x = workloads.make_custom([700, 3, 129, 64], 3, 64, torch.bfloat16, seed=22, with_dout=True)
    cu, (q, k, v, do), out, g1 = _run(x, 700, 0.125)
    cu_d = torch.from_numpy(cu).to(DEV)
    _, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, 700, 0.125, need_lse=True)
    g2 = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu_d, 700, 0.125)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_gradient_invariants_hold_per_sequence():
    """Rows of dS sum to zero, so dk sums to zero per (sequence, head); dv sums
    to the sum of dO over the sequence."""
    x = workloads.make_custom([90, 33, 250], 2, 64, torch.float32, seed=23, with_dout=True)
    cu, (_, _, _, do), _, (_, dk, dv) = _run(x, 250, 0.125)
    for i in range(3):
        rows = slice(int(cu[i]), int(cu[i + 1]))
        assert float(dk[rows].double().sum(0).abs().max()) <= 1e-4
        assert float((dv[rows].double().sum(0) - do[rows].double().sum(0)).abs().max()) <= 1e-4


@pytest.mark.parametrize("heads", [1, 3, 12])
def test_two_head_items_gradients(heads):
    """Sequences of at most 64 tokens run two heads per backward work item
    (rows 0-63 of every tile one head, rows 64-127 the next); an odd head count
    leaves a one-head item. Lengths sit on both sides of 64 and 128."""
    rng = np.random.default_rng(70 + heads)
    lengths = np.concatenate([[1, 2, 63, 64, 65, 127, 128, 129], rng.integers(1, 65, 60),
                              rng.integers(65, 400, 4)])
    rng.shuffle(lengths)
    x = workloads.make_custom(lengths, heads, 64, torch.bfloat16, seed=71, with_dout=True)
    s = int(lengths.max())
    cu, _, out, (dq, dk, dv) = _run(x, s, 0.125)
    rq, rk, rv = oracle.attention_bwd(x.q, x.k, x.v, x.dout, cu, 0.125)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(got, want, "bf16", f"two-head {name}, {heads} heads")


def test_long_document_backward_matches_oracle():
    """Full attention on documents of 4-8k tokens: a key item streams 33-63
    query blocks and a query item 33-63 key blocks, and none of the lengths is a
    multiple of 128 (4097 leaves a one-row last block). dq, dk and dv against
    the oracle's fp64 gradients at the bar of the outputs; both calls leave the
    device status word clear."""
    lengths = [7937, 6211, 4097]
    x = workloads.make_custom(lengths, 2, 64, torch.bfloat16, seed=31, with_dout=True)
    s, scale = max(lengths), 0.125
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    cu_d = torch.from_numpy(cu).to(DEV)
    q, k, v, do = (t.to(DEV) for t in (x.q, x.k, x.v, x.dout))
    n = k.shape[0]
    ws_f = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, 3, n, 2, 64, s),
                       dtype=torch.uint8, device=DEV)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, scale, need_lse=True,
                                          workspace=ws_f)
    assert pe.pe_read_device_status(ws_f) == 0
    ws_b = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, 3, n, 2, 64, s,
                                                    backward=True),
                       dtype=torch.uint8, device=DEV)
    dq, dk, dv = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu_d, s, scale,
                                            workspace=ws_b)
    assert pe.pe_read_device_status(ws_b) == 0
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, scale)
    check(out, ref, "bf16", "long-document out")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3
    rq, rk, rv = oracle.attention_bwd(x.q, x.k, x.v, x.dout, cu, scale)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check(got, want, "bf16", f"long-document {name}")
