"""Local (sliding-window) packed attention on the GPU against the fp64 oracle
with the same window: forward (full and first-token query) and backward, on
every kernel family, with ragged lengths that cross tile and block edges and
windows that are empty-sided, one-sided, narrower than a block, wider than a
block, and wider than every sequence."""

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

# Lengths crossing the 64-row (FFMA) and 128/256-row (tensor-core) tile edges.
LENGTHS = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 700, 2, 1100]
WINDOWS = [(64, 64), (0, 0), (3, 7), (130, 5), (300, 0), (0, 260), (-1, 40), (90, -1),
           (5000, 5000)]


def _lse_tol(tag):
    return 1e-4 if tag == "fp32" else 2e-3


def _inputs(dtype, d, lengths=LENGTHS, heads=2, seed=31, dout=False):
    x = workloads.make_custom(lengths, heads, d, dtype, seed=seed, with_dout=dout)
    s = max(lengths)
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    return x, s, cu, torch.from_numpy(cu).to(DEV)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.float32, 32), (torch.bfloat16, 128)])
@pytest.mark.parametrize("window", WINDOWS)
def test_local_forward_matches_oracle(dtype, d, window):
    x, s, cu, cu_d = _inputs(dtype, d)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, s, window[0], window[1], scale,
                                                need_lse=True)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, scale, window=window)
    tag = "fp32" if dtype == torch.float32 else "bf16"
    check(out, ref, tag, f"local out {window}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(tag)


def test_local_forward_uses_the_tensor_core_kernel():
    assert pe.pe_attention_kernel(torch.bfloat16, 64) == "tcgen05_bf16_d64"
    assert pe.pe_attention_kernel(torch.bfloat16, 64, backward=True) == "tcgen05_bf16_d64_bwd"


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("window", [(-1, -1), (5000, 5000), (1099, 1099)])
def test_unbounded_window_is_bitwise_full_attention(dtype, d, window):
    """A negative bound, or one reaching every key, runs the full-attention path."""
    x, s, cu, cu_d = _inputs(dtype, d)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, 0.125, need_lse=True)
    out2, lse2 = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, s, window[0], window[1], 0.125,
                                                  need_lse=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.float32, 16)])
@pytest.mark.parametrize("right", [0, 10, 200, 1500])
def test_local_first_token_query(dtype, d, right):
    """A first-token query sits at position 0: it sees keys 0 .. right."""
    lengths = LENGTHS + [3000, 2500]   # long enough for the 1024-key chunk split
    x, s, cu, cu_d = _inputs(dtype, d, lengths=lengths)
    first = cu[:-1].astype(np.int64)
    q = x.q[first].contiguous()
    k, v = x.k.to(DEV), x.v.to(DEV)
    out, lse = pe.pe_packed_attention_fwd_local(q.to(DEV), k, v, cu_d, s, 7, right, 0.2,
                                                query_is_first_token=True, need_lse=True)
    ref, ref_lse = oracle.attention_fwd(q, x.k, x.v, cu, s, 0.2, first_token=True,
                                        window=(7, right))
    tag = "fp32" if dtype == torch.float32 else "bf16"
    check(out, ref, tag, f"first-token right={right}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(tag)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.float32, 32), (torch.bfloat16, 128)])
@pytest.mark.parametrize("window", [(64, 64), (0, 0), (3, 150), (200, 1), (-1, 30)])
@pytest.mark.parametrize("first_token", [False, True])
def test_local_backward_matches_oracle(dtype, d, window, first_token):
    lengths = [1, 63, 65, 128, 129, 300, 2, 257, 520]
    x, s, cu, cu_d = _inputs(dtype, d, lengths=lengths, seed=33, dout=True)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t.to(DEV) for t in (x.q, x.k, x.v, x.dout))
    if first_token:
        first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
        q, do = q[first].contiguous(), do[first].contiguous()
    out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, s, window[0], window[1], scale,
                                                query_is_first_token=first_token, need_lse=True)
    dq, dk, dv = pe.pe_packed_attention_bwd_local(do, q, k, v, out, lse, cu_d, s, window[0],
                                                  window[1], scale,
                                                  query_is_first_token=first_token)
    tag = "fp32" if dtype == torch.float32 else "bf16"
    saved = None
    if tag == "bf16" and first_token:
        # First-token bf16 gradients against the oracle's own output rounded to
        # bf16, as the backward op forms Delta from the saved output (a
        # near-cancelled dS_j takes its sign from that rounding).
        ref_out, _ = oracle.attention_fwd(q.cpu(), x.k, x.v, cu, s, scale, first_token=True,
                                          window=window)
        saved = torch.from_numpy(ref_out).to(torch.bfloat16)
    rq, rk, rv = oracle.attention_bwd(q.cpu(), x.k, x.v, do.cpu(), cu, scale,
                                      first_token=first_token, window=window, out=saved)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(got, want, tag, f"local {name} {window} first_token={first_token}")


def test_local_backward_is_deterministic():
    x, s, cu, cu_d = _inputs(torch.bfloat16, 64, lengths=[700, 300, 129], seed=35, dout=True)
    q, k, v, do = (t.to(DEV) for t in (x.q, x.k, x.v, x.dout))
    out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, s, 64, 64, 0.125, need_lse=True)
    g1 = pe.pe_packed_attention_bwd_local(do, q, k, v, out, lse, cu_d, s, 64, 64, 0.125)
    g2 = pe.pe_packed_attention_bwd_local(do, q, k, v, out, lse, cu_d, s, 64, 64, 0.125)
    assert all(torch.equal(a, b) for a, b in zip(g1, g2))


def test_local64_long_documents_sampled_rows():
    """Long documents with ModernBERT's local-64 window at full length, checked
    on sampled (token, head) rows computed one by one by the oracle."""
    wl = workloads.WORKLOADS["longdoc_bf16"]
    lengths = workloads.draw_lengths("longdoc_bf16", np.random.default_rng(0))[:6]
    x = workloads.make_custom(lengths.tolist(), wl.num_heads, wl.head_dim, torch.bfloat16,
                              seed=39)
    _, cu, n = oracle.pack_sequences(x.lengths, wl.max_seq_len)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    cu_d = torch.from_numpy(cu).to(DEV)
    out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, wl.max_seq_len, 64, 64, wl.scale,
                                                need_lse=True)
    rng = np.random.default_rng(37)
    rows = np.concatenate([rng.integers(0, n, 400), cu[:-1], cu[1:] - 1]).astype(np.int64)
    hs = rng.integers(0, wl.num_heads, rows.shape[0]).astype(np.int64)
    ref, ref_lse = oracle.attention_fwd_rows(x.q, x.k, x.v, cu, wl.scale, False, rows, hs,
                                             window=(64, 64))
    got = out[torch.from_numpy(rows).to(DEV), torch.from_numpy(hs).to(DEV)]
    check(got, ref, "bf16", "local-64 long documents")
    got_lse = lse[torch.from_numpy(hs).to(DEV), torch.from_numpy(rows).to(DEV)]
    assert float(np.abs(to64(got_lse) - ref_lse).max()) <= 2e-3


@pytest.mark.parametrize("workload,window", [("longdoc_bf16", (64, 64)), ("longdoc_bf16", (3, 200)),
                                             ("train_bf16", (64, 64))])
def test_local_full_workload_pipeline_completes(workload, window):
    """Whole workloads (many items per CTA, so the K/V rings wrap many times,
    and single-tile items next to two-tile ones): every pipeline wait completes
    (device status clear) and sampled rows match the oracle, forward and, for
    the training workload, backward."""
    wl = workloads.WORKLOADS[workload]
    x = workloads.make_inputs(workload)
    _, cu, n = oracle.pack_sequences(x.lengths, wl.max_seq_len)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    cu_d = torch.from_numpy(cu).to(DEV)
    b = len(x.lengths)
    ws = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, b, n, wl.num_heads, wl.head_dim,
                                                  wl.max_seq_len, backward=True),
                     dtype=torch.uint8, device=DEV)
    out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, wl.max_seq_len, window[0],
                                                window[1], wl.scale, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    rng = np.random.default_rng(41)
    rows = np.concatenate([rng.integers(0, n, 300), cu[:-1], cu[1:] - 1]).astype(np.int64)
    hs = rng.integers(0, wl.num_heads, rows.shape[0]).astype(np.int64)
    ref, _ = oracle.attention_fwd_rows(x.q, x.k, x.v, cu, wl.scale, False, rows, hs,
                                       window=window)
    got = out[torch.from_numpy(rows).to(DEV), torch.from_numpy(hs).to(DEV)]
    check(got, ref, "bf16", f"{workload} local {window}")
    if wl.backward:
        do = x.dout.to(DEV)
        dq, dk, dv = pe.pe_packed_attention_bwd_local(do, q, k, v, out, lse, cu_d,
                                                      wl.max_seq_len, window[0], window[1],
                                                      wl.scale, workspace=ws)
        assert pe.pe_read_device_status(ws) == 0
        rq, rk, rv = oracle.attention_bwd(x.q, x.k, x.v, x.dout, cu, wl.scale, window=window)
        for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            check_grad(got, want, "bf16", f"{workload} local {name}")
