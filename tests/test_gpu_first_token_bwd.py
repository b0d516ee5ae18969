"""First-token query backward, streaming form, against the fp64 oracle.

In first-token mode each sequence's single query is its first token (page
"Source code for gigl.nn.packed_attention", function `packed_attention`,
`query_is_first_token`); every key row belongs to one query, so dk and dv are
written row by row as k and v stream through, and dq is summed per sequence.
When a token row is a whole number of 512-byte warp loads (at most 32
elements per lane) and head_dim is 32, 64 or 128, the token range is cut into
equal chunks and the dq sums of sequences that cross chunk edges are added in
chunk order by a second kernel. These tests put sequence boundaries on, next
to and far from those edges, cover every supported row width for both
dtypes, windows (rows beyond the window get zero gradients), the CUDA-core
fallback without room for the partial sums, determinism, and the workloads'
own shapes.

The backward op takes the forward's saved output and forms Delta = dO . O from
it. In bf16 that output is the exact one rounded, and on rows where dP_j and
Delta nearly cancel the rounding decides the sign of dS_j, whatever the
kernel. So bf16 gradients are compared with the oracle's gradients for the
oracle's own output rounded to bf16 (what a saved bf16 output holds); fp32
ones with the exact gradients.
"""

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check_grad, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _mixed_lengths(seed):
    """Short queries, mid-size and long sequences, and lengths at the chunk
    size (64 tokens at the least), shuffled so that boundaries fall anywhere
    relative to chunk edges."""
    rng = np.random.default_rng(seed)
    parts = [rng.integers(1, 41, 120), rng.integers(100, 301, 16), rng.integers(900, 2600, 3),
             np.array([1, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257])]
    lengths = np.concatenate(parts).astype(np.int32)
    rng.shuffle(lengths)
    return lengths


def _case(lengths, heads, d, dtype, seed, scale, window=None):
    x = workloads.make_custom(lengths, heads, d, dtype, seed=seed, with_dout=True)
    s = int(x.lengths.max())
    _, cu, _ = oracle.pack_sequences(x.lengths, s)
    cu_d = torch.from_numpy(cu).to(DEV)
    first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
    q1 = x.q.to(DEV)[first].contiguous()
    do1 = x.dout.to(DEV)[first].contiguous()
    k, v = x.k.to(DEV), x.v.to(DEV)
    if window is None:
        out, lse = pe.pe_packed_attention_fwd(q1, k, v, cu_d, s, scale,
                                              query_is_first_token=True, need_lse=True)
    else:
        out, lse = pe.pe_packed_attention_fwd_local(q1, k, v, cu_d, s, window[0], window[1],
                                                    scale, query_is_first_token=True,
                                                    need_lse=True)
    return x, s, cu, cu_d, (do1, q1, k, v, out, lse)


def _bwd(args, cu_d, s, scale, window=None, workspace=None):
    do1, q1, k, v, out, lse = args
    if window is None:
        return pe.pe_packed_attention_bwd(do1, q1, k, v, out, lse, cu_d, s, scale,
                                          query_is_first_token=True, workspace=workspace)
    return pe.pe_packed_attention_bwd_local(do1, q1, k, v, out, lse, cu_d, s, window[0],
                                            window[1], scale, query_is_first_token=True,
                                            workspace=workspace)


def _oracle(x, cu, args, scale, window=(-1, -1)):
    do1, q1 = args[0].cpu(), args[1].cpu()
    saved = None
    if q1.dtype == torch.bfloat16:
        ref_out, _ = oracle.attention_fwd(q1, x.k, x.v, cu, int(x.lengths.max()), scale,
                                          first_token=True, window=window)
        saved = torch.from_numpy(ref_out).to(torch.bfloat16)
    return oracle.attention_bwd(q1, x.k, x.v, do1, cu, scale, first_token=True, window=window,
                                out=saved)


def _tag(dtype):
    return "fp32" if dtype == torch.float32 else "bf16"


# Row widths 512 .. 3072 bytes for bf16 and 512 .. 4096 bytes for fp32.
SHAPES = [(torch.bfloat16, 4, 64), (torch.bfloat16, 8, 64), (torch.bfloat16, 12, 64),
          (torch.bfloat16, 16, 64), (torch.bfloat16, 8, 32), (torch.bfloat16, 8, 128),
          (torch.bfloat16, 10, 128), (torch.bfloat16, 24, 64),
          (torch.float32, 2, 64), (torch.float32, 8, 64), (torch.float32, 12, 64),
          (torch.float32, 16, 64), (torch.float32, 14, 64), (torch.float32, 16, 32),
          (torch.float32, 4, 128), (torch.float32, 10, 64)]


@pytest.mark.parametrize("dtype,heads,d", SHAPES)
def test_streaming_first_token_backward_matches_oracle(dtype, heads, d):
    assert pe.pe_attention_kernel(dtype, d, query_is_first_token=True,
                                  backward=True) == "first_token_bwd"
    scale = 1.0 / np.sqrt(d)
    x, s, cu, cu_d, args = _case(_mixed_lengths(7), heads, d, dtype, seed=91, scale=scale)
    dq, dk, dv = _bwd(args, cu_d, s, scale)
    rq, rk, rv = _oracle(x, cu, args, scale)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(got, want, _tag(dtype), f"first-token {name} {heads}x{d}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("right", [0, 5, 64, 700])
def test_streaming_first_token_backward_with_window(dtype, right):
    heads, d = (8, 64) if dtype == torch.bfloat16 else (4, 64)
    window = (3, right)
    x, s, cu, cu_d, args = _case(_mixed_lengths(11), heads, d, dtype, seed=93, scale=0.125,
                                 window=window)
    dq, dk, dv = _bwd(args, cu_d, s, 0.125, window=window)
    rq, rk, rv = _oracle(x, cu, args, 0.125, window=window)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(got, want, _tag(dtype), f"first-token window right={right} {name}")
    # Keys beyond the window: exactly zero gradients.
    pos = oracle.packed_positions(cu)
    hidden = torch.from_numpy(pos > right)
    assert torch.count_nonzero(dk.cpu()[hidden]) == 0
    assert torch.count_nonzero(dv.cpu()[hidden]) == 0


def test_streaming_first_token_backward_fallback_and_determinism():
    """Bitwise reproducible; a workspace without room for the partial sums
    runs the CUDA-core backward, which agrees within the parity bar."""
    lengths = _mixed_lengths(13)
    heads, d, scale = 16, 64, 0.125
    x, s, cu, cu_d, args = _case(lengths, heads, d, torch.bfloat16, seed=95, scale=scale)
    a = _bwd(args, cu_d, s, scale)
    b = _bwd(args, cu_d, s, scale)
    for ga, gb in zip(a, b):
        assert torch.equal(ga, gb)
    n, b_ = int(cu[-1]), len(lengths)
    r16 = lambda x: (x + 15) // 16 * 16
    # Status word and tile plan, then Delta [H, B] fp32: what the CUDA-core
    # backward needs, without the streaming kernel's partial sums.
    base = 32 + 2 * r16(4 * b_) + r16(4 * heads * b_)
    full = pe.attention_workspace_bytes(torch.bfloat16, b_, n, heads, d, s, True, True)
    assert full > base
    minimal = torch.empty(base, dtype=torch.uint8, device=DEV)
    c = _bwd(args, cu_d, s, scale, workspace=minimal)
    for name, gs, gc in zip(("dq", "dk", "dv"), a, c):
        check_grad(gc, to64(gs), "bf16", f"fallback {name}")


def test_wide_bf16_rows_fall_back_and_match():
    """bf16 rows of 4096 bytes (16 heads of 128) are wider than the streaming
    backward takes: they run the CUDA-core backward, with the same results."""
    scale = 1.0 / np.sqrt(128)
    lengths = _mixed_lengths(17)[:60]
    x, s, cu, cu_d, args = _case(lengths, 16, 128, torch.bfloat16, seed=96, scale=scale)
    dq, dk, dv = _bwd(args, cu_d, s, scale)
    rq, rk, rv = _oracle(x, cu, args, scale)
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(got, want, "bf16", f"16x128 fallback {name}")


def test_streaming_first_token_backward_single_sequence_and_tiny():
    for lengths in ([1], [5000], [1, 1, 1], [64] * 33):
        arr = np.array(lengths, np.int32)
        x, s, cu, cu_d, args = _case(arr, 8, 64, torch.float32, seed=97, scale=0.125)
        dq, dk, dv = _bwd(args, cu_d, s, 0.125)
        rq, rk, rv = _oracle(x, cu, args, 0.125)
        for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            check_grad(got, want, "fp32", f"lengths {lengths[:3]}.. {name}")


@pytest.mark.parametrize("name", ["contrastive_bf16", "graph_fp32"])
def test_streaming_first_token_backward_workload_shapes(name):
    wl = workloads.WORKLOADS[name]
    lengths = workloads.draw_lengths(name, np.random.default_rng(0))
    x, s, cu, cu_d, args = _case(lengths, wl.num_heads, wl.head_dim, wl.torch_dtype, seed=0,
                                 scale=wl.scale)
    dq, dk, dv = _bwd(args, cu_d, s, wl.scale)
    rq, rk, rv = _oracle(x, cu, args, wl.scale)
    for g, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        check_grad(got, want, _tag(wl.torch_dtype), f"{name} first-token {g}")


def test_streaming_first_token_backward_long_documents_sampled():
    """The long-document workload at full size: all of dq, and dk, dv on the
    rows of a sample of sequences (the oracle's cost grows with the rows)."""
    name = "longdoc_bf16"
    wl = workloads.WORKLOADS[name]
    lengths = workloads.draw_lengths(name, np.random.default_rng(0))
    x, s, cu, cu_d, args = _case(lengths, wl.num_heads, wl.head_dim, wl.torch_dtype, seed=0,
                                 scale=wl.scale)
    dq, dk, dv = _bwd(args, cu_d, s, wl.scale)
    rq, rk, rv = _oracle(x, cu, args, wl.scale)
    check_grad(dq, rq, "bf16", "long documents first-token dq")
    rng = np.random.default_rng(1)
    for i in rng.choice(len(lengths), size=min(24, len(lengths)), replace=False):
        a, b = int(cu[i]), int(cu[i + 1])
        check_grad(dk[a:b], rk[a:b], "bf16", f"long documents dk seq {i}")
        check_grad(dv[a:b], rv[a:b], "bf16", f"long documents dv seq {i}")


def test_first_token_backward_status_on_bad_layout():
    """A layout that fails the device check computes nothing and reports it."""
    x, s, cu, cu_d, args = _case(np.array([5, 7, 9], np.int32), 8, 64, torch.bfloat16,
                                 seed=99, scale=0.125)
    bad = cu_d.clone()
    bad[2] = bad[1]  # an empty sequence
    n, b_ = int(cu[-1]), 3
    ws = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, b_, n, 8, 64, s, True, True),
                     dtype=torch.uint8, device=DEV)
    _bwd(args, bad, s, 0.125, workspace=ws)
    assert pe.pe_read_device_status(ws) == 2  # PE_ERR_BAD_LENGTH
