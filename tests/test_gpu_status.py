"""The device status word of the attention calls.

1. Layout check. A caller may build cu_seqlens itself (from NeMo-style
   row metadata, say) instead of taking it from pe_pack_sequences. Before any
   kernel reads q, k or v through it, the call checks on the device that
   cu[0] = 0, cu[B] = N and 1 <= cu[i+1] - cu[i] <= max_seq_len; a layout that
   fails records PE_ERR_BAD_LENGTH or PE_ERR_INVALID_ARG in the status word
   and the call computes nothing (page "nemo_automodel.components.models.
   common.packing": inconsistent packing metadata fails loudly; page "Source
   code for gigl.nn.packed_attention", packed_attention: every sequence holds
   at least one token). Every malformed layout below keeps its entries inside
   [0, N], so even a broken check could not read past the buffers.
2. Bounded waits. Every pipeline wait of the tensor-core kernels gives up
   after a limit, records PE_ERR_DEVICE_TIMEOUT, drains its copies and MMAs and
   exits. With the limit set to 1 ns the waits run out; the status says so, and
   the next call on the same workspace with the default limit is correct.
"""

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BAD_LENGTH, INVALID_ARG, TIMEOUT = 2, 1, 7

# (cu_seqlens, N, max_seq_len, expected status): every entry within [0, N].
MALFORMED = [
    ([0, 100, 50, 300], 300, 300, BAD_LENGTH),    # not monotone
    ([0, 100, 100, 300], 300, 300, BAD_LENGTH),   # an empty sequence
    ([0, 100, 300], 300, 150, BAD_LENGTH),        # a length above max_seq_len
    ([0, 100, 200], 300, 300, INVALID_ARG),       # cu[B] < N
    ([10, 100, 300], 300, 300, INVALID_ARG),      # cu[0] != 0
]

# (dtype, head_dim, first_token): the tensor-core forward, the FFMA forward,
# the streaming first-token kernel and its per-(sequence, head) fallback.
# (4 heads of 32 bf16 elements are 256-byte token rows, which the streaming
# kernel does not take.)
FORWARD_PATHS = [(torch.bfloat16, 64, False), (torch.float32, 64, False),
                 (torch.bfloat16, 64, True), (torch.bfloat16, 32, True)]


def _inputs(n, b, h, d, dtype, first_token, seed=3):
    g = torch.Generator().manual_seed(seed)
    k, v = (torch.randn(n, h, d, generator=g).to(dtype).to(DEV) for _ in range(2))
    q = torch.randn(b if first_token else n, h, d, generator=g).to(dtype).to(DEV)
    return q, k, v


def _workspace(dtype, b, n, h, d, s, first_token, backward):
    nbytes = pe.attention_workspace_bytes(dtype, b, n, h, d, s, first_token, backward)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("cu_list,n,s,want", MALFORMED)
@pytest.mark.parametrize("dtype,d,first_token", FORWARD_PATHS)
def test_forward_rejects_a_malformed_layout_on_the_device(cu_list, n, s, want, dtype, d,
                                                          first_token):
    b, h = len(cu_list) - 1, 4
    q, k, v = _inputs(n, b, h, d, dtype, first_token)
    cu = torch.tensor(cu_list, dtype=torch.int32, device=DEV)
    ws = _workspace(dtype, b, n, h, d, s, first_token, False)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((h, q.shape[0]), float("nan"), device=DEV)
    pe.pe_packed_attention_fwd(q, k, v, cu, s, 0.125, query_is_first_token=first_token,
                               out=out, lse=lse, workspace=ws)
    assert pe.pe_read_device_status(ws) == want
    # Nothing was computed.
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    # A valid layout (as many sequences) on the same workspace clears the status
    # and computes.
    good = [0, 100, n] if b == 2 else [0, 100, 150, n]
    cu_ok = torch.tensor(good, dtype=torch.int32, device=DEV)
    out2, _ = pe.pe_packed_attention_fwd(q, k, v, cu_ok, 300, 0.125,
                                         query_is_first_token=first_token, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    ref, _ = oracle.attention_fwd(q.cpu(), k.cpu(), v.cpu(), np.array(good, dtype=np.int32), 300,
                                  0.125, first_token=first_token)
    check(out2, ref, "fp32" if dtype == torch.float32 else "bf16", "after a rejected layout")


@pytest.mark.parametrize("cu_list,n,s,want", MALFORMED)
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.float32, 64)])
def test_backward_rejects_a_malformed_layout_on_the_device(cu_list, n, s, want, dtype, d):
    b, h = len(cu_list) - 1, 4
    q, k, v = _inputs(n, b, h, d, dtype, False)
    do = torch.randn_like(q)
    out = torch.randn_like(q)
    lse = torch.zeros(h, n, device=DEV)
    cu = torch.tensor(cu_list, dtype=torch.int32, device=DEV)
    ws = _workspace(dtype, b, n, h, d, s, False, True)
    dq, dk, dv = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu, s, 0.125, workspace=ws)
    assert pe.pe_read_device_status(ws) == want


def test_noalloc_forward_reports_a_malformed_layout():
    n, b, h, d = 300, 3, 4, 64
    q, k, v = _inputs(n, b, h, d, torch.bfloat16, False)
    cu = torch.tensor([0, 100, 50, 300], dtype=torch.int32, device=DEV)
    out = torch.full_like(q, float("nan"))
    pe.pe_packed_attention_fwd_noalloc(q, k, v, cu, 300, 0.125, out=out)
    assert pe.pe_read_noalloc_status() == BAD_LENGTH
    assert torch.isnan(out.float()).all()


def _long_inputs(dtype=torch.bfloat16):
    lengths = [4096, 3001, 2500, 1]
    x = workloads.make_custom(lengths, 4, 64, dtype, seed=12, with_dout=True)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).to(DEV)
    return x, cu, max(lengths)


def test_forward_wait_timeout_is_reported_and_the_next_call_is_correct():
    """With a 1 ns limit the tensor-core forward's waits give up: the status word
    says PE_ERR_DEVICE_TIMEOUT. With the default limit restored, the next call on
    the same workspace clears it and matches a call made before (bitwise: the
    forward is deterministic)."""
    x, cu, s = _long_inputs()
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    n, h, d = k.shape
    ws = _workspace(torch.bfloat16, 4, n, h, d, s, False, False)
    ref, ref_lse = pe.pe_packed_attention_fwd(q, k, v, cu, s, 0.125, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    previous = pe.pe_set_wait_limit_ns(1)
    try:
        pe.pe_packed_attention_fwd(q, k, v, cu, s, 0.125, need_lse=True, workspace=ws)
        assert pe.pe_read_device_status(ws) == TIMEOUT
    finally:
        pe.pe_set_wait_limit_ns(previous)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu, s, 0.125, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_backward_wait_timeout_is_reported_and_the_next_call_is_correct():
    x, cu, s = _long_inputs()
    q, k, v, do = (t.to(DEV) for t in (x.q, x.k, x.v, x.dout))
    n, h, d = k.shape
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu, s, 0.125, need_lse=True)
    ws = _workspace(torch.bfloat16, 4, n, h, d, s, False, True)
    ref = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu, s, 0.125, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    previous = pe.pe_set_wait_limit_ns(1)
    try:
        pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu, s, 0.125, workspace=ws)
        assert pe.pe_read_device_status(ws) == TIMEOUT
    finally:
        pe.pe_set_wait_limit_ns(previous)
    got = pe.pe_packed_attention_bwd(do, q, k, v, out, lse, cu, s, 0.125, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
