"""Batches of many short sequences on the tensor-core forward (thousands of
single-tile items next to longer sequences): checked against the fp64 oracle
and a closed form, with the device status word."""

import math

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(lengths, heads=3, d=64, seed=51, window=None, dtype=torch.bfloat16):
    x = workloads.make_custom(lengths, heads, d, dtype, seed=seed)
    s = int(max(lengths))
    _, cu, n = oracle.pack_sequences(x.lengths, s)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    cu_d = torch.from_numpy(cu).to(DEV)
    ws = torch.empty(pe.attention_workspace_bytes(dtype, len(lengths), n, heads, d, s),
                     dtype=torch.uint8, device=DEV)
    if window is None:
        out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, 1 / math.sqrt(d), need_lse=True,
                                              workspace=ws)
    else:
        out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, s, window[0], window[1],
                                                    1 / math.sqrt(d), need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    return x, s, cu, out, lse


def test_single_token_sequences_return_their_values():
    """3000 sequences of one token: each row sees only its own key, so the
    output is v exactly and lse = scale * q.k."""
    lengths = [1] * 3000
    x, s, cu, out, lse = _run(lengths)
    assert torch.equal(out.cpu(), x.v)
    want = np.einsum("nhd,nhd->hn", to64(x.q), to64(x.k)) / 8.0
    assert float(np.abs(to64(lse) - want).max()) <= 1e-5


@pytest.mark.parametrize("window", [None, (3, 5), (0, 0), (64, 64)])
@pytest.mark.parametrize("seed", [0, 1])
def test_short_sequence_groups_match_oracle(window, seed):
    """Short sequences of every length up to one tile, with longer ones
    interleaved."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 129, 700)
    lengths[::37] = rng.integers(129, 900, lengths[::37].shape[0])
    x, s, cu, out, lse = _run(lengths.tolist(), seed=52 + seed, window=window)
    w = window or (-1, -1)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, 1 / 8.0, window=w)
    check(out, ref, "bf16", f"groups {window}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3


def test_contrastive_workload_groups_match_oracle():
    x = workloads.make_inputs("contrastive_bf16")
    wl = x.workload
    _, cu, n = oracle.pack_sequences(x.lengths, wl.max_seq_len)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    out, lse = pe.pe_packed_attention_fwd(q, k, v, torch.from_numpy(cu).to(DEV),
                                          wl.max_seq_len, wl.scale, need_lse=True)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, wl.max_seq_len, wl.scale)
    check(out, ref, "bf16", "contrastive")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3


@pytest.mark.parametrize("heads", [1, 2, 3, 4, 5, 7, 12])
def test_multi_head_items_match_oracle(heads):
    """Sequences of at most 128 tokens run two heads per work item (tile t takes
    head h + t), and those of at most 64 tokens four (two per tile, 64 rows
    each); head counts that do not divide leave items with fewer heads (a
    missing head's half repeats a loaded one and is not stored). Lengths sit on
    both sides of 64, the 128-token tile and the 256-token item."""
    rng = np.random.default_rng(60 + heads)
    lengths = np.concatenate([[1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257],
                              rng.integers(1, 129, 120), rng.integers(129, 600, 6)])
    rng.shuffle(lengths)
    x, s, cu, out, lse = _run(lengths.tolist(), heads=heads, seed=61)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, 1 / 8.0)
    check(out, ref, "bf16", f"multi-head items, {heads} heads")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3
