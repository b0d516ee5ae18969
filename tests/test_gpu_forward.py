"""Packed attention forward on the GPU against the fp64 oracle.

Small and mid-size workloads compare every output element and every
log-sum-exp; the long-document workload compares sampled (row, head) pairs
that the oracle computes one by one, chosen to cover every sequence, both ends
of every sequence and the rows around 128-row tile boundaries.
"""

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


def _device_inputs(x):
    _, cu, _ = oracle.pack_sequences(x.lengths, int(x.workload.max_seq_len))
    cu_d = torch.from_numpy(cu).to(DEV)
    return cu, cu_d, x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)


def _lse_tol(dtype):
    return 1e-4 if dtype == "fp32" else 2e-3


@pytest.mark.parametrize("name", ["tiny_fp32", "graph_fp32", "contrastive_bf16"])
def test_full_and_first_token_match_oracle(name):
    x = workloads.make_inputs(name)
    wl = x.workload
    cu, cu_d, q, k, v = _device_inputs(x)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, wl.max_seq_len, wl.scale, need_lse=True)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, wl.max_seq_len, wl.scale)
    check(out, ref, wl.dtype, f"{name} out")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(wl.dtype)
    first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
    out1, lse1 = pe.pe_packed_attention_fwd(q[first], k, v, cu_d, wl.max_seq_len, wl.scale,
                                            query_is_first_token=True, need_lse=True)
    assert out1.shape == (len(x.lengths), wl.num_heads, wl.head_dim)
    check(out1, ref[cu[:-1]], wl.dtype, f"{name} first-token out")
    assert float(np.abs(to64(lse1) - ref_lse[:, cu[:-1]]).max()) <= _lse_tol(wl.dtype)


def _sample_rows(lengths, cu, heads, rng, per_seq=24):
    rows = []
    for i, n in enumerate(lengths.tolist()):
        start = int(cu[i])
        cand = {0, n - 1, min(n - 1, 127), min(n - 1, 128), min(n - 1, 255), min(n - 1, 256),
                n // 2, max(0, n - 129)}
        cand.update(rng.integers(0, n, per_seq - len(cand)).tolist())
        rows.extend(start + r for r in sorted(cand))
    rows = np.array(rows, np.int64)
    hs = rng.integers(0, heads, rows.shape[0])
    return rows, hs


def test_longdoc_sampled_rows_match_oracle():
    x = workloads.make_inputs("longdoc_bf16")
    wl = x.workload
    cu, cu_d, q, k, v = _device_inputs(x)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, wl.max_seq_len, wl.scale, need_lse=True)
    rng = np.random.default_rng(1)
    rows, hs = _sample_rows(x.lengths, cu, wl.num_heads, rng)
    ref, ref_lse = oracle.attention_fwd_rows(x.q, x.k, x.v, cu, wl.scale, False, rows, hs)
    got = out[torch.from_numpy(rows).to(DEV), torch.from_numpy(hs).to(DEV)]
    check(got, ref, "bf16", "longdoc sampled rows")
    got_lse = lse[torch.from_numpy(hs).to(DEV), torch.from_numpy(rows).to(DEV)]
    assert float(np.abs(to64(got_lse) - ref_lse).max()) <= 2e-3
    # Properties that hold at any size: finite everywhere, and each output row
    # is a convex combination of its sequence's values (within bf16 rounding).
    assert torch.isfinite(out.float()).all()
    assert float(out.float().abs().max()) <= float(v.float().abs().max()) + 0.05


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.float32, 64), (torch.float32, 8),
                                     (torch.bfloat16, 128), (torch.float32, 24),
                                     (torch.bfloat16, 32)])
def test_ragged_tile_boundaries(dtype, d):
    lengths = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 1, 511, 7]
    x = workloads.make_custom(lengths, 3, d, dtype, seed=5)
    s = max(lengths)
    cu, cu_d, q, k, v = _device_inputs(x)
    scale = 1.0 / math.sqrt(d)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, scale, need_lse=True)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, scale)
    tag = "fp32" if dtype == torch.float32 else "bf16"
    check(out, ref, tag, f"ragged d={d}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(tag)
    if d in (8, 16, 32, 64, 128):
        first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
        out1, _ = pe.pe_packed_attention_fwd(q[first], k, v, cu_d, s, scale,
                                             query_is_first_token=True)
        check(out1, ref[cu[:-1]], tag, f"ragged first-token d={d}")


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 72), (torch.float32, 128),
                                     (torch.float32, 16), (torch.bfloat16, 96)])
@pytest.mark.parametrize("window", [None, (10, 40), (40, 3)])
def test_ffma_half_tile_boundaries(dtype, d, window):
    """The FFMA kernel computes 32 rows of a tile with at most 32 real rows and
    32 keys of a block with at most 32 real keys: tails of 31, 32 and 33 rows
    and keys on each side of those edges, with and without a window."""
    lengths = [31, 32, 33, 95, 96, 97, 160, 161, 4, 40, 225]
    x = workloads.make_custom(lengths, 2, d, dtype, seed=9)
    s = max(lengths)
    cu, cu_d, q, k, v = _device_inputs(x)
    scale = 1.0 / math.sqrt(d)
    if window is None:
        out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, scale, need_lse=True)
    else:
        out, lse = pe.pe_packed_attention_fwd_local(q, k, v, cu_d, s, window[0], window[1], scale,
                                                    need_lse=True)
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, scale, window=window or (-1, -1))
    tag = "fp32" if dtype == torch.float32 else "bf16"
    check(out, ref, tag, f"half tiles d={d} window={window}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(tag)


def test_length_one_sequences_output_their_value():
    x = workloads.make_custom([1] * 300, 4, 64, torch.bfloat16, seed=6)
    cu, cu_d, q, k, v = _device_inputs(x)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, 1, 0.125, need_lse=True)
    assert torch.equal(out, v)
    want = 0.125 * (x.q.double() * x.k.double()).sum(-1).T.numpy()
    assert float(np.abs(to64(lse) - want).max()) <= 1e-5


def test_single_long_sequence_and_scale_choice():
    x = workloads.make_custom([3000], 2, 64, torch.bfloat16, seed=7)
    cu, cu_d, q, k, v = _device_inputs(x)
    for scale in (0.05, 0.125, 0.4):
        out, _ = pe.pe_packed_attention_fwd(q, k, v, cu_d, 3000, scale)
        ref, _ = oracle.attention_fwd(x.q, x.k, x.v, cu, 3000, scale)
        check(out, ref, "bf16", f"single sequence scale={scale}")


def test_cross_sequence_isolation_and_determinism():
    x = workloads.make_custom([200, 37, 129, 1, 700], 4, 64, torch.bfloat16, seed=8)
    cu, cu_d, q, k, v = _device_inputs(x)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, 700, 0.125, need_lse=True)
    out2, lse2 = pe.pe_packed_attention_fwd(q, k, v, cu_d, 700, 0.125, need_lse=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    j0, j1 = int(cu[1]), int(cu[2])
    k2, v2 = k.clone(), v.clone()
    k2[j0:j1] = torch.randn_like(k2[j0:j1]) * 3
    v2[j0:j1] = torch.randn_like(v2[j0:j1]) * 3
    out3, lse3 = pe.pe_packed_attention_fwd(q, k2, v2, cu_d, 700, 0.125, need_lse=True)
    keep = torch.ones(out.shape[0], dtype=torch.bool, device=DEV)
    keep[j0:j1] = False
    assert torch.equal(out3[keep], out[keep])
    assert torch.equal(lse3[:, keep], lse[:, keep])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_no_reads_or_writes_outside_the_buffers(dtype):
    """Inputs and output sit between NaN guard rows: the guards must stay NaN
    and must not leak into the result."""
    lengths = [130, 5, 64, 257]
    x = workloads.make_custom(lengths, 2, 64, dtype, seed=9)
    cu, cu_d, _, _, _ = _device_inputs(x)
    n, g = int(sum(lengths)), 256

    def guarded(t):
        buf = torch.full((n + 2 * g,) + tuple(t.shape[1:]), float("nan"), dtype=dtype, device=DEV)
        buf[g:g + n] = t.to(DEV)
        return buf, buf[g:g + n]

    qb, q = guarded(x.q)
    kb, k = guarded(x.k)
    vb, v = guarded(x.v)
    ob, o = guarded(torch.zeros_like(x.q))
    pe.pe_packed_attention_fwd(q, k, v, cu_d, 257, 0.125, out=o)
    torch.cuda.synchronize()
    assert torch.isnan(ob[:g].float()).all() and torch.isnan(ob[g + n:].float()).all()
    ref, _ = oracle.attention_fwd(x.q, x.k, x.v, cu, 257, 0.125)
    check(o, ref, "fp32" if dtype == torch.float32 else "bf16", "guarded")


def test_empty_batch_is_a_no_op():
    cu_d = torch.zeros(1, dtype=torch.int32, device=DEV)
    e = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    out, _ = pe.pe_packed_attention_fwd(e, e, e, cu_d, 4, 0.125)
    assert out.shape == (0, 2, 64)


def test_unsupported_arguments_raise():
    x = workloads.make_custom([4, 5], 2, 64, torch.bfloat16)
    _, cu_d, q, k, v = _device_inputs(x)
    with pytest.raises(pe.PackedAttentionError) as e:
        pe.pe_packed_attention_fwd(q, k, v, cu_d, 5, -1.0)
    assert e.value.status == 1
    with pytest.raises(pe.PackedAttentionError) as e:
        pe.pe_packed_attention_fwd(q[:, :, :12].contiguous(), k[:, :, :12].contiguous(),
                                   v[:, :, :12].contiguous(), cu_d, 5, 0.3)
    assert e.value.status == 4


def test_bf16_d64_runs_on_tensor_cores_and_reports_clean_status():
    assert pe.pe_attention_kernel(torch.bfloat16, 64) == "tcgen05_bf16_d64"
    assert pe.pe_attention_kernel(torch.float32, 64) == "tcgen05_f32_d64"
    assert pe.pe_attention_kernel(torch.float32, 32) == "simt_ffma"
    assert pe.pe_attention_kernel(torch.bfloat16, 64, query_is_first_token=True) == \
        "first_token_gemv"
    # Lengths chosen so work items hit every case of the 256-row query pair:
    # second tile empty, second tile partial, both full, and a single row.
    lengths = [128, 129, 256, 257, 384, 385, 512, 1, 100, 640, 1000]
    x = workloads.make_custom(lengths, 5, 64, torch.bfloat16, seed=31)
    s = max(lengths)
    cu, cu_d, q, k, v = _device_inputs(x)
    ws = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, len(lengths), q.shape[0], 5, 64,
                                                  s), dtype=torch.uint8, device=DEV)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, 0.125, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, 0.125)
    check(out, ref, "bf16", "tensor-core pairs")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3


def test_many_work_items_per_cta():
    """More work items than CTAs, so each persistent CTA runs many items and
    the K/V ring and barriers wrap around many times."""
    rng = np.random.default_rng(32)
    lengths = rng.integers(1, 700, 400).astype(np.int32)
    x = workloads.make_custom(lengths, 8, 64, torch.bfloat16, seed=33)
    s = int(lengths.max())
    cu, cu_d, q, k, v = _device_inputs(x)
    out, _ = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, 0.125)
    ref, _ = oracle.attention_fwd(x.q, x.k, x.v, cu, s, 0.125)
    check(out, ref, "bf16", "many items")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_first_token_split_over_key_chunks(dtype):
    """Sequences longer than one 1024-key chunk are split across CTAs and the
    chunk partials merged; lengths straddle the chunk edges, and max_seq_len
    leaves whole chunks past the end of most sequences."""
    lengths = [1, 1023, 1024, 1025, 3000, 2048, 4100, 4500, 3900, 4999]  # mean > 2 chunks
    x = workloads.make_custom(lengths, 3, 64, dtype, seed=34)
    s = 5000
    cu, cu_d, q, k, v = _device_inputs(x)
    first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
    out, lse = pe.pe_packed_attention_fwd(q[first].contiguous(), k, v, cu_d, s, 0.125,
                                          query_is_first_token=True, need_lse=True)
    rows = cu[:-1].astype(np.int64).repeat(3)
    heads = np.tile(np.arange(3), len(lengths))
    ref, ref_lse = oracle.attention_fwd_rows(x.q, x.k, x.v, cu, 0.125, False, rows, heads)
    tag = "fp32" if dtype == torch.float32 else "bf16"
    got = out[torch.arange(len(lengths)).repeat_interleave(3), torch.from_numpy(heads).to(DEV)]
    check(got, ref, tag, "first-token split")
    got_lse = lse[torch.from_numpy(heads).to(DEV), torch.arange(len(lengths)).repeat_interleave(3).to(DEV)]
    assert float(np.abs(to64(got_lse) - ref_lse).max()) <= _lse_tol(tag)
    # With only the base workspace (no room for chunk partials) the call runs
    # one CTA per (sequence, head) and gives the same answer.
    small = torch.empty(pe.attention_workspace_bytes(dtype, len(lengths), q.shape[0], 3, 64, s),
                        dtype=torch.uint8, device=DEV)
    out2, _ = pe.pe_packed_attention_fwd(q[first].contiguous(), k, v, cu_d, s, 0.125,
                                         query_is_first_token=True, workspace=small)
    check(out2[torch.arange(len(lengths)).repeat_interleave(3), torch.from_numpy(heads).to(DEV)],
          ref, tag, "first-token single pass")


@pytest.mark.parametrize("heads", [4, 5, 6])
def test_odd_block_tails_share_items_across_heads(heads):
    """A sequence of an odd number of 128-row blocks (above 128 tokens) ends in
    one query tile per head; the tensor-core forward runs those last tiles of
    two heads in one work item, each against its own head's keys (the last
    head alone when the head count is odd). Lengths put the tail at every
    offset in its block, next to even-block sequences."""
    lengths = [257, 300, 383, 384, 640, 641, 700, 896, 1100, 1152, 129, 256, 512, 1000, 2000]
    x = workloads.make_custom(lengths, heads, 64, torch.bfloat16, seed=37)
    s = max(lengths)
    cu, cu_d, q, k, v = _device_inputs(x)
    ws = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, len(lengths), q.shape[0], heads,
                                                  64, s), dtype=torch.uint8, device=DEV)
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu_d, s, 0.125, need_lse=True, workspace=ws)
    assert pe.pe_read_device_status(ws) == 0
    ref, ref_lse = oracle.attention_fwd(x.q, x.k, x.v, cu, s, 0.125)
    check(out, ref, "bf16", f"odd-block tails, {heads} heads")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3
