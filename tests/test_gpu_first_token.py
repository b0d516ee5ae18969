"""First-token query mode, streaming form, against the fp64 oracle.

In first-token mode each sequence's single query is its first token (page
"Source code for gigl.nn.packed_attention", function `packed_attention`,
`query_is_first_token`), so the expected output of sequence i is row cu[i] of
the full forward. When a token row (heads x head_dim elements) is a whole
number of 512-byte warp loads and head_dim is 32, 64 or 128, the library cuts
the token range into equal chunks of whole rows and merges the partial states
of sequences that cross chunk edges; these tests put sequence boundaries on,
next to and far from those edges, cover every supported row width, windows,
the fallback without room for partials, determinism, and a token count large
enough that the workspace's chunk grows past its minimum.
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
CHUNK = 64  # shortest token chunk; the workspace's chunk doubles past 16384 chunks


def _mixed_lengths(seed):
    """Short queries, mid-size and long sequences, and lengths at the chunk
    size, shuffled so that boundaries fall anywhere relative to chunk edges."""
    rng = np.random.default_rng(seed)
    parts = [rng.integers(1, 41, 150), rng.integers(100, 301, 20), rng.integers(900, 2600, 4),
             np.array([1, 1, 127, 128, 129, 255, 256, 257, 384])]
    lengths = np.concatenate(parts).astype(np.int32)
    rng.shuffle(lengths)
    return lengths


def _first_token_case(lengths, heads, d, dtype, seed):
    x = workloads.make_custom(lengths, heads, d, dtype, seed=seed)
    _, cu, _ = oracle.pack_sequences(x.lengths, int(x.lengths.max()))
    cu_d = torch.from_numpy(cu).to(DEV)
    first = torch.from_numpy(cu[:-1].astype(np.int64)).to(DEV)
    q1 = x.q.to(DEV)[first].contiguous()
    return x, cu, cu_d, q1, x.k.to(DEV), x.v.to(DEV)


def _oracle_first(x, cu, scale, window=(-1, -1)):
    b, h = len(x.lengths), x.k.shape[1]
    rows = cu[:-1].astype(np.int64).repeat(h)
    heads = np.tile(np.arange(h), b)
    ref, ref_lse = oracle.attention_fwd_rows(x.q, x.k, x.v, cu, scale, False, rows, heads,
                                             window=window)
    return ref.reshape(b, h, -1), ref_lse.reshape(b, h).T


def _tag(dtype):
    return "fp32" if dtype == torch.float32 else "bf16"


def _lse_tol(dtype):
    return 1e-4 if dtype == torch.float32 else 2e-3


# (dtype, heads, head_dim): token rows of 1..8 warp loads of 512 bytes.
SHAPES = [
    (torch.bfloat16, 4, 64),    # 512 B
    (torch.bfloat16, 12, 64),   # 1536 B (contrastive batch)
    (torch.bfloat16, 16, 64),   # 2048 B (long documents)
    (torch.float32, 8, 64),     # 2048 B (graph workload)
    (torch.float32, 2, 64),     # 512 B
    (torch.bfloat16, 10, 128),  # 2560 B
    (torch.bfloat16, 16, 128),  # 4096 B
    (torch.float32, 16, 32),    # 2048 B
    (torch.bfloat16, 8, 32),    # 512 B
    (torch.float32, 6, 128),    # 3072 B
    (torch.float32, 7, 128),    # 3584 B
]


@pytest.mark.parametrize("dtype,heads,d", SHAPES)
def test_streaming_first_token_matches_oracle(dtype, heads, d):
    lengths = _mixed_lengths(60 + heads + d)
    x, cu, cu_d, q1, k, v = _first_token_case(lengths, heads, d, dtype, seed=61)
    scale = float(d) ** -0.5
    s = int(lengths.max())
    out, lse = pe.pe_packed_attention_fwd(q1, k, v, cu_d, s, scale, query_is_first_token=True,
                                          need_lse=True)
    ref, ref_lse = _oracle_first(x, cu, scale)
    check(out, ref, _tag(dtype), f"first-token {dtype} {heads}x{d}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("right", [0, 5, 127, 128, 300])
def test_streaming_first_token_with_window(dtype, right):
    """A window's right bound limits the first query to keys 0..right, so
    sequences that cross chunk edges may see keys in one chunk only."""
    lengths = _mixed_lengths(70 + right)
    heads, d = (8, 64) if dtype == torch.bfloat16 else (4, 64)
    x, cu, cu_d, q1, k, v = _first_token_case(lengths, heads, d, dtype, seed=71)
    out, lse = pe.pe_packed_attention_fwd_local(q1, k, v, cu_d, int(lengths.max()), 64, right,
                                                0.125, query_is_first_token=True, need_lse=True)
    ref, ref_lse = _oracle_first(x, cu, 0.125, window=(64, right))
    check(out, ref, _tag(dtype), f"first-token window right={right}")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= _lse_tol(dtype)


def test_streaming_first_token_fallback_and_determinism():
    """Without room for partial states the call runs one CTA per (sequence,
    head) and agrees with the oracle too; the streaming form is bitwise
    reproducible."""
    lengths = _mixed_lengths(80)
    x, cu, cu_d, q1, k, v = _first_token_case(lengths, 16, 64, torch.bfloat16, seed=81)
    s = int(lengths.max())
    ref, _ = _oracle_first(x, cu, 0.125)
    a, _ = pe.pe_packed_attention_fwd(q1, k, v, cu_d, s, 0.125, query_is_first_token=True)
    b, _ = pe.pe_packed_attention_fwd(q1, k, v, cu_d, s, 0.125, query_is_first_token=True)
    assert torch.equal(a, b)
    small = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, len(lengths), k.shape[0], 16,
                                                     64, s), dtype=torch.uint8, device=DEV)
    c, _ = pe.pe_packed_attention_fwd(q1, k, v, cu_d, s, 0.125, query_is_first_token=True,
                                      workspace=small)
    check(c, ref, "bf16", "first-token single pass")
    check(a, ref, "bf16", "first-token streaming")


def test_streaming_first_token_single_sequence_and_single_chunk():
    """One sequence spanning many chunks, and a batch that fits in one chunk."""
    for lengths in ([5000], [3, 1, 60, 2, 40]):
        x, cu, cu_d, q1, k, v = _first_token_case(np.array(lengths, np.int32), 4, 64,
                                                  torch.float32, seed=91)
        out, lse = pe.pe_packed_attention_fwd(q1, k, v, cu_d, max(lengths), 0.125,
                                              query_is_first_token=True, need_lse=True)
        ref, ref_lse = _oracle_first(x, cu, 0.125)
        check(out, ref, "fp32", f"first-token {lengths[:3]}")
        assert float(np.abs(to64(lse) - ref_lse).max()) <= 1e-4


def test_streaming_first_token_long_documents():
    """The long-document workload (32 documents of 2048..8192 tokens, 16 x 64
    bf16): every document spans several chunks."""
    x = workloads.make_inputs("longdoc_bf16")
    wl = x.workload
    _, cu, _ = oracle.pack_sequences(x.lengths, wl.max_seq_len)
    cu_d = torch.from_numpy(cu).to(DEV)
    first = torch.from_numpy(cu[:-1].astype(np.int64))
    q1 = x.q[first].contiguous().to(DEV)
    out, lse = pe.pe_packed_attention_fwd(q1, x.k.to(DEV), x.v.to(DEV), cu_d, wl.max_seq_len,
                                          wl.scale, query_is_first_token=True, need_lse=True)
    ref, ref_lse = _oracle_first(x, cu, wl.scale)
    check(out, ref, "bf16", "long documents first-token")
    assert float(np.abs(to64(lse) - ref_lse).max()) <= 2e-3


def test_streaming_first_token_beyond_minimum_chunk():
    """1.1 M tokens of 512-byte rows: past 16384 chunks of 64 tokens the
    workspace is sized for 128-token chunks. Inputs are drawn on the device
    from a seeded torch generator; the oracle checks sampled sequences from
    their own slices."""
    rng = np.random.default_rng(95)
    lengths = rng.integers(1, 4000, 560).astype(np.int32)
    n = int(lengths.sum())
    assert n > 16384 * CHUNK
    heads, d = 4, 64
    gen = torch.Generator(device=DEV)
    gen.manual_seed(96)
    k = torch.randn((n, heads, d), generator=gen, device=DEV).to(torch.bfloat16)
    v = torch.randn((n, heads, d), generator=gen, device=DEV).to(torch.bfloat16)
    q1 = torch.randn((len(lengths), heads, d), generator=gen, device=DEV).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cu_d = torch.from_numpy(cu).to(DEV)
    out, lse = pe.pe_packed_attention_fwd(q1, k, v, cu_d, int(lengths.max()), 0.125,
                                          query_is_first_token=True, need_lse=True)
    pick = np.unique(np.concatenate([[0, len(lengths) - 1], rng.integers(0, len(lengths), 30)]))
    for i in pick.tolist():
        a, b = int(cu[i]), int(cu[i + 1])
        qi = torch.zeros((b - a, heads, d), dtype=torch.bfloat16)
        qi[0] = q1[i].cpu()
        sub_cu = np.array([0, b - a], np.int32)
        ref, ref_lse = oracle.attention_fwd_rows(qi, k[a:b].cpu(), v[a:b].cpu(), sub_cu, 0.125,
                                                 False, np.zeros(heads, np.int64),
                                                 np.arange(heads))
        check(out[i], ref, "bf16", f"sequence {i} of {len(lengths)}")
        assert float(np.abs(to64(lse[:, i]) - ref_lse).max()) <= 2e-3
