"""Pins the fp64 oracle to facts fixed outside the oracle itself (CPU only).

Each test checks the oracle against one of:
  * values printed on the pages (tests/golden, each with its citation);
  * closed forms of softmax attention;
  * library routines on special cases (torch SDPA and autograd in fp64,
    scipy's softmax, numpy boolean indexing);
  * finite differences of the oracle's own forward (for the backward);
  * invariants of the definition.
A dropped term, a wrong sign or index, or a transposed operand anywhere in the
oracle makes at least one of these fail.
"""

import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
from oracle import OracleError
from padding_free_packed_gb300 import workloads


def _random_case(seed, b_max=7, s_max=13, h=3, d=8):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, b_max + 1))
    s = int(rng.integers(1, s_max + 1))
    lengths = rng.integers(1, s + 1, b).astype(np.int32)
    n = int(lengths.sum())
    q = rng.standard_normal((n, h, d))
    k = rng.standard_normal((n, h, d))
    v = rng.standard_normal((n, h, d))
    return lengths, s, q, k, v


def _padded(x, lengths, s):
    """Test-side padding with numpy boolean indexing: [B, S, ...], zeros at pads."""
    b = len(lengths)
    mask = np.arange(s)[None, :] < np.asarray(lengths)[:, None]
    grid = np.zeros((b, s) + x.shape[1:], dtype=x.dtype)
    grid[mask] = x
    return grid, mask


# --------------------------------------------------------------------------- pack

def test_pack_worked_example(golden):
    g = golden("pack_worked_example.txt")
    flat, cu, n = oracle.pack_sequences(g["lengths"], g["max_seq_len"][0])
    assert flat.tolist() == g["flat_index"]
    assert cu.tolist() == g["cu_seqlens"]
    assert n == g["num_tokens"][0]


def test_pack_cu_seqlens_example(golden):
    g = golden("pack_cu_seqlens_example.txt")
    flat, cu, n = oracle.pack_sequences(g["lengths"], g["max_seq_len"][0])
    assert cu.tolist() == g["cu_seqlens"]
    assert n == g["num_tokens"][0]
    assert cu.dtype == np.int32


@pytest.mark.parametrize("seed", range(12))
def test_pack_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    b = int(rng.integers(1, 60))
    s = int(rng.integers(1, 50))
    lengths = rng.integers(1, s + 1, b).astype(np.int32)
    flat, cu, n = oracle.pack_sequences(lengths, s)
    assert n == int(lengths.sum())
    assert cu.tolist() == [0] + np.cumsum(lengths).tolist()
    assert np.all(np.diff(flat) > 0)
    seq = flat // s
    assert np.all(np.diff(seq) >= 0)
    assert np.bincount(seq, minlength=b).tolist() == lengths.tolist()
    assert np.all(flat % s < lengths[seq])
    # flat_index lists exactly the real cells of the padded grid (numpy's own
    # boolean-mask order is row-major, i.e. i ascending then j ascending).
    mask = np.arange(s)[None, :] < lengths[:, None]
    assert flat.tolist() == np.flatnonzero(mask.reshape(-1)).tolist()


def test_pack_edge_cases():
    flat, cu, n = oracle.pack_sequences(np.zeros(0, np.int32), 4)
    assert n == 0 and cu.tolist() == [0] and flat.size == 0
    flat, cu, n = oracle.pack_sequences([1] * 5, 4)
    assert flat.tolist() == [0, 4, 8, 12, 16]
    flat, cu, n = oracle.pack_sequences([4, 4], 4)
    assert flat.tolist() == list(range(8))
    with pytest.raises(OracleError) as e:
        oracle.pack_sequences([3, 0, 2], 4)
    assert e.value.code == 2
    with pytest.raises(OracleError) as e:
        oracle.pack_sequences([3, 5], 4)
    assert e.value.code == 2
    with pytest.raises(OracleError) as e:
        oracle.pack_sequences([-1], 4)
    assert e.value.code == 2
    big = 1 << 30
    _, cu, n = oracle.pack_sequences([big, big - 1], big, want_index=False)
    assert n == (1 << 31) - 1
    with pytest.raises(OracleError) as e:
        oracle.pack_sequences([big, big], big, want_index=False)
    assert e.value.code == 3


@pytest.mark.parametrize("seed", range(4))
def test_gather_scatter_round_trip(seed):
    rng = np.random.default_rng(200 + seed)
    b, s = int(rng.integers(1, 9)), int(rng.integers(1, 17))
    lengths = rng.integers(1, s + 1, b).astype(np.int32)
    grid = rng.standard_normal((b, s, 3, 5)).astype(np.float32)
    flat, cu, n = oracle.pack_sequences(lengths, s)
    packed = oracle.gather_rows(grid.reshape(b * s, 3, 5), flat)
    mask = np.arange(s)[None, :] < lengths[:, None]
    np.testing.assert_array_equal(packed, grid[mask])
    back = oracle.scatter_rows(packed, cu, s)
    np.testing.assert_array_equal(back[mask], grid[mask])
    assert np.all(back[~mask] == 0)


# --------------------------------------------------------------------------- forward

def test_forward_shapes_worked_example(golden):
    g = golden("pack_worked_example.txt")
    _, cu, n = oracle.pack_sequences(g["lengths"], g["max_seq_len"][0])
    h, d = g["heads"][0], g["head_dim"][0]
    rng = np.random.default_rng(0)
    x = rng.standard_normal((n, h, d))
    o, lse = oracle.attention_fwd(x, x, x, cu, g["max_seq_len"][0], 1 / math.sqrt(d))
    assert list(o.shape) == g["full_output_shape"]
    assert lse.shape == (h, n)
    o1, _ = oracle.attention_fwd(x[cu[:-1]], x, x, cu, g["max_seq_len"][0], 1 / math.sqrt(d),
                                 first_token=True)
    assert list(o1.shape) == g["first_token_output_shape"]


@pytest.mark.parametrize("seed", range(6))
def test_forward_matches_sdpa_on_padded_grid(seed):
    """The reference path itself: SDPA with padded keys masked, on a padded grid."""
    lengths, s, q, k, v = _random_case(seed)
    _, cu, n = oracle.pack_sequences(lengths, s)
    scale = 0.37 + 0.1 * seed
    o, lse = oracle.attention_fwd(q, k, v, cu, s, scale)
    qg, mask = _padded(q, lengths, s)
    kg, _ = _padded(k, lengths, s)
    vg, _ = _padded(v, lengths, s)
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (qg, kg, vg))
    attn_mask = torch.from_numpy(mask)[:, None, None, :]
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=attn_mask, scale=scale)
    ref = ref.transpose(1, 2).numpy()[mask]
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    scores = torch.einsum("bhqd,bhkd->bhqk", tq, tk) * scale
    scores = scores.masked_fill(~attn_mask, float("-inf"))
    ref_lse = torch.logsumexp(scores, dim=-1).transpose(1, 2).numpy()[mask]  # [N, H]
    np.testing.assert_allclose(lse.T, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_first_token_equals_rows_of_full_output(seed):
    lengths, s, q, k, v = _random_case(10 + seed)
    _, cu, _ = oracle.pack_sequences(lengths, s)
    o, lse = oracle.attention_fwd(q, k, v, cu, s, 0.5)
    first = cu[:-1].astype(np.int64)
    o1, lse1 = oracle.attention_fwd(q[first], k, v, cu, s, 0.5, first_token=True)
    np.testing.assert_array_equal(o1, o[first])
    np.testing.assert_array_equal(lse1, lse[:, first])


def test_closed_forms():
    rng = np.random.default_rng(7)
    h, d, scale = 2, 8, 0.3
    # A length-1 sequence outputs its own v; its lse is scale * q.k.
    lengths = np.array([1, 4, 1], np.int32)
    _, cu, n = oracle.pack_sequences(lengths, 4)
    q, k, v = (rng.standard_normal((n, h, d)) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, cu, 4, scale)
    for t in (0, 5):
        np.testing.assert_allclose(o[t], v[t], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[:, t], scale * np.sum(q[t] * k[t], axis=-1), atol=1e-14)
    # q = 0 (or scale = 0) gives the mean of the sequence's values and lse = log L.
    for zero_q in (True, False):
        qq = np.zeros_like(q) if zero_q else q
        o, lse = oracle.attention_fwd(qq, k, v, cu, 4, 0.0 if not zero_q else scale)
        for i in range(len(lengths)):
            rows = slice(cu[i], cu[i + 1])
            np.testing.assert_allclose(o[rows], np.broadcast_to(v[rows].mean(0), o[rows].shape),
                                       atol=1e-14)
            np.testing.assert_allclose(lse[:, rows], math.log(lengths[i]), atol=1e-14)
    # Constant values give that constant back.
    const = rng.standard_normal((1, h, d))
    o, _ = oracle.attention_fwd(q, k, np.broadcast_to(const, v.shape), cu, 4, scale)
    np.testing.assert_allclose(o, np.broadcast_to(const, o.shape), atol=1e-14)


def test_one_full_sequence_is_textbook_attention():
    """B = 1, L = S: dense softmax(scale Q K^T) V, computed with scipy's softmax."""
    rng = np.random.default_rng(8)
    s, h, d, scale = 17, 2, 8, 0.41
    q, k, v = (rng.standard_normal((s, h, d)) for _ in range(3))
    _, cu, _ = oracle.pack_sequences([s], s)
    o, _ = oracle.attention_fwd(q, k, v, cu, s, scale)
    for hh in range(h):
        w = scipy.special.softmax(scale * q[:, hh] @ k[:, hh].T, axis=1)
        np.testing.assert_allclose(o[:, hh], w @ v[:, hh], atol=1e-13)


def test_block_diagonal_brute_force_on_tiny_workload():
    """Full token-by-token score matrix, keeping pairs in the same grid row."""
    x = workloads.make_inputs("tiny_fp32")
    s = x.workload.max_seq_len
    flat, cu, n = oracle.pack_sequences(x.lengths, s)
    q, k, v = (t.double().numpy() for t in (x.q, x.k, x.v))
    o, _ = oracle.attention_fwd(q, k, v, cu, s, x.workload.scale)
    same = (flat[:, None] // s) == (flat[None, :] // s)
    for hh in range(x.workload.num_heads):
        scores = x.workload.scale * q[:, hh] @ k[:, hh].T
        scores = np.where(same, scores, -np.inf)
        w = scipy.special.softmax(scores, axis=1)
        np.testing.assert_allclose(o[:, hh], w @ v[:, hh], atol=1e-13)


@pytest.mark.parametrize("first_token", [False, True])
def test_sampled_rows_match_full_forward(first_token):
    lengths, s, q, k, v = _random_case(31, b_max=9, s_max=40, h=4, d=16)
    _, cu, n = oracle.pack_sequences(lengths, s)
    if first_token:
        q = q[cu[:-1].astype(np.int64)]
    o, lse = oracle.attention_fwd(q, k, v, cu, s, 0.25, first_token=first_token)
    rng = np.random.default_rng(3)
    rows = rng.integers(0, q.shape[0], 50)
    heads = rng.integers(0, 4, 50)
    o_r, lse_r = oracle.attention_fwd_rows(q, k, v, cu, 0.25, first_token, rows, heads)
    np.testing.assert_allclose(o_r, o[rows, heads], atol=1e-14)
    np.testing.assert_allclose(lse_r, lse[heads, rows], atol=1e-14)


def test_cross_sequence_isolation():
    lengths, s, q, k, v = _random_case(41, b_max=6)
    if len(lengths) < 2:
        lengths = np.array([3, 4], np.int32)
        s = 4
        rng = np.random.default_rng(0)
        q, k, v = (rng.standard_normal((7, 3, 8)) for _ in range(3))
    _, cu, _ = oracle.pack_sequences(lengths, s)
    o, lse = oracle.attention_fwd(q, k, v, cu, s, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[cu[1]:cu[2]] += 3.0
    v2[cu[1]:cu[2]] -= 5.0
    o2, lse2 = oracle.attention_fwd(q, k2, v2, cu, s, 0.5)
    keep = np.ones(q.shape[0], bool)
    keep[cu[1]:cu[2]] = False
    np.testing.assert_array_equal(o2[keep], o[keep])
    np.testing.assert_array_equal(lse2[:, keep], lse[:, keep])
    assert not np.array_equal(o2[~keep], o[~keep])


# --------------------------------------------------------------------------- backward

def _loss(q, k, v, dout, cu, s, scale, first_token):
    o, _ = oracle.attention_fwd(q, k, v, cu, s, scale, first_token=first_token, threads=1)
    return float(np.sum(o * dout))


@pytest.mark.parametrize("first_token", [False, True])
def test_backward_matches_finite_differences(first_token):
    rng = np.random.default_rng(5)
    lengths = np.array([3, 1, 4], np.int32)
    s, h, d, scale = 4, 2, 4, 0.6
    _, cu, n = oracle.pack_sequences(lengths, s)
    nq = len(lengths) if first_token else n
    q = rng.standard_normal((nq, h, d))
    k, v = rng.standard_normal((n, h, d)), rng.standard_normal((n, h, d))
    dout = rng.standard_normal((nq, h, d))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, cu, scale, first_token=first_token)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = _loss(args["q"], args["k"], args["v"], dout, cu, s, scale, first_token)
            args[name] = xm
            fm = _loss(args["q"], args["k"], args["v"], dout, cu, s, scale, first_token)
            fd[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, fd, rtol=0, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("seed", range(3))
def test_backward_matches_torch_autograd_on_padded_grid(seed):
    lengths, s, q, k, v = _random_case(50 + seed)
    _, cu, n = oracle.pack_sequences(lengths, s)
    rng = np.random.default_rng(60 + seed)
    dout = rng.standard_normal(q.shape)
    scale = 0.45
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, cu, scale)
    grids = [_padded(x, lengths, s)[0] for x in (q, k, v, dout)]
    mask = _padded(q, lengths, s)[1]
    tq, tk, tv = (torch.from_numpy(g).transpose(1, 2).requires_grad_(True) for g in grids[:3])
    attn_mask = torch.from_numpy(mask)[:, None, None, :]
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=attn_mask, scale=scale)
    out.backward(torch.from_numpy(grids[3]).transpose(1, 2))
    for g, t in ((dq, tq), (dk, tk), (dv, tv)):
        ref = t.grad.transpose(1, 2).numpy()[mask]
        np.testing.assert_allclose(g, ref, rtol=0, atol=1e-12)


def test_backward_invariants():
    """Rows of dS sum to zero, so dK sums to zero per (sequence, head); rows of P
    sum to one, so dV sums to the sum of dO per (sequence, head)."""
    lengths, s, q, k, v = _random_case(70, b_max=8, s_max=20)
    _, cu, _ = oracle.pack_sequences(lengths, s)
    dout = np.random.default_rng(71).standard_normal(q.shape)
    _, dk, dv = oracle.attention_bwd(q, k, v, dout, cu, 0.35)
    for i in range(len(lengths)):
        rows = slice(cu[i], cu[i + 1])
        np.testing.assert_allclose(dk[rows].sum(0), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv[rows].sum(0), dout[rows].sum(0), atol=1e-12)


@pytest.mark.parametrize("first_token", [False, True])
def test_backward_with_saved_output(first_token):
    """The backward op takes the forward's saved output, and Delta = dO . O is
    formed from it. Given the exact output, the gradients are the exact ones;
    a perturbation E of the saved output moves only the Delta term, by brute
    force on a tiny case: dq_r -= scale (dO_r . E_r) sum_j P_rj k_j,
    dk_j -= scale sum_r P_rj (dO_r . E_r) q_r, dv unchanged."""
    lengths, s, q, k, v = _random_case(72, b_max=5, s_max=9)
    _, cu, _ = oracle.pack_sequences(lengths, s)
    rng = np.random.default_rng(73)
    first = cu[:-1].astype(np.int64)
    qq = q[first] if first_token else q
    dout = rng.standard_normal(qq.shape)
    scale = 0.4
    out, _ = oracle.attention_fwd(q, k, v, cu, s, scale)
    out = out[first] if first_token else out
    exact = oracle.attention_bwd(qq, k, v, dout, cu, scale, first_token=first_token)
    same = oracle.attention_bwd(qq, k, v, dout, cu, scale, first_token=first_token, out=out)
    for a, b in zip(exact, same):
        np.testing.assert_allclose(b, a, atol=1e-12)
    pert = rng.standard_normal(out.shape) * 1e-2
    moved = oracle.attention_bwd(qq, k, v, dout, cu, scale, first_token=first_token,
                                 out=out + pert)
    want_dq, want_dk = exact[0].copy(), exact[1].copy()
    for i in range(len(lengths)):
        a, b = int(cu[i]), int(cu[i + 1])
        rows = [i] if first_token else list(range(a, b))
        for r in rows:
            for h in range(k.shape[1]):
                logits = scale * np.array([qq[r, h] @ k[j, h] for j in range(a, b)])
                p = np.exp(logits - logits.max())
                p /= p.sum()
                e = float(dout[r, h] @ pert[r, h])
                want_dq[r, h] -= scale * e * sum(p[t] * k[a + t, h] for t in range(b - a))
                for t in range(b - a):
                    want_dk[a + t, h] -= scale * p[t] * e * qq[r, h]
    np.testing.assert_allclose(moved[0], want_dq, atol=1e-12)
    np.testing.assert_allclose(moved[1], want_dk, atol=1e-12)
    np.testing.assert_allclose(moved[2], exact[2], atol=1e-12)


# --------------------------------------------------------------------------- local attention
# Reading of the packed-encoders README's "local-64" mode and FlashAttention's
# sliding-window pruning: the key at position j is visible from the query at
# position r of the same sequence iff r - left <= j <= r + right (negative =
# unbounded); a first-token query sits at position 0.

WINDOWS = [(0, 0), (1, 1), (2, 0), (0, 3), (3, 5), (-1, 2), (4, -1), (-1, -1), (100, 100)]


def _band_mask_grid(lengths, s, window, first_token):
    """[B, Sq, S] boolean from positions on the padded grid: key j real and inside the window."""
    wl, wr = window
    rq = np.zeros((1, 1)) if first_token else np.arange(s)[:, None]
    j = np.arange(s)[None, :]
    band = np.ones((rq.shape[0], s), dtype=bool)
    if wl >= 0:
        band &= j >= rq - wl
    if wr >= 0:
        band &= j <= rq + wr
    real = np.arange(s)[None, None, :] < np.asarray(lengths)[:, None, None]
    return band[None, :, :] & real


@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("first_token", [False, True])
def test_local_forward_matches_sdpa_band_mask(window, first_token):
    for seed in range(3):
        lengths, s, q, k, v = _random_case(80 + seed, s_max=17)
        _, cu, n = oracle.pack_sequences(lengths, s)
        scale = 0.41
        first = cu[:-1].astype(np.int64)
        qq = q[first] if first_token else q
        o, lse = oracle.attention_fwd(qq, k, v, cu, s, scale, first_token=first_token,
                                      window=window)
        qg, mask = _padded(q, lengths, s)
        kg, _ = _padded(k, lengths, s)
        vg, _ = _padded(v, lengths, s)
        if first_token:
            qg = qg[:, :1]
        tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (qg, kg, vg))
        band = torch.from_numpy(_band_mask_grid(lengths, s, window, first_token))[:, None]
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=band, scale=scale)
        ref = ref.transpose(1, 2).numpy()
        ref = ref[:, 0] if first_token else ref[mask]
        scores = (torch.einsum("bhqd,bhkd->bhqk", tq, tk) * scale).masked_fill(~band, float("-inf"))
        ref_lse = torch.logsumexp(scores, dim=-1).transpose(1, 2).numpy()
        ref_lse = ref_lse[:, 0] if first_token else ref_lse[mask]
        # Rows of padded queries may be fully masked in SDPA (NaN); only real rows are compared.
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.T, ref_lse, rtol=0, atol=1e-12)


def test_local_window_zero_is_the_value_row():
    """Window (0, 0): each query sees only its own key, so o_r = v_r and
    lse_r = scale * q_r . k_r exactly (a softmax over one element)."""
    lengths, s, q, k, v = _random_case(90, s_max=9)
    _, cu, _ = oracle.pack_sequences(lengths, s)
    o, lse = oracle.attention_fwd(q, k, v, cu, s, 0.7, window=(0, 0))
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse.T, 0.7 * np.einsum("nhd,nhd->nh", q, k), rtol=0, atol=1e-13)


def test_local_window_counts_keys():
    """With v = 1 in one coordinate and q = 0 (uniform weights), the output is
    1 and lse = log(number of visible keys) = log(min(r+R, L-1) - max(r-L', 0) + 1)."""
    lengths = np.array([9, 1, 5], np.int32)
    s, h, d = 9, 1, 2
    _, cu, n = oracle.pack_sequences(lengths, s)
    q = np.zeros((n, h, d))
    k = np.random.default_rng(91).standard_normal((n, h, d))
    v = np.zeros((n, h, d))
    v[..., 0] = 1.0
    for wl, wr in [(2, 1), (0, 4), (3, 0)]:
        o, lse = oracle.attention_fwd(q, k, v, cu, s, 1.0, window=(wl, wr))
        np.testing.assert_allclose(o[..., 0], 1.0, rtol=0, atol=1e-15)
        for i, length in enumerate(lengths):
            for r in range(length):
                count = min(r + wr, length - 1) - max(r - wl, 0) + 1
                assert abs(lse[0, cu[i] + r] - math.log(count)) < 1e-14


@pytest.mark.parametrize("window", [(1, 2), (0, 0), (3, -1)])
def test_local_sampled_rows_match_full_forward(window):
    lengths, s, q, k, v = _random_case(93, s_max=15)
    _, cu, n = oracle.pack_sequences(lengths, s)
    o, lse = oracle.attention_fwd(q, k, v, cu, s, 0.5, window=window)
    rng = np.random.default_rng(94)
    rows = rng.integers(0, n, 20)
    heads = rng.integers(0, q.shape[1], 20)
    o2, lse2 = oracle.attention_fwd_rows(q, k, v, cu, 0.5, False, rows, heads, window=window)
    np.testing.assert_allclose(o2, o[rows, heads], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse[heads, rows], rtol=0, atol=1e-13)


@pytest.mark.parametrize("window", [(1, 1), (2, 0), (0, 3), (-1, 1)])
@pytest.mark.parametrize("first_token", [False, True])
def test_local_backward_matches_torch_autograd(window, first_token):
    lengths, s, q, k, v = _random_case(95, s_max=12)
    _, cu, n = oracle.pack_sequences(lengths, s)
    first = cu[:-1].astype(np.int64)
    qq = q[first] if first_token else q
    dout = np.random.default_rng(96).standard_normal(qq.shape)
    scale = 0.55
    dq, dk, dv = oracle.attention_bwd(qq, k, v, dout, cu, scale, first_token=first_token,
                                      window=window)
    qg, mask = _padded(q, lengths, s)
    kg, _ = _padded(k, lengths, s)
    vg, _ = _padded(v, lengths, s)
    if first_token:
        qg = qg[:, :1]
        gg = dout[:, None]
    else:
        gg = _padded(dout, lengths, s)[0]
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2).requires_grad_(True) for x in (qg, kg, vg))
    band = torch.from_numpy(_band_mask_grid(lengths, s, window, first_token))[:, None]
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=band, scale=scale)
    # Padded query rows of the grid carry no gradient: their dO is zero.
    out.backward(torch.from_numpy(np.ascontiguousarray(gg)).transpose(1, 2))
    ref_dq = tq.grad.transpose(1, 2).numpy()
    ref_dq = ref_dq[:, 0] if first_token else ref_dq[mask]
    np.testing.assert_allclose(dq, ref_dq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.transpose(1, 2).numpy()[mask], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.transpose(1, 2).numpy()[mask], rtol=0, atol=1e-12)


def test_local_backward_matches_finite_differences():
    rng = np.random.default_rng(97)
    lengths = np.array([5, 2], np.int32)
    s, h, d, scale, window = 5, 1, 3, 0.8, (1, 2)
    _, cu, n = oracle.pack_sequences(lengths, s)
    q, k, v, dout = (rng.standard_normal((n, h, d)) for _ in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, cu, scale, window=window)
    eps = 1e-6

    def loss(qx, kx, vx):
        o, _ = oracle.attention_fwd(qx, kx, vx, cu, s, scale, threads=1, window=window)
        return float(np.sum(o * dout))

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = {"q": q, "k": k, "v": v}
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args[name] = xp
            fp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = loss(args["q"], args["k"], args["v"])
            fd[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, fd, rtol=0, atol=2e-8, err_msg=name)


# --------------------------------------------------------------------------- packed-row metadata
# Page "nemo_automodel.components.models.common.packing": indexed packing masks
# (document i of a row marked i, 0 = padding) and
# flatten_packed_sequence_metadata (row-local token indices and cumulative
# lengths, -1 padded, to one flat stream).

def test_indexed_mask_worked_example(golden):
    g = golden("indexed_packing_mask_example.txt")
    flat, cu = oracle.pack_document_ids([g["row"]])
    assert flat.tolist() == g["flat_index"] and cu.tolist() == g["cu_seqlens"]
    flat2, cu2 = oracle.flatten_packed_metadata([g["row_token_indices"]], [g["row_cu_seqlens"]],
                                                g["sequence_length"][0])
    assert flat2.tolist() == g["flat_index"] and cu2.tolist() == g["cu_seqlens"]


def _packed_rows(seed, b=6, s=40, max_docs=5, sparse=False):
    """Rows built from random document lengths (numpy only): the id mask, the
    two NeMo-style row-local layouts, and the flat outputs they stand for."""
    rng = np.random.default_rng(seed)
    ids = np.zeros((b, s), np.int32)
    tok = np.full((b, s), -1, np.int64)
    rcu = np.full((b, max_docs + 1), -1, np.int32)
    flat, cu, total = [], [0], 0
    for i in range(b):
        docs = []
        room = s
        for _ in range(int(rng.integers(0, max_docs + 1))):
            if room == 0:
                break
            docs.append(int(rng.integers(1, min(room, 12) + 1)))
            room -= docs[-1]
        n = sum(docs)
        ids[i, :n] = np.repeat(np.arange(1, len(docs) + 1), docs)
        # Row-local positions: the first n positions, or (sparse) n sorted distinct ones.
        pos = np.sort(rng.choice(s, n, replace=False)) if sparse else np.arange(n)
        tok[i, :n] = pos
        rcu[i, :len(docs) + 1] = np.concatenate([[0], np.cumsum(docs)])
        flat.extend((i * s + pos).tolist())
        cu.extend((total + np.cumsum(docs)).tolist())
        total += n
    return ids, tok, rcu, np.array(flat, np.int64), np.array(cu, np.int32)


@pytest.mark.parametrize("seed", range(8))
def test_packed_rows_match_independent_construction(seed):
    ids, tok, rcu, flat, cu = _packed_rows(seed)
    f1, c1 = oracle.pack_document_ids(ids)
    np.testing.assert_array_equal(f1, flat)
    np.testing.assert_array_equal(c1, cu)
    f2, c2 = oracle.flatten_packed_metadata(tok, rcu, ids.shape[1])
    np.testing.assert_array_equal(f2, flat)
    np.testing.assert_array_equal(c2, cu)
    # The row-local token indices need not be the first positions of a row.
    _, tok_s, rcu_s, flat_s, cu_s = _packed_rows(seed, sparse=True)
    f3, c3 = oracle.flatten_packed_metadata(tok_s, rcu_s, ids.shape[1])
    np.testing.assert_array_equal(f3, flat_s)
    np.testing.assert_array_equal(c3, cu_s)


def test_one_document_per_row_is_pack_sequences():
    lengths = np.array([5, 1, 9, 3], np.int32)
    s = 9
    ids = (np.arange(s)[None, :] < lengths[:, None]).astype(np.int32)
    flat, cu = oracle.pack_document_ids(ids)
    flat_p, cu_p, _ = oracle.pack_sequences(lengths, s)
    np.testing.assert_array_equal(flat, flat_p)
    np.testing.assert_array_equal(cu, cu_p)


@pytest.mark.parametrize("row", [
    [1, 1, 3, 0],     # document 2 skipped
    [1, 0, 1, 0],     # a document after padding
    [2, 2, 0, 0],     # numbering does not start at 1
    [1, 2, 1, 0],     # document 1 split in two
    [1, -1, 0, 0],    # negative id
    [0, 1, 1, 0],     # padding before the first document
])
def test_indexed_mask_rejects_malformed_rows(row):
    with pytest.raises(OracleError):
        oracle.pack_document_ids([row])


@pytest.mark.parametrize("tok,rcu", [
    ([0, 1, 2, -1], [1, 3, -1]),      # boundaries do not start at 0
    ([0, 1, 2, -1], [0, 2, 2, 3]),    # an empty document
    ([0, 1, 2, -1], [0, 2, -1, -1]),  # boundaries end before the tokens do
    ([0, 1, 2, -1], [0, 3, 4, -1]),   # boundaries end after them
    ([0, -1, 2, -1], [0, 2, -1, -1]), # token padding not trailing
    ([0, 1, 2, -1], [0, -1, 3, -1]),  # boundary padding not trailing
    ([0, 1, 4, -1], [0, 3, -1, -1]),  # index outside the row
])
def test_flatten_rejects_inconsistent_layouts(tok, rcu):
    with pytest.raises(OracleError):
        oracle.flatten_packed_metadata([tok], [rcu], 4)


def test_empty_rows_and_batch():
    flat, cu = oracle.pack_document_ids(np.zeros((3, 4), np.int32))
    assert flat.size == 0 and cu.tolist() == [0]
    flat, cu = oracle.flatten_packed_metadata(np.full((2, 3), -1), [[0, -1], [0, -1]], 3)
    assert flat.size == 0 and cu.tolist() == [0]


# --------------------------------------------------------------------------- layer tail
# Page "packed-encoders 0.1.0": fused LayerNorm / residual-LayerNorm / RoPE
# (split-half convention) / GeGLU on the flat token buffer, with position ids
# restarting at every sequence.

def test_packed_positions_worked_example(golden):
    g = golden("packed_position_ids_example.txt")
    _, cu, _ = oracle.pack_sequences(g["lengths"], max(g["lengths"]))
    assert cu.tolist() == g["cu_seqlens"]
    assert oracle.packed_positions(cu).tolist() == g["position_ids"]


def test_rope_is_a_complex_rotation_of_split_halves():
    """Pairs (i, i + D/2) as complex numbers x_i + j x_{i+D/2}, multiplied by
    exp(j * pos * theta^(-2i/D))."""
    rng = np.random.default_rng(101)
    n, h, d, theta = 37, 3, 16, 10000.0
    x = rng.standard_normal((n, h, d))
    pos = rng.integers(0, 9000, n)
    got = oracle.rope(x, pos, theta)
    angle = pos[:, None] * theta ** (-np.arange(0, d, 2) / d)            # [n, d/2]
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * angle)[:, None, :]
    np.testing.assert_allclose(got[..., : d // 2], z.real, rtol=0, atol=1e-10)
    np.testing.assert_allclose(got[..., d // 2:], z.imag, rtol=0, atol=1e-10)


def test_rope_invariants():
    rng = np.random.default_rng(102)
    n, h, d = 9, 2, 8
    x = rng.standard_normal((n, h, d))
    # Position 0 is the identity; every pair keeps its norm.
    np.testing.assert_allclose(oracle.rope(x, np.zeros(n, np.int64), 500.0), x, atol=1e-15)
    y = oracle.rope(x, np.arange(n) * 7, 500.0)
    np.testing.assert_allclose(x[..., :4] ** 2 + x[..., 4:] ** 2, y[..., :4] ** 2 + y[..., 4:] ** 2,
                               rtol=1e-12)
    # Scores depend only on the position difference.
    q, k = rng.standard_normal((1, 1, d)), rng.standard_normal((1, 1, d))
    def score(m, p):
        return float(np.sum(oracle.rope(q, [m], 500.0) * oracle.rope(k, [p], 500.0)))
    assert abs(score(11, 4) - score(31, 24)) < 1e-10


@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("with_residual", [True, False])
def test_layernorm_matches_torch(with_bias, with_residual):
    rng = np.random.default_rng(103)
    n, c, eps = 13, 48, 1e-5
    x = rng.standard_normal((n, c)) * 3 + 1
    r = rng.standard_normal((n, c)) if with_residual else None
    w = rng.standard_normal(c)
    b = rng.standard_normal(c) if with_bias else None
    got = oracle.layernorm(x, w, b, eps, residual=r)
    h = x + r if with_residual else x
    ref = F.layer_norm(torch.from_numpy(h), (c,), torch.from_numpy(w),
                       None if b is None else torch.from_numpy(b), eps).numpy()
    if with_residual:
        got, got_h = got
        np.testing.assert_array_equal(got_h, h)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_geglu_matches_torch_exact_gelu():
    rng = np.random.default_rng(104)
    x = rng.standard_normal((11, 2 * 24)) * 4
    got = oracle.geglu(x)
    t = torch.from_numpy(x)
    ref = (F.gelu(t[:, :24], approximate="none") * t[:, 24:]).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert oracle.geglu(np.array([[0.0, 5.0]]))[0, 0] == 0.0


# --------------------------------------------------------------------------- input recipes

def test_workload_recipes():
    """Token counts of the seeded synthetic workloads (draw order: lengths first)."""
    expect = {"tiny_fp32": (8, 91), "graph_fp32": (1024, 90487),
              "contrastive_bf16": (320, 32299), "longdoc_bf16": (32, 169151)}
    for name, (b, n) in expect.items():
        lengths = workloads.draw_lengths(name, np.random.default_rng(0))
        assert lengths.shape == (b,) and int(lengths.sum()) == n, name
        assert lengths.min() >= 1 and lengths.max() <= workloads.WORKLOADS[name].max_seq_len
    x = workloads.make_inputs("tiny_fp32")
    assert x.q.dtype == torch.float32 and tuple(x.q.shape) == (91, 2, 8)


def test_packed_row_recipe_keeps_the_documents_in_order():
    """The packed-rows input recipe lays the workload's documents out in order:
    the oracle's conversion of its mask gives back exactly their lengths."""
    lengths, ids, q, _, _ = workloads.make_packed_row_inputs("contrastive_bf16", 2048)
    _, cu = oracle.pack_document_ids(ids)
    np.testing.assert_array_equal(np.diff(cu), lengths)
    assert q.shape[:2] == ids.shape and ids.shape[1] == 2048
