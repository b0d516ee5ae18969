"""Why the bf16 gradient bar skips near-cancelled rows in the cosine check.

The forward rounds P to bf16 before P V and stores O in bf16; the backward
rounds P (for dV = P^T dO) and dS = P o (dP - Delta) (for dq = scale dS k and
dk = scale dS^T q), and forms Delta = rowsum(dO o O) from the stored O. This
test replays exactly those roundings in numpy (fp32 products and sums, round
to nearest even where the kernels round) on the local-window gradient case
whose worst row motivated the reading, and compares the result with the
oracle's fp64 gradients:

* the replay itself misses the 0.999 cosine bar on some rows: the bar is
  unattainable by any implementation that rounds where this one must;
* every such row has an exact norm below a tenth of the tensor's median row
  norm (a near-cancellation: with a right-hand window of 1 the first query of
  a sequence sees two keys and dq_0 = scale P_0 P_1 (dP_0 - dP_1)(k_0 - k_1));
* with those rows left to the absolute bar, the replay passes, as the GPU
  kernels must.
"""

import math

import numpy as np
import torch

import oracle
from padding_free_packed_gb300 import workloads
from parity import BF16_ATOL, BF16_COS, GRAD_COS_MIN_NORM_FRAC, row_cosine

LENGTHS = [1, 63, 65, 128, 129, 300, 2, 257, 520]
WINDOW = (200, 1)


def bf16(x):
    """Round float32 values to bfloat16 (nearest, ties to even), kept as float32."""
    a = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    a = ((a + 0x7FFF + ((a >> 16) & 1)) >> 16) << 16
    return a.astype(np.uint32).view(np.float32)


def _replay(q, k, v, do, cu, scale):
    """The bf16 forward and backward pipelines, per (sequence, head), in float32."""
    n, h, d = k.shape
    dq, dk, dv = (np.zeros((n, h, d), np.float32) for _ in range(3))
    wl, wr = WINDOW
    log2e = np.float32(math.log2(math.e))
    for i in range(len(cu) - 1):
        s0, s1 = int(cu[i]), int(cu[i + 1])
        pos = np.arange(s1 - s0)
        visible = (pos[None, :] >= pos[:, None] - wl) & (pos[None, :] <= pos[:, None] + wr)
        for hh in range(h):
            qs, ks, vs, dos = (t[s0:s1, hh].astype(np.float32) for t in (q, k, v, do))
            s = np.where(visible, (qs @ ks.T).astype(np.float32) * np.float32(scale) * log2e,
                         -np.inf).astype(np.float32)
            # Forward: P = 2^(s - m) rounded to bf16 for P V, l summed in fp32.
            m = s.max(axis=1, keepdims=True)
            pf = np.exp2(s - m).astype(np.float32)
            l = pf.sum(axis=1, keepdims=True, dtype=np.float32)
            o = bf16((bf16(pf) @ vs) / l)
            lse2 = (m + np.log2(l)).astype(np.float32)
            # Backward: P recomputed from the saved log-sum-exp.
            p = np.exp2(s - lse2).astype(np.float32)
            dp = (dos @ vs.T).astype(np.float32)
            delta = np.sum(dos * o, axis=1, dtype=np.float32)
            ds = bf16(p * (dp - delta[:, None]))
            dq[s0:s1, hh] = bf16(np.float32(scale) * (ds @ ks))
            dk[s0:s1, hh] = bf16(np.float32(scale) * (ds.T @ qs))
            dv[s0:s1, hh] = bf16(bf16(p).T @ dos)
    return dq, dk, dv


def test_bf16_rounding_alone_breaks_the_cosine_bar_only_on_near_cancelled_rows(oracle_lib):
    x = workloads.make_custom(LENGTHS, 2, 64, torch.bfloat16, seed=33, with_dout=True)
    _, cu, _ = oracle.pack_sequences(x.lengths, max(LENGTHS))
    scale = 1.0 / math.sqrt(64)
    q, k, v, do = (t.float().numpy() for t in (x.q, x.k, x.v, x.dout))
    got = _replay(q, k, v, do, cu, scale)
    want = oracle.attention_bwd(x.q, x.k, x.v, x.dout, cu, scale, window=WINDOW)
    worst_all, worst_kept = 1.0, 1.0
    for g, w in zip(got, want):
        g64 = g.astype(np.float64)
        assert float(np.abs(g64 - w).max()) <= BF16_ATOL
        cos = row_cosine(g64, w)
        norms = np.linalg.norm(w.reshape(-1, w.shape[-1]), axis=1)
        kept = norms >= GRAD_COS_MIN_NORM_FRAC * np.median(norms)
        worst_all = min(worst_all, float(cos.min()))
        worst_kept = min(worst_kept, float(cos[kept].min()))
        # Every row below the cosine bar is a near-cancellation.
        assert np.all(kept[cos < BF16_COS] == False)  # noqa: E712
    assert worst_all < BF16_COS        # rounding alone misses the strict bar ...
    assert worst_kept >= BF16_COS      # ... only on the rows the reading exempts
