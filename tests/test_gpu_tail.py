"""The packed encoder layer tail on the GPU against the fp64 oracle: packed
position ids, split-half RoPE, (residual-)LayerNorm, GeGLU (page
"packed-encoders 0.1.0"), and the whole tail captured in a CUDA graph.

Tolerances: fp32 max abs error <= 1e-4. In bf16 these kernels compute in fp32
on the same bf16 inputs as the oracle and round once at the output, so the
bound is |err| <= 2^-8 |y| + 1e-5 per element (round-to-nearest bf16 is within
half an ulp, at most 2^-8 of the magnitude); unlike attention outputs, their
values are not bounded by the inputs' scale, so a fixed absolute bar does not
fit them."""

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


def _close(got, want, dtype, what):
    got, want = to64(got), np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape and np.all(np.isfinite(got)), what
    err = np.abs(got - want)
    if dtype == torch.float32:
        assert float(err.max()) <= 1e-4, f"{what}: {float(err.max()):.3e}"
    else:
        bound = 2.0 ** -8 * np.abs(want) + 1e-5
        worst = float((err - bound).max())
        assert worst <= 0, f"{what}: error exceeds 2^-8|y| + 1e-5 by {worst:.3e}"


def test_positions_worked_example(golden):
    g = golden("packed_position_ids_example.txt")
    cu = torch.tensor(g["cu_seqlens"], dtype=torch.int32, device=DEV)
    assert pe.pe_packed_positions(cu, 16).cpu().tolist() == g["position_ids"]


def test_positions_match_oracle():
    lengths = np.random.default_rng(201).integers(1, 900, 1500)
    _, cu, n = oracle.pack_sequences(lengths, int(lengths.max()))
    got = pe.pe_packed_positions(torch.from_numpy(cu).to(DEV), n).cpu().numpy()
    assert np.array_equal(got, oracle.packed_positions(cu))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d,hq,hk,theta", [(64, 12, 12, 160000.0), (128, 4, 2, 10000.0),
                                           (32, 3, 0, 10000.0)])
def test_rope_matches_oracle(dtype, d, hq, hk, theta):
    lengths = [8192, 5000, 1, 37, 700]
    _, cu, n = oracle.pack_sequences(lengths, 8192)
    rng = np.random.default_rng(202)
    q = torch.from_numpy(rng.standard_normal((n, hq, d))).to(dtype)
    k = torch.from_numpy(rng.standard_normal((n, hk, d))).to(dtype) if hk else None
    pos = oracle.packed_positions(cu)
    qd, kd = q.to(DEV), (k.to(DEV) if k is not None else None)
    pe.pe_rope_packed(qd, kd, torch.from_numpy(pos).to(DEV), theta)
    _close(qd, oracle.rope(q, pos, theta), dtype, "rope q")
    if k is not None:
        _close(kd, oracle.rope(k, pos, theta), dtype, "rope k")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("c", [768, 1024, 1000, 64, 128, 256, 2048])
@pytest.mark.parametrize("with_bias,with_residual", [(False, True), (True, False), (False, False)])
def test_layernorm_matches_oracle(dtype, c, with_bias, with_residual):
    rng = np.random.default_rng(203)
    n = 3000
    x = torch.from_numpy(rng.standard_normal((n, c)) * 2 + 0.5).to(dtype)
    r = torch.from_numpy(rng.standard_normal((n, c))).to(dtype) if with_residual else None
    w = torch.from_numpy(rng.uniform(0.5, 1.5, c)).to(dtype)
    b = torch.from_numpy(rng.normal(0, 0.1, c)).to(dtype) if with_bias else None
    res = pe.pe_layernorm(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV), 1e-5,
                          residual=None if r is None else r.to(DEV))
    if with_residual:
        y, h = res
        hx = x + r                                  # the sum as stored, in the I/O dtype
        assert torch.equal(h.cpu(), hx)
        ref = oracle.layernorm(hx, w, b, 1e-5)
    else:
        y = res
        ref = oracle.layernorm(x, w, b, 1e-5)
    _close(y, ref, dtype, f"layernorm c={c}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("f", [1152, 100, 7])
def test_geglu_matches_oracle(dtype, f):
    x = torch.from_numpy(np.random.default_rng(204).standard_normal((2500, 2 * f)) * 1.5).to(dtype)
    _close(pe.pe_geglu(x.to(DEV)), oracle.geglu(x), dtype, f"geglu f={f}")


def test_gelu_against_exact_gelu_on_a_dense_range():
    """GeGLU's GELU takes erf from Abramowitz and Stegun's formula 7.1.26
    (|error| <= 1.5e-7 in erf, so |error| <= 0.75e-7 |x| in GELU before fp32
    rounding): with a gate of 1, fp32 outputs over [-12, 12] stay within
    3e-6 max(1, |x|) of the exact GELU in fp64."""
    x = np.linspace(-12.0, 12.0, 200001).astype(np.float32)
    inp = torch.from_numpy(np.stack([x, np.ones_like(x)], axis=1))
    got = to64(pe.pe_geglu(inp.to(DEV))).ravel()
    exact = to64(torch.nn.functional.gelu(torch.from_numpy(x.astype(np.float64))))
    err = np.abs(got - exact)
    assert float((err - 3e-6 * np.maximum(1.0, np.abs(x))).max()) <= 0


def test_layer_tail_in_a_cuda_graph():
    """positions -> RoPE(q, k) -> attention -> residual-LayerNorm -> GeGLU,
    captured once and replayed on new inputs, equals the eager calls."""
    lengths = [300, 17, 129, 1000, 64]
    h, d, c = 4, 64, 256
    _, cu_np, n = oracle.pack_sequences(lengths, 1000)
    cu = torch.from_numpy(cu_np).to(DEV)
    gen = torch.Generator(device=DEV).manual_seed(205)
    mk = lambda *s: torch.randn(*s, generator=gen, device=DEV).to(torch.bfloat16)
    q, k, v = mk(n, h, d), mk(n, h, d), mk(n, h, d)
    resid, w = mk(n, c), mk(c)
    mlp_in = mk(n, 2 * c)
    ws = torch.empty(pe.attention_workspace_bytes(torch.bfloat16, len(lengths), n, h, d, 1000),
                     dtype=torch.uint8, device=DEV)
    static = [t.clone() for t in (q, k, v, resid, mlp_in)]

    def tail(q_, k_, v_, r_, m_):
        pos = pe.pe_packed_positions(cu, n)
        pe.pe_rope_packed(q_, k_, pos, 160000.0)
        out, _ = pe.pe_packed_attention_fwd(q_, k_, v_, cu, 1000, 0.125, workspace=ws)
        y, hsum = pe.pe_layernorm(out.reshape(n, c), w, None, 1e-5, residual=r_)
        return y, hsum, pe.pe_geglu(m_)

    tail(*[t.clone() for t in static])                # warm-up: library and tensor-map setup
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = tail(*static)
    for trial in range(2):
        fresh = [mk(*t.shape) for t in static]
        for dst, src in zip(static, fresh):
            dst.copy_(src)
        graph.replay()
        want = tail(*[t.clone() for t in fresh])
        torch.cuda.synchronize()
        for got, ref in zip(outs, want):
            assert torch.equal(got, ref), f"replay {trial} differs from the eager tail"
