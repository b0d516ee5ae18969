"""fp64 CPU oracle for padding-free packed attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library neither imports nor
calls it, and it imports nothing from the CUDA library. The arithmetic lives in
``oracle.c`` (plain fp64 loops over the definitions on the page "Source code
for gigl.nn.packed_attention"); this module only builds that file with gcc and
marshals numpy arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_STATUS = {0: "ok", 2: "bad length (L < 1 or L > max_seq_len)",
           3: "token count does not fit in int32", 4: "out of memory", 5: "invalid argument"}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle status {code}: {_STATUS.get(code, 'unknown')}")
        self.code = code


def build(force: bool = False) -> str:
    """Compiles oracle.c into liboracle.so with gcc (plain -O2, IEEE fp64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, i32p, i64p, dp = (ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                               ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double))
        vp = ctypes.c_void_p
        lib.orc_pack_sequences.argtypes = [i32p, i64, i64, i64p, i32p, i64p]
        lib.orc_pack_sequences.restype = ctypes.c_int
        lib.orc_gather_rows.argtypes = [vp, i64p, i64, i64, vp]
        lib.orc_gather_rows.restype = None
        lib.orc_scatter_rows.argtypes = [vp, i32p, i64, i64, i64, vp]
        lib.orc_scatter_rows.restype = None
        lib.orc_attention_fwd.argtypes = [dp, dp, dp, i32p, i64, i64, i64, i64,
                                          ctypes.c_double, ctypes.c_int, dp, dp, ctypes.c_int]
        lib.orc_attention_fwd.restype = ctypes.c_int
        lib.orc_attention_fwd_rows.argtypes = [dp, dp, dp, i32p, i64, i64, i64, ctypes.c_double,
                                               ctypes.c_int, i64p, i64p, i64, dp, dp, ctypes.c_int]
        lib.orc_attention_fwd_rows.restype = ctypes.c_int
        lib.orc_attention_bwd.argtypes = [dp, dp, dp, dp, i32p, i64, i64, i64, ctypes.c_double,
                                          ctypes.c_int, dp, dp, dp, ctypes.c_int]
        lib.orc_attention_bwd.restype = ctypes.c_int
        lib.orc_attention_fwd_local.argtypes = [dp, dp, dp, i32p, i64, i64, i64, i64,
                                                ctypes.c_double, ctypes.c_int, i64, i64, dp, dp,
                                                ctypes.c_int]
        lib.orc_attention_fwd_local.restype = ctypes.c_int
        lib.orc_attention_fwd_rows_local.argtypes = [dp, dp, dp, i32p, i64, i64, i64,
                                                     ctypes.c_double, ctypes.c_int, i64, i64,
                                                     i64p, i64p, i64, dp, dp, ctypes.c_int]
        lib.orc_attention_fwd_rows_local.restype = ctypes.c_int
        lib.orc_attention_bwd_local.argtypes = [dp, dp, dp, dp, i32p, i64, i64, i64,
                                                ctypes.c_double, ctypes.c_int, i64, i64, dp, dp,
                                                dp, ctypes.c_int]
        lib.orc_attention_bwd_local.restype = ctypes.c_int
        lib.orc_attention_bwd_saved.argtypes = [dp, dp, dp, dp, dp, i32p, i64, i64, i64,
                                                ctypes.c_double, ctypes.c_int, i64, i64, dp, dp,
                                                dp, ctypes.c_int]
        lib.orc_attention_bwd_saved.restype = ctypes.c_int
        lib.orc_pack_document_ids.argtypes = [i32p, i64, i64, i64p, i32p, i64p, i64p]
        lib.orc_pack_document_ids.restype = ctypes.c_int
        lib.orc_flatten_packed_metadata.argtypes = [i64p, i32p, i64, i64, i64, i64p, i32p, i64p,
                                                    i64p]
        lib.orc_flatten_packed_metadata.restype = ctypes.c_int
        lib.orc_packed_positions.argtypes = [i32p, i64, i64p]
        lib.orc_packed_positions.restype = None
        lib.orc_rope.argtypes = [dp, i64p, i64, i64, i64, ctypes.c_double]
        lib.orc_rope.restype = None
        lib.orc_layernorm.argtypes = [dp, dp, dp, dp, i64, i64, ctypes.c_double, dp, dp]
        lib.orc_layernorm.restype = None
        lib.orc_geglu.argtypes = [dp, i64, i64, dp]
        lib.orc_geglu.restype = None
        lib.orc_hardware_threads.argtypes = []
        lib.orc_hardware_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(x) -> np.ndarray:
    """Widens a torch tensor or array to a contiguous float64 numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def hardware_threads() -> int:
    return int(_load().orc_hardware_threads())


def default_threads() -> int:
    return int(os.environ.get("PE_ORACLE_THREADS", hardware_threads()))


def pack_sequences(lengths, max_seq_len: int, want_index: bool = True):
    """Returns (flat_index int64 [N] or None, cu_seqlens int32 [B+1], N)."""
    lib = _load()
    lengths = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
    b = int(lengths.shape[0])
    cu = np.zeros(b + 1, dtype=np.int32)
    n = ctypes.c_int64(0)
    rc = lib.orc_pack_sequences(_ptr(lengths, ctypes.c_int32), b, int(max_seq_len), None,
                                _ptr(cu, ctypes.c_int32), ctypes.byref(n))
    if rc != 0:
        raise OracleError(rc)
    if not want_index:
        return None, cu, int(n.value)
    flat = np.zeros(max(int(n.value), 1), dtype=np.int64)
    rc = lib.orc_pack_sequences(_ptr(lengths, ctypes.c_int32), b, int(max_seq_len),
                                _ptr(flat, ctypes.c_int64), None, ctypes.byref(n))
    if rc != 0:
        raise OracleError(rc)
    return flat[: n.value].copy(), cu, int(n.value)


def pack_document_ids(ids):
    """Indexed packing mask [B, S] (document i of a row marked i, 0 = padding)
    -> (flat_index int64 [N], cu_seqlens int32 [D+1])."""
    lib = _load()
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    b, s = ids.shape
    n, d = ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib.orc_pack_document_ids(_ptr(ids, ctypes.c_int32), b, s, None, None,
                                   ctypes.byref(n), ctypes.byref(d))
    if rc != 0:
        raise OracleError(rc)
    flat = np.zeros(max(n.value, 1), dtype=np.int64)
    cu = np.zeros(d.value + 1, dtype=np.int32)
    rc = lib.orc_pack_document_ids(_ptr(ids, ctypes.c_int32), b, s, _ptr(flat, ctypes.c_int64),
                                   _ptr(cu, ctypes.c_int32), ctypes.byref(n), ctypes.byref(d))
    if rc != 0:
        raise OracleError(rc)
    return flat[: n.value].copy(), cu


def flatten_packed_metadata(token_indices, row_cu_seqlens, sequence_length: int):
    """Row-local token indices [B, S] and row-local cumulative lengths [B, M+1]
    (both -1 padded) -> (flat_index int64 [N], cu_seqlens int32 [D+1])."""
    lib = _load()
    tok = np.ascontiguousarray(np.asarray(token_indices, dtype=np.int64))
    rcu = np.ascontiguousarray(np.asarray(row_cu_seqlens, dtype=np.int32))
    b, s = tok.shape
    assert s == int(sequence_length) and rcu.shape[0] == b
    n, d = ctypes.c_int64(0), ctypes.c_int64(0)
    args = (_ptr(tok, ctypes.c_int64), _ptr(rcu, ctypes.c_int32), b, s, rcu.shape[1])
    rc = lib.orc_flatten_packed_metadata(*args, None, None, ctypes.byref(n), ctypes.byref(d))
    if rc != 0:
        raise OracleError(rc)
    flat = np.zeros(max(n.value, 1), dtype=np.int64)
    cu = np.zeros(d.value + 1, dtype=np.int32)
    rc = lib.orc_flatten_packed_metadata(*args, _ptr(flat, ctypes.c_int64),
                                         _ptr(cu, ctypes.c_int32), ctypes.byref(n),
                                         ctypes.byref(d))
    if rc != 0:
        raise OracleError(rc)
    return flat[: n.value].copy(), cu


def gather_rows(padded_rows: np.ndarray, flat_index: np.ndarray) -> np.ndarray:
    """packed[t] = padded_rows[flat_index[t]]; padded_rows is [B*S, ...]."""
    lib = _load()
    rows = np.ascontiguousarray(padded_rows)
    row_shape = rows.shape[1:]
    row_bytes = int(np.prod(row_shape, dtype=np.int64)) * rows.itemsize
    flat_index = np.ascontiguousarray(flat_index, dtype=np.int64)
    out = np.empty((flat_index.shape[0],) + row_shape, dtype=rows.dtype)
    lib.orc_gather_rows(rows.ctypes.data, _ptr(flat_index, ctypes.c_int64),
                        int(flat_index.shape[0]), row_bytes, out.ctypes.data)
    return out


def scatter_rows(packed: np.ndarray, cu_seqlens: np.ndarray, max_seq_len: int) -> np.ndarray:
    """to_dense_batch with fill 0: returns the [B, S, ...] grid."""
    lib = _load()
    packed = np.ascontiguousarray(packed)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    b = int(cu.shape[0]) - 1
    row_shape = packed.shape[1:]
    row_bytes = int(np.prod(row_shape)) * packed.itemsize
    out = np.empty((b, int(max_seq_len)) + row_shape, dtype=packed.dtype)
    lib.orc_scatter_rows(packed.ctypes.data, _ptr(cu, ctypes.c_int32), b, int(max_seq_len),
                         row_bytes, out.ctypes.data)
    return out


def attention_fwd(q, k, v, cu_seqlens, max_seq_len: int, scale: float,
                  first_token: bool = False, threads: int | None = None,
                  window: tuple[int, int] = (-1, -1)):
    """Padded-grid packed attention forward. Returns (o [Nq,H,D], lse [H,Nq]) in fp64.

    window = (left, right): the key at position j is visible from the query at
    position r iff r - left <= j <= r + right; a negative bound is unbounded."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    b = int(cu.shape[0]) - 1
    n, h, d = k.shape
    nq = b if first_token else n
    assert q.shape == (nq, h, d), (q.shape, nq, h, d)
    o = np.zeros((nq, h, d), dtype=np.float64)
    lse = np.zeros((h, nq), dtype=np.float64)
    rc = lib.orc_attention_fwd_local(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                     _ptr(v, ctypes.c_double), _ptr(cu, ctypes.c_int32), b,
                                     int(max_seq_len), h, d, float(scale), int(bool(first_token)),
                                     int(window[0]), int(window[1]),
                                     _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                     threads or default_threads())
    if rc != 0:
        raise OracleError(rc)
    return o, lse


def attention_fwd_rows(q, k, v, cu_seqlens, scale: float, first_token: bool,
                       rows, heads, threads: int | None = None,
                       window: tuple[int, int] = (-1, -1)):
    """Forward for chosen (row, head) pairs. Returns (o [R,D], lse [R]) in fp64."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    b = int(cu.shape[0]) - 1
    _, h, d = k.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int64)
    r = int(rows.shape[0])
    o = np.zeros((r, d), dtype=np.float64)
    lse = np.zeros((r,), dtype=np.float64)
    rc = lib.orc_attention_fwd_rows_local(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                    _ptr(v, ctypes.c_double), _ptr(cu, ctypes.c_int32), b, h, d,
                                    float(scale), int(bool(first_token)),
                                    int(window[0]), int(window[1]),
                                    _ptr(rows, ctypes.c_int64), _ptr(heads, ctypes.c_int64), r,
                                    _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                    threads or default_threads())
    if rc != 0:
        raise OracleError(rc)
    return o, lse


def attention_bwd(q, k, v, dout, cu_seqlens, scale: float, first_token: bool = False,
                  threads: int | None = None, window: tuple[int, int] = (-1, -1),
                  out=None):
    """Analytic gradients. Returns (dq, dk, dv) in fp64.

    out: the forward output as the backward op receives it (shaped like q).
    When given, Delta = dO . out is formed from it as saved (a bf16 output is
    the exact one rounded), the backward op of page "Source code for
    gigl.nn.packed_attention" taking the saved output; None forms Delta from
    the exact fp64 output."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    b = int(cu.shape[0]) - 1
    _, h, d = k.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    saved = None
    if out is not None:
        saved = _f64(out)
        if saved.shape != q.shape:
            raise ValueError(f"out shape {saved.shape} != q shape {q.shape}")
    rc = lib.orc_attention_bwd_saved(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                               _ptr(v, ctypes.c_double), _ptr(dout, ctypes.c_double),
                               None if saved is None else _ptr(saved, ctypes.c_double),
                               _ptr(cu, ctypes.c_int32), b, h, d, float(scale),
                               int(bool(first_token)), int(window[0]), int(window[1]),
                               _ptr(dq, ctypes.c_double),
                               _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
                               threads or default_threads())
    if rc != 0:
        raise OracleError(rc)
    return dq, dk, dv


# --------------------------------------------------------------------------- layer tail

def packed_positions(cu_seqlens) -> np.ndarray:
    """Position of every token inside its own sequence (int64 [N])."""
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    lib.orc_packed_positions(_ptr(cu, ctypes.c_int32), int(cu.shape[0]) - 1,
                             _ptr(pos, ctypes.c_int64))
    return pos


def rope(x, positions, theta: float) -> np.ndarray:
    """Split-half rotary embedding of x [N, H, D] at the given positions (fp64 copy)."""
    lib = _load()
    y = _f64(x).copy()
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    n, h, d = y.shape
    lib.orc_rope(_ptr(y, ctypes.c_double), _ptr(pos, ctypes.c_int64), n, h, d, float(theta))
    return y


def layernorm(x, weight, bias=None, eps: float = 1e-5, residual=None):
    """LayerNorm over the last dim of x [N, C] (of x + residual when given).
    Returns y, plus h = x + residual when a residual is given."""
    lib = _load()
    xx = _f64(x)
    n, c = xx.shape
    w = _f64(weight)
    b = None if bias is None else _f64(bias)
    r = None if residual is None else _f64(residual)
    y = np.zeros_like(xx)
    h = np.zeros_like(xx) if residual is not None else None
    dp = lambda a: None if a is None else _ptr(a, ctypes.c_double)
    lib.orc_layernorm(dp(xx), dp(r), dp(w), dp(b), n, c, float(eps), dp(y), dp(h))
    return (y, h) if residual is not None else y


def geglu(x) -> np.ndarray:
    """gelu(x[:, :F]) * x[:, F:] for x [N, 2F], exact GELU."""
    lib = _load()
    xx = _f64(x)
    n, f2 = xx.shape
    y = np.zeros((n, f2 // 2), dtype=np.float64)
    lib.orc_geglu(_ptr(xx, ctypes.c_double), n, f2 // 2, _ptr(y, ctypes.c_double))
    return y
