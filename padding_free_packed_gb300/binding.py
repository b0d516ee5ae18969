"""Thin Python binding over libpe's C ABI (include/pe.h).

Argument marshalling only: every step of the packed-attention path runs in the
library's CUDA kernels. PyTorch provides device memory (outputs and
workspaces are torch tensors) and the current CUDA stream. There is no CPU
fallback: if libpe.so is missing or the device is not sm_103a the calls raise.
"""

from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpe.so")

PE_BF16 = 0
PE_FP32 = 1

EXPORTED = (
    "pe_status_string", "pe_abi_version", "pe_pack_workspace_size", "pe_pack_sequences",
    "pe_gather_packed", "pe_scatter_padded", "pe_attention_workspace_size",
    "pe_packed_attention_fwd", "pe_packed_attention_bwd", "pe_packed_attention_fwd_local",
    "pe_packed_attention_bwd_local", "pe_read_device_status", "pe_attention_kernel",
    "pe_rows_workspace_size", "pe_pack_document_ids", "pe_flatten_packed_metadata",
    "pe_packed_positions", "pe_rope_packed", "pe_layernorm", "pe_geglu", "pe_upload_packed",
    "pe_download_padded", "pe_packed_attention_fwd_noalloc", "pe_read_noalloc_status",
    "pe_set_wait_limit_ns", "pe_attention_kernel_local",
)

_lib = None


class PackedAttentionError(RuntimeError):
    def __init__(self, call: str, status: int, text: str):
        super().__init__(f"{call} failed with status {status}: {text}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Loads libpe.so and declares its signatures. Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libpe.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    c = ctypes
    i32, i64, vp, sz = c.c_int32, c.c_int64, c.c_void_p, c.c_size_t
    lib.pe_status_string.argtypes = [c.c_int]
    lib.pe_status_string.restype = c.c_char_p
    lib.pe_abi_version.argtypes = []
    lib.pe_abi_version.restype = c.c_int
    lib.pe_pack_workspace_size.argtypes = [i32]
    lib.pe_pack_workspace_size.restype = sz
    lib.pe_pack_sequences.argtypes = [vp, i32, i32, vp, vp, c.POINTER(i64), vp, sz, vp]
    lib.pe_pack_sequences.restype = c.c_int
    lib.pe_gather_packed.argtypes = [vp, vp, i64, i64, vp, vp]
    lib.pe_gather_packed.restype = c.c_int
    lib.pe_scatter_padded.argtypes = [vp, vp, i32, i32, i64, vp, vp]
    lib.pe_scatter_padded.restype = c.c_int
    lib.pe_attention_workspace_size.argtypes = [c.c_int, i32, i64, i32, i32, i32, c.c_int, c.c_int]
    lib.pe_attention_workspace_size.restype = sz
    lib.pe_packed_attention_fwd.argtypes = [c.c_int, i32, i64, i32, i32, i32, vp, vp, vp, vp,
                                            c.c_float, c.c_int, vp, vp, vp, sz, vp]
    lib.pe_packed_attention_fwd.restype = c.c_int
    lib.pe_packed_attention_bwd.argtypes = [c.c_int, i32, i64, i32, i32, i32, vp, vp, vp, vp,
                                            c.c_float, c.c_int, vp, vp, vp, vp, vp, vp, vp, sz,
                                            vp]
    lib.pe_packed_attention_bwd.restype = c.c_int
    lib.pe_packed_attention_fwd_local.argtypes = [c.c_int, i32, i64, i32, i32, i32, vp, vp, vp,
                                                  vp, c.c_float, i32, i32, c.c_int, vp, vp, vp,
                                                  sz, vp]
    lib.pe_packed_attention_fwd_local.restype = c.c_int
    lib.pe_packed_attention_bwd_local.argtypes = [c.c_int, i32, i64, i32, i32, i32, vp, vp, vp,
                                                  vp, c.c_float, i32, i32, c.c_int, vp, vp, vp,
                                                  vp, vp, vp, vp, sz, vp]
    lib.pe_packed_attention_bwd_local.restype = c.c_int
    lib.pe_rows_workspace_size.argtypes = [i32]
    lib.pe_rows_workspace_size.restype = sz
    lib.pe_pack_document_ids.argtypes = [vp, i32, i32, vp, vp, c.POINTER(i64), c.POINTER(i32),
                                         vp, sz, vp]
    lib.pe_pack_document_ids.restype = c.c_int
    lib.pe_flatten_packed_metadata.argtypes = [vp, vp, i32, i32, i32, vp, vp, c.POINTER(i64),
                                               c.POINTER(i32), vp, sz, vp]
    lib.pe_flatten_packed_metadata.restype = c.c_int
    lib.pe_upload_packed.argtypes = [vp, vp, i32, i32, i64, vp, vp]
    lib.pe_upload_packed.restype = c.c_int
    lib.pe_download_padded.argtypes = [vp, vp, i32, i32, i64, vp, vp]
    lib.pe_download_padded.restype = c.c_int
    lib.pe_packed_positions.argtypes = [vp, i32, i64, vp, vp]
    lib.pe_packed_positions.restype = c.c_int
    lib.pe_rope_packed.argtypes = [c.c_int, vp, i32, vp, i32, vp, i64, i32, c.c_double, vp]
    lib.pe_rope_packed.restype = c.c_int
    lib.pe_layernorm.argtypes = [c.c_int, vp, vp, vp, vp, i64, i32, c.c_float, vp, vp, vp]
    lib.pe_layernorm.restype = c.c_int
    lib.pe_geglu.argtypes = [c.c_int, vp, i64, i32, vp, vp]
    lib.pe_geglu.restype = c.c_int
    lib.pe_attention_kernel.argtypes = [c.c_int, i32, c.c_int, c.c_int]
    lib.pe_attention_kernel.restype = c.c_char_p
    lib.pe_attention_kernel_local.argtypes = [c.c_int, i32, i32, i32, i32, c.c_int, c.c_int]
    lib.pe_attention_kernel_local.restype = c.c_char_p
    lib.pe_read_device_status.argtypes = [vp, vp]
    lib.pe_read_device_status.restype = c.c_int
    lib.pe_read_noalloc_status.argtypes = [vp]
    lib.pe_read_noalloc_status.restype = c.c_int
    lib.pe_set_wait_limit_ns.argtypes = [c.c_uint64]
    lib.pe_set_wait_limit_ns.restype = c.c_uint64
    lib.pe_packed_attention_fwd_noalloc.argtypes = [c.c_int, i32, i64, i32, i32, i32, vp, vp, vp,
                                                    vp, c.c_float, c.c_int, vp, vp, vp]
    lib.pe_packed_attention_fwd_noalloc.restype = c.c_int
    _lib = lib
    return lib


def _check(call: str, status: int):
    if status != 0:
        text = load_library().pe_status_string(status).decode()
        raise PackedAttentionError(call, status, text)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return PE_BF16
    if dtype == torch.float32:
        return PE_FP32
    raise TypeError(f"unsupported dtype {dtype}: bfloat16 or float32 only")


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    return t.contiguous()


def _cuda_or_pinned(t: torch.Tensor, name: str) -> torch.Tensor:
    """A CUDA tensor, or a pinned host tensor that kernels address directly."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def pe_pack_sequences(lengths: torch.Tensor, max_seq_len: int):
    """Returns (flat_index int64 [N], cu_seqlens int32 [B+1], N) for device lengths."""
    lib = load_library()
    lengths = _cuda(lengths, "lengths").to(torch.int32)
    b = int(lengths.numel())
    dev = lengths.device
    flat = torch.empty(max(b * int(max_seq_len), 1), dtype=torch.int64, device=dev)
    cu = torch.empty(b + 1, dtype=torch.int32, device=dev)
    ws = _workspace(lib.pe_pack_workspace_size(b), dev)
    n = ctypes.c_int64(0)
    _check("pe_pack_sequences",
           lib.pe_pack_sequences(_ptr(lengths), b, int(max_seq_len), _ptr(flat), _ptr(cu),
                                 ctypes.byref(n), _ptr(ws), ws.numel(), _stream(dev)))
    return flat[: n.value], cu, int(n.value)


def pe_pack_document_ids(document_ids: torch.Tensor):
    """Indexed packing mask [B, S] (document i of a row marked i, 0 = padding)
    -> (flat_index int64 [N] into the [B, S] layout, cu_seqlens int32 [D+1], N)."""
    lib = load_library()
    ids = _cuda(document_ids, "document_ids").to(torch.int32)
    b, s = (int(x) for x in ids.shape)
    dev = ids.device
    flat = torch.empty(max(b * s, 1), dtype=torch.int64, device=dev)
    cu = torch.empty(b * s + 1, dtype=torch.int32, device=dev)
    ws = _workspace(lib.pe_rows_workspace_size(b), dev)
    n, d = ctypes.c_int64(0), ctypes.c_int32(0)
    _check("pe_pack_document_ids",
           lib.pe_pack_document_ids(_ptr(ids), b, s, _ptr(flat), _ptr(cu), ctypes.byref(n),
                                    ctypes.byref(d), _ptr(ws), ws.numel(), _stream(dev)))
    return flat[: n.value], cu[: d.value + 1], int(n.value)


def pe_flatten_packed_metadata(token_indices: torch.Tensor, row_cu_seqlens: torch.Tensor):
    """Row-local token indices [B, S] and row-local cumulative lengths [B, M+1]
    (both -1 padded) -> (flat_index int64 [N], cu_seqlens int32 [D+1], N)."""
    lib = load_library()
    tok = _cuda(token_indices, "token_indices").to(torch.int64)
    rcu = _cuda(row_cu_seqlens, "row_cu_seqlens").to(torch.int32)
    b, s = (int(x) for x in tok.shape)
    m1 = int(rcu.shape[1])
    if int(rcu.shape[0]) != b:
        raise ValueError("token_indices and row_cu_seqlens disagree on the number of rows")
    dev = tok.device
    flat = torch.empty(max(b * s, 1), dtype=torch.int64, device=dev)
    cu = torch.empty(b * max(m1 - 1, 0) + 1, dtype=torch.int32, device=dev)
    ws = _workspace(lib.pe_rows_workspace_size(b), dev)
    n, d = ctypes.c_int64(0), ctypes.c_int32(0)
    _check("pe_flatten_packed_metadata",
           lib.pe_flatten_packed_metadata(_ptr(tok), _ptr(rcu), b, s, m1, _ptr(flat), _ptr(cu),
                                          ctypes.byref(n), ctypes.byref(d), _ptr(ws), ws.numel(),
                                          _stream(dev)))
    return flat[: n.value], cu[: d.value + 1], int(n.value)


def pe_gather_packed(padded: torch.Tensor, flat_index: torch.Tensor, num_tokens: int | None = None,
                     out: torch.Tensor | None = None):
    """packed[t] = padded.flatten(0, 1)[flat_index[t]] for a [B, S, ...] grid.
    The grid may be pinned host memory: only the real rows cross the host link."""
    lib = load_library()
    padded = _cuda_or_pinned(padded, "padded")
    flat_index = _cuda(flat_index, "flat_index")
    dev = flat_index.device
    n = int(flat_index.numel()) if num_tokens is None else int(num_tokens)
    row_shape = tuple(padded.shape[2:])
    packed = (torch.empty((n,) + row_shape, dtype=padded.dtype, device=dev) if out is None
              else out)
    row_bytes = padded.element_size() * math.prod(row_shape)
    _check("pe_gather_packed",
           lib.pe_gather_packed(_ptr(padded), _ptr(flat_index), n, row_bytes, _ptr(packed),
                                _stream(dev)))
    return packed


def pe_upload_packed(padded_host: torch.Tensor, lengths_host, out: torch.Tensor) -> torch.Tensor:
    """Copies the real rows of a host [B, S, ...] grid into the packed device
    buffer `out` [sum L, ...] with one asynchronous copy per sequence on the
    current stream of out's device (pinned host memory for asynchrony)."""
    lib = load_library()
    if padded_host.is_cuda or not padded_host.is_contiguous():
        raise ValueError("padded_host must be a contiguous host tensor")
    lengths = np.ascontiguousarray(np.asarray(lengths_host, dtype=np.int32))
    b, s = int(padded_host.shape[0]), int(padded_host.shape[1])
    if lengths.shape != (b,):
        raise ValueError("one length per grid row")
    row_bytes = padded_host.element_size() * math.prod(tuple(padded_host.shape[2:]))
    # Checked before anything is enqueued: every copy writes L_i rows into out.
    if out.dtype != padded_host.dtype or not out.is_contiguous() or out.numel() != int(
            lengths.sum()) * (row_bytes // padded_host.element_size()):
        raise ValueError("out must be contiguous and hold sum(L) rows of the grid's row shape "
                         "and dtype")
    out = _cuda(out, "out")
    _check("pe_upload_packed",
           lib.pe_upload_packed(_ptr(padded_host), lengths.ctypes.data, b, s, row_bytes,
                                _ptr(out), _stream(out.device)))
    return out


def pe_download_padded(packed: torch.Tensor, lengths_host, out_host: torch.Tensor) -> torch.Tensor:
    """Copies the packed device rows [sum L, ...] into the real rows of the host
    [B, S, ...] grid `out_host` with one asynchronous copy per sequence on the
    current stream of packed's device (pinned host memory for asynchrony). Pad
    rows of out_host are not written: allocate it zeroed for to_dense_batch's
    zero fill."""
    lib = load_library()
    if out_host.is_cuda or not out_host.is_contiguous():
        raise ValueError("out_host must be a contiguous host tensor")
    lengths = np.ascontiguousarray(np.asarray(lengths_host, dtype=np.int32))
    b, s = int(out_host.shape[0]), int(out_host.shape[1])
    if lengths.shape != (b,):
        raise ValueError("one length per grid row")
    row_bytes = out_host.element_size() * math.prod(tuple(out_host.shape[2:]))
    if packed.dtype != out_host.dtype or not packed.is_contiguous() or packed.numel() != int(
            lengths.sum()) * (row_bytes // out_host.element_size()):
        raise ValueError("packed must be contiguous and hold sum(L) rows of the grid's row "
                         "shape and dtype")
    packed = _cuda(packed, "packed")
    _check("pe_download_padded",
           lib.pe_download_padded(_ptr(packed), lengths.ctypes.data, b, s, row_bytes,
                                  _ptr(out_host), _stream(packed.device)))
    return out_host


def pe_scatter_padded(packed: torch.Tensor, cu_seqlens: torch.Tensor, max_seq_len: int,
                      out: torch.Tensor | None = None):
    """Returns the zero-padded [B, S, ...] grid of a packed [N, ...] buffer; `out`
    may be pinned host memory (the rows are then written across the host link)."""
    lib = load_library()
    packed = _cuda(packed, "packed")
    if out is not None:
        out = _cuda_or_pinned(out, "out")
    cu_seqlens = _cuda(cu_seqlens, "cu_seqlens")
    b = int(cu_seqlens.numel()) - 1
    row_shape = tuple(packed.shape[1:])
    if out is None:
        out = torch.empty((b, int(max_seq_len)) + row_shape, dtype=packed.dtype,
                          device=packed.device)
    row_bytes = packed.element_size() * math.prod(row_shape)
    _check("pe_scatter_padded",
           lib.pe_scatter_padded(_ptr(packed), _ptr(cu_seqlens), b, int(max_seq_len), row_bytes,
                                 _ptr(out), _stream(packed.device)))
    return out


def attention_workspace_bytes(dtype, num_sequences, num_tokens, num_heads, head_dim,
                              max_seq_len, query_is_first_token=False, backward=False) -> int:
    return int(load_library().pe_attention_workspace_size(
        _dtype_code(dtype), int(num_sequences), int(num_tokens), int(num_heads), int(head_dim),
        int(max_seq_len), int(bool(query_is_first_token)), int(bool(backward))))


def pe_packed_attention_fwd(q, k, v, cu_seqlens, max_seq_len: int, scale: float | None = None,
                            query_is_first_token: bool = False, need_lse: bool = False,
                            out=None, lse=None, workspace=None):
    """Packed attention forward. Returns (out, lse or None)."""
    return _forward(None, q, k, v, cu_seqlens, max_seq_len, scale, query_is_first_token,
                    need_lse, out, lse, workspace)


def pe_packed_attention_fwd_local(q, k, v, cu_seqlens, max_seq_len: int, window_left: int,
                                  window_right: int, scale: float | None = None,
                                  query_is_first_token: bool = False, need_lse: bool = False,
                                  out=None, lse=None, workspace=None):
    """Local (sliding-window) packed attention forward: the query at position r
    sees keys r - window_left .. r + window_right of its own sequence (a negative
    bound is unbounded). Returns (out, lse or None)."""
    return _forward((int(window_left), int(window_right)), q, k, v, cu_seqlens, max_seq_len,
                    scale, query_is_first_token, need_lse, out, lse, workspace)


def _forward(window, q, k, v, cu_seqlens, max_seq_len, scale, query_is_first_token, need_lse,
             out, lse, workspace):
    lib = load_library()
    q, k, v = _cuda(q, "q"), _cuda(k, "k"), _cuda(v, "v")
    cu_seqlens = _cuda(cu_seqlens, "cu_seqlens")
    n, h, d = k.shape
    b = int(cu_seqlens.numel()) - 1
    nq = b if query_is_first_token else n
    if tuple(q.shape) != (nq, h, d) or v.shape != k.shape or q.dtype != k.dtype:
        raise ValueError(f"shape/dtype mismatch: q {tuple(q.shape)} k {tuple(k.shape)}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if need_lse and lse is None:
        lse = torch.empty((h, nq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(attention_workspace_bytes(q.dtype, b, n, h, d, max_seq_len,
                                                         query_is_first_token, False), q.device)
    head = (_dtype_code(q.dtype), b, n, h, d, int(max_seq_len), _ptr(q), _ptr(k), _ptr(v),
            _ptr(cu_seqlens), scale)
    tail = (int(bool(query_is_first_token)), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel(), _stream(q.device))
    if window is None:
        _check("pe_packed_attention_fwd", lib.pe_packed_attention_fwd(*head, *tail))
    else:
        _check("pe_packed_attention_fwd_local",
               lib.pe_packed_attention_fwd_local(*head, window[0], window[1], *tail))
    return out, lse


def pe_packed_attention_bwd(dout, q, k, v, out, lse, cu_seqlens, max_seq_len: int,
                            scale: float | None = None, query_is_first_token: bool = False,
                            workspace=None):
    """Packed attention backward. Returns (dq, dk, dv)."""
    return _backward(None, dout, q, k, v, out, lse, cu_seqlens, max_seq_len, scale,
                     query_is_first_token, workspace)


def pe_packed_attention_bwd_local(dout, q, k, v, out, lse, cu_seqlens, max_seq_len: int,
                                  window_left: int, window_right: int,
                                  scale: float | None = None, query_is_first_token: bool = False,
                                  workspace=None):
    """Local (sliding-window) packed attention backward; out and lse come from
    pe_packed_attention_fwd_local with the same window. Returns (dq, dk, dv)."""
    return _backward((int(window_left), int(window_right)), dout, q, k, v, out, lse, cu_seqlens,
                     max_seq_len, scale, query_is_first_token, workspace)


def _backward(window, dout, q, k, v, out, lse, cu_seqlens, max_seq_len, scale,
              query_is_first_token, workspace):
    lib = load_library()
    q, k, v = _cuda(q, "q"), _cuda(k, "k"), _cuda(v, "v")
    out, dout, lse = _cuda(out, "out"), _cuda(dout, "dout"), _cuda(lse, "lse")
    cu_seqlens = _cuda(cu_seqlens, "cu_seqlens")
    n, h, d = k.shape
    b = int(cu_seqlens.numel()) - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = _workspace(attention_workspace_bytes(q.dtype, b, n, h, d, max_seq_len,
                                                         query_is_first_token, True), q.device)
    head = (_dtype_code(q.dtype), b, n, h, d, int(max_seq_len), _ptr(q), _ptr(k), _ptr(v),
            _ptr(cu_seqlens), scale)
    tail = (int(bool(query_is_first_token)), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
            _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), _stream(q.device))
    if window is None:
        _check("pe_packed_attention_bwd", lib.pe_packed_attention_bwd(*head, *tail))
    else:
        _check("pe_packed_attention_bwd_local",
               lib.pe_packed_attention_bwd_local(*head, window[0], window[1], *tail))
    return dq, dk, dv


def pe_attention_kernel(dtype: torch.dtype, head_dim: int, query_is_first_token: bool = False,
                        backward: bool = False, window=None, max_seq_len: int | None = None) -> str:
    """Kernel family the forward (or backward) dispatches to for these arguments;
    with window = (left, right) and max_seq_len, that of the local calls."""
    lib = load_library()
    if window is None:
        return lib.pe_attention_kernel(
            _dtype_code(dtype), int(head_dim), int(bool(query_is_first_token)),
            int(bool(backward))).decode()
    if max_seq_len is None:
        raise ValueError("a window needs max_seq_len")
    return lib.pe_attention_kernel_local(
        _dtype_code(dtype), int(head_dim), int(max_seq_len), int(window[0]), int(window[1]),
        int(bool(query_is_first_token)), int(bool(backward))).decode()


def pe_read_device_status(workspace: torch.Tensor) -> int:
    """Device-side status left in an attention workspace (0 = the layout passed
    its check and every pipeline wait completed)."""
    lib = load_library()
    return int(lib.pe_read_device_status(_ptr(workspace), _stream(workspace.device)))


def pe_set_wait_limit_ns(ns: int) -> int:
    """Process-wide limit of the kernels' bounded pipeline waits (0 = the
    default 2 s); returns the previous limit."""
    return int(load_library().pe_set_wait_limit_ns(int(ns)))


def pe_packed_attention_fwd_noalloc(q, k, v, cu_seqlens, max_seq_len: int,
                                    scale: float | None = None,
                                    query_is_first_token: bool = False, need_lse: bool = False,
                                    out=None, lse=None):
    """The forward without a workspace: the library's static device array holds
    its scratch. Returns (out, lse or None)."""
    lib = load_library()
    q, k, v = _cuda(q, "q"), _cuda(k, "k"), _cuda(v, "v")
    cu_seqlens = _cuda(cu_seqlens, "cu_seqlens")
    n, h, d = k.shape
    b = int(cu_seqlens.numel()) - 1
    nq = b if query_is_first_token else n
    if tuple(q.shape) != (nq, h, d) or v.shape != k.shape or q.dtype != k.dtype:
        raise ValueError(f"shape/dtype mismatch: q {tuple(q.shape)} k {tuple(k.shape)}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if need_lse and lse is None:
        lse = torch.empty((h, nq), dtype=torch.float32, device=q.device)
    _check("pe_packed_attention_fwd_noalloc",
           lib.pe_packed_attention_fwd_noalloc(
               _dtype_code(q.dtype), b, n, h, d, int(max_seq_len), _ptr(q), _ptr(k), _ptr(v),
               _ptr(cu_seqlens), scale, int(bool(query_is_first_token)), _ptr(out), _ptr(lse),
               _stream(q.device)))
    return out, lse


def pe_read_noalloc_status(device=None) -> int:
    """Device-side status of the last allocation-free forward on the device."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    return int(load_library().pe_read_noalloc_status(_stream(dev)))


# --------------------------------------------------------------------------- layer tail

def pe_packed_positions(cu_seqlens: torch.Tensor, num_tokens: int, out=None) -> torch.Tensor:
    """Position of every token inside its own sequence (int32 [num_tokens])."""
    lib = load_library()
    cu = _cuda(cu_seqlens, "cu_seqlens")
    if out is None:
        out = torch.empty(int(num_tokens), dtype=torch.int32, device=cu.device)
    _check("pe_packed_positions",
           lib.pe_packed_positions(_ptr(cu), int(cu.numel()) - 1, int(num_tokens), _ptr(out),
                                   _stream(cu.device)))
    return out


def pe_rope_packed(q: torch.Tensor, k: torch.Tensor | None, positions: torch.Tensor,
                   theta: float) -> None:
    """Split-half rotary embedding, in place, on q [N, Hq, D] and k [N, Hk, D]."""
    lib = load_library()
    if not (q.is_cuda and q.is_contiguous()) or (k is not None and not k.is_contiguous()):
        raise ValueError("q and k must be contiguous CUDA tensors (rotated in place)")
    positions = _cuda(positions, "positions").to(torch.int32)
    n, hq, d = q.shape
    hk = 0 if k is None else int(k.shape[1])
    _check("pe_rope_packed",
           lib.pe_rope_packed(_dtype_code(q.dtype), _ptr(q), hq, _ptr(k), hk, _ptr(positions), n,
                              d, float(theta), _stream(q.device)))


def pe_layernorm(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None = None,
                 eps: float = 1e-5, residual: torch.Tensor | None = None, out=None):
    """LayerNorm over the last dim of x [N, C]; with a residual, of h = x + residual
    (rounded to x's dtype), returning (y, h). Otherwise returns y."""
    lib = load_library()
    x = _cuda(x, "x")
    n, c = x.shape
    weight = _cuda(weight, "weight").to(x.dtype)
    bias = None if bias is None else _cuda(bias, "bias").to(x.dtype)
    residual = None if residual is None else _cuda(residual, "residual")
    y = torch.empty_like(x) if out is None else out
    h = torch.empty_like(x) if residual is not None else None
    _check("pe_layernorm",
           lib.pe_layernorm(_dtype_code(x.dtype), _ptr(x), _ptr(residual), _ptr(weight),
                            _ptr(bias), n, c, float(eps), _ptr(y), _ptr(h), _stream(x.device)))
    return (y, h) if residual is not None else y


def pe_geglu(x: torch.Tensor, out=None) -> torch.Tensor:
    """gelu(x[:, :F]) * x[:, F:] for x [N, 2F] (exact GELU)."""
    lib = load_library()
    x = _cuda(x, "x")
    n, f2 = x.shape
    y = torch.empty((n, f2 // 2), dtype=x.dtype, device=x.device) if out is None else out
    _check("pe_geglu", lib.pe_geglu(_dtype_code(x.dtype), _ptr(x), n, f2 // 2, _ptr(y),
                                    _stream(x.device)))
    return y
