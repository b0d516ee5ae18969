"""The C ABI library loads and exports every symbol include/pe.h declares;
host-side argument checks answer without a GPU (no compute is launched)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from padding_free_packed_gb300 import binding
    from padding_free_packed_gb300 import build
    if build.is_stale():
        build.build()
    return binding.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("pe_pack_sequences", "pe_gather_packed", "pe_scatter_padded",
                 "pe_packed_attention_fwd", "pe_packed_attention_bwd"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from padding_free_packed_gb300 import binding
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(binding.EXPORTED) <= set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.pe_abi_version() == 3
    for code in range(8):
        assert lib.pe_status_string(code)
    assert lib.pe_status_string(0) == b"ok"


def test_workspace_sizes(lib):
    fwd = lib.pe_attention_workspace_size(0, 320, 32299, 12, 64, 8192, 0, 0)
    bwd = lib.pe_attention_workspace_size(0, 320, 32299, 12, 64, 8192, 0, 1)
    assert fwd >= 16 and bwd >= fwd + 12 * 32299 * 4
    assert lib.pe_attention_workspace_size(0, -1, 0, 1, 64, 1, 0, 0) == 0
    assert lib.pe_pack_workspace_size(10) >= 16


def _fwd(lib, **kw):
    args = dict(dtype=0, B=2, N=10, H=2, D=64, S=8, q=16, k=16, v=16, cu=16, scale=0.125,
                first=0, out=16, lse=None, ws=16, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.pe_packed_attention_fwd(args["dtype"], args["B"], args["N"], args["H"], args["D"],
                                       args["S"], args["q"], args["k"], args["v"], args["cu"],
                                       args["scale"], args["first"], args["out"], args["lse"],
                                       args["ws"], args["ws_bytes"], args["stream"])


def test_host_checks_reject_bad_arguments(lib):
    # Fake, never-dereferenced addresses: every case fails in the host checks.
    assert _fwd(lib, scale=-1.0) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, scale=float("inf")) == 1
    assert _fwd(lib, D=12) == 4
    assert _fwd(lib, D=136) == 4
    assert _fwd(lib, dtype=7) == 1
    assert _fwd(lib, N=1 << 31) == 3
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, q=24) == 4       # not 16-byte aligned
    assert _fwd(lib, ws_bytes=8) == 5
    assert _fwd(lib, ws=None) == 5
    assert _fwd(lib, H=0) == 1
    assert _fwd(lib, B=0, N=5) == 1   # tokens without sequences
    n = ctypes.c_int64(0)
    assert lib.pe_pack_sequences(16, -1, 4, 16, 16, ctypes.byref(n), 16, 64, None) == 1
    assert lib.pe_pack_sequences(16, 3, 0, 16, 16, ctypes.byref(n), 16, 64, None) == 1
    assert lib.pe_pack_sequences(16, 3, 4, 16, 16, ctypes.byref(n), None, 64, None) == 5
    assert lib.pe_gather_packed(16, 16, 0, 16, 16, None) == 0   # nothing to move
    assert lib.pe_gather_packed(16, 16, -1, 16, 16, None) == 1
    assert lib.pe_scatter_padded(16, 16, 0, 4, 16, 16, None) == 0


def test_host_copies_check_lengths_before_any_copy(lib):
    """pe_upload_packed and pe_download_padded read the host lengths and reject
    bad ones before enqueuing anything (fake, never-used device addresses)."""
    bad = (ctypes.c_int32 * 2)(5, 4)     # 5 > max_seq_len 4
    zero = (ctypes.c_int32 * 2)(0, 4)
    for fn in (lib.pe_upload_packed, lib.pe_download_padded):
        assert fn(16, bad, 2, 4, 32, 16, None) == 2
        assert fn(16, zero, 2, 4, 32, 16, None) == 2
        assert fn(16, bad, -1, 4, 32, 16, None) == 1
        assert fn(16, bad, 2, 0, 32, 16, None) == 1
        assert fn(16, bad, 2, 4, 0, 16, None) == 1
        assert fn(16, None, 2, 4, 32, 16, None) == 1
        assert fn(16, bad, 0, 4, 32, 16, None) == 0   # nothing to move


def test_wait_limit_round_trip(lib):
    """pe_set_wait_limit_ns returns the previous limit; 0 restores the 2 s default."""
    first = lib.pe_set_wait_limit_ns(5000)
    try:
        assert first == 2_000_000_000
        assert lib.pe_set_wait_limit_ns(0) == 5000
        assert lib.pe_set_wait_limit_ns(0) == 2_000_000_000
    finally:
        lib.pe_set_wait_limit_ns(0)


@pytest.mark.parametrize("call", ["upload", "download"])
def test_host_copy_bindings_check_the_device_buffer_first(lib, call):
    """The bindings of the per-sequence host copies refuse a device buffer that
    does not hold exactly sum(L) rows of the grid's row shape and dtype before
    any copy is enqueued (the buffers here are host tensors: the size check
    comes first, so nothing reaches the library)."""
    import torch
    from padding_free_packed_gb300 import binding
    grid = torch.zeros(3, 8, 2, 4)
    lengths = [8, 1, 5]
    for wrong in (torch.zeros(13, 2, 4), torch.zeros(15, 2, 4),
                  torch.zeros(14, 2, 4, dtype=torch.float64), torch.zeros(14, 4, 2).transpose(1, 2)):
        with pytest.raises(ValueError, match="sum\\(L\\) rows"):
            if call == "upload":
                binding.pe_upload_packed(grid, lengths, wrong)
            else:
                binding.pe_download_padded(wrong, lengths, grid)


def test_no_gpu_means_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib) == 4


def _round16(x):
    return (x + 15) // 16 * 16


def _plan_bytes(b):
    return 32 + 2 * _round16(4 * b)


def _stream_partials(n, h, d):
    chunk = 64
    while -(-n // chunk) > 16384:
        chunk *= 2
    return _round16(-(-n // chunk) * 2 * h * (d + 2) * 4)


def _split_partials(b, h, d, s):
    ns = 1 if s <= 1024 else -(-s // 1024)
    return 0 if ns == 1 else _round16(b * h * ns * (d + 2) * 4)


@pytest.mark.parametrize("dtype,b,n,h,d,s,streaming", [
    (0, 32, 169151, 16, 64, 8192, True),     # long documents: 2 KiB bf16 rows
    (0, 600, 2_000_000, 4, 64, 8192, True),  # past 16384 chunks of 64: chunk 128
    (1, 1024, 90487, 8, 64, 256, True),      # graph workload: 2 KiB fp32 rows
    (0, 320, 32299, 12, 64, 8192, True),     # contrastive: 1.5 KiB rows
    (0, 10, 40000, 3, 64, 5000, False),      # 384-byte rows: per-(sequence, head) split
    (0, 10, 40000, 16, 96, 5000, False),     # head_dim 96: per-(sequence, head) split
    (1, 8, 91, 2, 8, 32, False),             # tiny rows, short sequences: no partials
])
def test_first_token_workspace_holds_the_partial_states(lib, dtype, b, n, h, d, s, streaming):
    """First-token forwards report room for partial softmax states: equal token
    chunks (>= 64 tokens, at most 16384 of them) with two states of H*(d+2)
    fp32 each when a token row is 1..8 x 512 bytes and head_dim is 32, 64 or
    128; otherwise 1024-key chunks per (sequence, head) when max_seq_len > 1024."""
    got = lib.pe_attention_workspace_size(dtype, b, n, h, d, s, 1, 0)
    extra = _stream_partials(n, h, d) if streaming else _split_partials(b, h, d, s)
    assert got == _plan_bytes(b) + extra
    # Without the first-token flag only the plan is needed.
    assert lib.pe_attention_workspace_size(dtype, b, n, h, d, s, 0, 0) == _plan_bytes(b)


def _bwd_stream_sums(n, h, d):
    chunk = 64
    while -(-n // chunk) > 16384:
        chunk *= 2
    return _round16(-(-n // chunk) * 2 * h * d * 4)


@pytest.mark.parametrize("dtype,b,n,h,d,s,streaming", [
    (0, 32, 169151, 16, 64, 8192, True),     # long documents: 2 KiB bf16 rows
    (0, 32, 169151, 24, 64, 8192, True),     # 3 KiB bf16 rows: the widest bf16 rows streamed
    (0, 32, 169151, 16, 128, 8192, False),   # 4 KiB bf16 rows: CUDA-core backward
    (1, 1024, 90487, 8, 64, 256, True),      # graph workload: 2 KiB fp32 rows
    (1, 1024, 90487, 16, 64, 256, True),     # 4 KiB fp32 rows
    (1, 1024, 90487, 20, 64, 256, False),    # 5 KiB fp32 rows: too wide
    (0, 600, 2_000_000, 4, 64, 8192, True),  # past 16384 chunks of 64: chunk 128
    (0, 10, 40000, 3, 64, 5000, False),      # 384-byte rows
    (0, 10, 40000, 16, 96, 5000, False),     # head_dim 96
])
def test_first_token_backward_workspace_holds_the_chunk_sums(lib, dtype, b, n, h, d, s,
                                                              streaming):
    """First-token backwards need the plan and Delta [H, B] fp32; the streaming
    form adds per-chunk dq sums (two H*d fp32 slots per token chunk) when a
    token row is 512-byte loads up to 3 KiB in bf16 or 4 KiB in fp32 and
    head_dim is 32, 64 or 128."""
    got = lib.pe_attention_workspace_size(dtype, b, n, h, d, s, 1, 1)
    base = _plan_bytes(b) + _round16(4 * h * b)
    assert got == base + (_bwd_stream_sums(n, h, d) if streaming else 0)


def test_kernel_families(lib):
    """The kernel family each (dtype, head_dim, mode, direction) runs."""
    lib.pe_attention_kernel.restype = ctypes.c_char_p
    fam = lambda *a: lib.pe_attention_kernel(*a).decode()
    assert fam(0, 64, 0, 0) == "tcgen05_bf16_d64"
    assert fam(0, 128, 0, 0) == "tcgen05_bf16_d128"
    assert fam(1, 64, 0, 0) == "tcgen05_f32_d64"
    assert fam(1, 32, 0, 0) == "simt_ffma"
    assert fam(0, 64, 1, 0) == "first_token_gemv"
    assert fam(0, 64, 0, 1) == "tcgen05_bf16_d64_bwd"
    assert fam(0, 128, 0, 1) == "tcgen05_bf16_d128_bwd"
    assert fam(1, 64, 0, 1) == "simt_ffma_bwd"
    assert fam(0, 64, 1, 1) == "first_token_bwd"
    assert fam(1, 128, 1, 1) == "first_token_bwd"
    assert fam(0, 96, 1, 1) == "simt_ffma_bwd"
    assert fam(0, 12, 0, 0) == "unsupported"


def test_kernel_families_with_a_window(lib):
    """Local calls: only the full-query forward changes family, and only off
    bf16 head_dim 64; a window reaching every key is full attention."""
    lib.pe_attention_kernel_local.restype = ctypes.c_char_p
    fam = lambda *a: lib.pe_attention_kernel_local(*a).decode()
    # (dtype, head_dim, max_seq_len, left, right, first_token, backward)
    assert fam(0, 64, 8192, 64, 64, 0, 0) == "tcgen05_bf16_d64"
    assert fam(0, 128, 8192, 64, 64, 0, 0) == "simt_ffma"
    assert fam(1, 64, 8192, 64, 64, 0, 0) == "simt_ffma"
    assert fam(1, 64, 8192, -1, -1, 0, 0) == "tcgen05_f32_d64"
    assert fam(0, 128, 100, 99, 200, 0, 0) == "tcgen05_bf16_d128"   # reaches every key
    assert fam(0, 128, 100, 98, -1, 0, 0) == "simt_ffma"
    assert fam(0, 64, 8192, 64, 64, 0, 1) == "tcgen05_bf16_d64_bwd"
    assert fam(0, 128, 8192, 64, 64, 0, 1) == "tcgen05_bf16_d128_bwd"
    assert fam(1, 64, 8192, 64, 64, 0, 1) == "simt_ffma_bwd"
    assert fam(1, 64, 8192, 64, 64, 1, 0) == "first_token_gemv"
    assert fam(0, 64, 8192, 0, 64, 1, 1) == "first_token_bwd"
    assert fam(0, 12, 8192, 64, 64, 0, 0) == "unsupported"
    assert fam(0, 64, 0, 64, 64, 0, 0) == "unsupported"


C_CALLER = r"""
#include <stdio.h>
#include "pe.h"

int main(void) {
  int code;
  printf("abi %d\n", pe_abi_version());
  for (code = 0; code <= 7; ++code) printf("status %d %s\n", code, pe_status_string(code));
  printf("ws %lu\n", (unsigned long)pe_attention_workspace_size(PE_BF16, 3, 6, 2, 64, 3, 0, 1));
  printf("family %s\n", pe_attention_kernel(PE_BF16, 64, 0, 0));
  printf("local %s\n", pe_attention_kernel_local(PE_FP32, 64, 8192, 64, 64, 0, 0));
  return 0;
}
"""


def test_header_is_plain_c_and_links_from_c(lib, tmp_path):
    """A C99 program (gcc, -Wall -Wextra -pedantic -Werror) includes the header,
    links the library and calls its host-only entry points; what it prints
    matches the same calls made through ctypes."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    from padding_free_packed_gb300 import binding
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(binding.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lpe", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    lines = out.splitlines()
    assert lines[0] == f"abi {lib.pe_abi_version()}"
    lib.pe_status_string.restype = ctypes.c_char_p
    for code in range(8):
        assert lines[1 + code] == f"status {code} {lib.pe_status_string(code).decode()}"
    assert lines[9] == f"ws {lib.pe_attention_workspace_size(0, 3, 6, 2, 64, 3, 0, 1)}"
    assert lines[10] == "family tcgen05_bf16_d64"
    assert lines[11] == "local simt_ffma"
