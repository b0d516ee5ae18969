"""pack_sequences, gather and scatter on the GPU: bit-exact against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pack(lengths, s):
    return pe.pe_pack_sequences(torch.as_tensor(np.asarray(lengths, np.int32), device=DEV), s)


def test_worked_example(golden):
    g = golden("pack_worked_example.txt")
    flat, cu, n = _pack(g["lengths"], g["max_seq_len"][0])
    assert flat.cpu().tolist() == g["flat_index"]
    assert cu.cpu().tolist() == g["cu_seqlens"]
    assert n == g["num_tokens"][0]
    g2 = golden("pack_cu_seqlens_example.txt")
    _, cu2, n2 = _pack(g2["lengths"], g2["max_seq_len"][0])
    assert cu2.cpu().tolist() == g2["cu_seqlens"] and n2 == g2["num_tokens"][0]


@pytest.mark.parametrize("seed", range(8))
def test_random_lengths_bit_exact(seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 3000))
    s = int(rng.integers(1, 700))
    lengths = rng.integers(1, s + 1, b).astype(np.int32)
    flat, cu, n = _pack(lengths, s)
    o_flat, o_cu, o_n = oracle.pack_sequences(lengths, s)
    assert n == o_n
    assert np.array_equal(flat.cpu().numpy(), o_flat)
    assert np.array_equal(cu.cpu().numpy(), o_cu)
    assert cu.dtype == torch.int32 and flat.dtype == torch.int64


@pytest.mark.parametrize("name", ["tiny_fp32", "graph_fp32", "contrastive_bf16", "longdoc_bf16"])
def test_workload_lengths_bit_exact(name):
    wl = workloads.WORKLOADS[name]
    lengths = workloads.draw_lengths(name, np.random.default_rng(0))
    flat, cu, n = _pack(lengths, wl.max_seq_len)
    o_flat, o_cu, o_n = oracle.pack_sequences(lengths, wl.max_seq_len)
    assert n == o_n and np.array_equal(flat.cpu().numpy(), o_flat)
    assert np.array_equal(cu.cpu().numpy(), o_cu)


def test_edge_cases():
    flat, cu, n = _pack(np.zeros(0, np.int32), 5)
    assert n == 0 and cu.cpu().tolist() == [0] and flat.numel() == 0
    for lengths, s in (([1] * 700, 3), ([9] * 33, 9), ([1], 1), ([4096], 4096),
                       (list(range(1, 2500)), 2500)):
        flat, cu, n = _pack(lengths, s)
        o_flat, o_cu, o_n = oracle.pack_sequences(lengths, s)
        assert n == o_n and np.array_equal(flat.cpu().numpy(), o_flat)
        assert np.array_equal(cu.cpu().numpy(), o_cu)


def test_bad_lengths_are_reported():
    for lengths, s in (([3, 0, 2], 4), ([3, 5], 4), ([-2, 1], 4), ([1] * 2000 + [0], 4)):
        with pytest.raises(pe.PackedAttentionError) as e:
            _pack(lengths, s)
        assert e.value.status == 2
    # Token count beyond int32: the fill kernel is skipped, the status says why.
    big = 1 << 30
    with pytest.raises(pe.PackedAttentionError) as e:
        _pack([big, big], big)
    assert e.value.status == 3


@pytest.mark.parametrize("row_shape,dtype", [((16, 64), torch.bfloat16), ((8, 64), torch.float32),
                                             ((3,), torch.float32), ((5,), torch.uint8),
                                             ((2, 8), torch.float32)])
def test_gather_scatter_bit_exact(row_shape, dtype):
    rng = np.random.default_rng(11)
    b, s = 37, 50
    lengths = rng.integers(1, s + 1, b).astype(np.int32)
    flat, cu, n = _pack(lengths, s)
    o_flat, o_cu, _ = oracle.pack_sequences(lengths, s)
    grid = torch.randint(0, 255, (b, s) + row_shape, dtype=torch.uint8) if dtype == torch.uint8 \
        else torch.randn((b, s) + row_shape).to(dtype)
    packed = pe.pe_gather_packed(grid.to(DEV), flat, n)
    want = oracle.gather_rows(grid.view(torch.uint8).reshape(b * s, -1).numpy(), o_flat)
    assert np.array_equal(packed.cpu().view(torch.uint8).reshape(n, -1).numpy(), want)
    back = pe.pe_scatter_padded(packed, cu, s)
    want_grid = oracle.scatter_rows(packed.cpu().view(torch.uint8).reshape(n, -1).numpy(), o_cu, s)
    assert np.array_equal(back.cpu().view(torch.uint8).reshape(b, s, -1).numpy(), want_grid)


def test_gather_misaligned_pointers_use_narrow_path():
    rng = np.random.default_rng(12)
    lengths = rng.integers(1, 20, 9).astype(np.int32)
    flat, cu, n = _pack(lengths, 20)
    o_flat, _, _ = oracle.pack_sequences(lengths, 20)
    base = torch.randint(0, 255, (9 * 20 * 32 + 3,), dtype=torch.uint8, device=DEV)
    padded = base[3:].view(9, 20, 32)  # 3 bytes past a 16-byte boundary
    packed = pe.pe_gather_packed(padded, flat, n)
    want = oracle.gather_rows(padded.cpu().reshape(180, 32).numpy(), o_flat)
    assert np.array_equal(packed.cpu().numpy(), want)


def test_longdoc_gather_and_scatter_full_size():
    lengths, gq, _, _ = workloads.make_padded_inputs("longdoc_bf16")
    wl = workloads.WORKLOADS["longdoc_bf16"]
    flat, cu, n = _pack(lengths, wl.max_seq_len)
    o_flat, o_cu, _ = oracle.pack_sequences(lengths, wl.max_seq_len)
    packed = pe.pe_gather_packed(gq.to(DEV), flat, n)
    want = oracle.gather_rows(gq.view(torch.uint8).reshape(len(lengths) * wl.max_seq_len, -1)
                              .numpy(), o_flat)
    assert np.array_equal(packed.cpu().view(torch.uint8).reshape(n, -1).numpy(), want)
    back = pe.pe_scatter_padded(packed, cu, wl.max_seq_len)
    want_grid = oracle.scatter_rows(want, o_cu, wl.max_seq_len)
    assert np.array_equal(back.cpu().view(torch.uint8).reshape(len(lengths), wl.max_seq_len, -1)
                          .numpy(), want_grid)


@pytest.mark.parametrize("dtype,row", [(torch.bfloat16, (4, 64)), (torch.float32, (3, 5))])
def test_host_grids_upload_gather_and_scatter(dtype, row):
    """Host-resident padded grids: pe_upload_packed (copy engines, one copy per
    sequence) and pe_gather_packed on pinned host memory both give the device
    gather's packed buffer bit for bit; pe_scatter_padded into pinned host
    memory gives the device scatter's grid."""
    lengths = np.array([1, 77, 128, 5, 300, 2], np.int32)
    s = 300
    rng = np.random.default_rng(11)
    grid = torch.from_numpy(rng.standard_normal((len(lengths), s) + row).astype(np.float32))
    grid = grid.to(dtype).pin_memory()
    flat, cu, n = pe.pe_pack_sequences(torch.from_numpy(lengths).to(DEV), s)
    want = pe.pe_gather_packed(grid.to(DEV), flat, n)
    up = torch.empty_like(want)
    pe.pe_upload_packed(grid, lengths, out=up)
    torch.cuda.synchronize()
    assert torch.equal(up, want)
    assert torch.equal(pe.pe_gather_packed(grid, flat, n), want)
    host = torch.empty_like(grid).pin_memory()
    pe.pe_scatter_padded(want, cu, s, out=host)
    torch.cuda.synchronize()
    assert torch.equal(host, pe.pe_scatter_padded(want, cu, s).cpu())


def test_upload_rejects_bad_lengths():
    grid = torch.zeros((2, 4, 8), dtype=torch.float32).pin_memory()
    # (out holds sum(L) rows, so the binding's size check passes and the
    # library's length check answers.)
    with pytest.raises(pe.PackedAttentionError):
        pe.pe_upload_packed(grid, [5, 4], out=torch.empty((9, 8), device=DEV))  # 5 > max_seq_len
    with pytest.raises(pe.PackedAttentionError):
        pe.pe_upload_packed(grid, [0, 4], out=torch.empty((4, 8), device=DEV))


@pytest.mark.parametrize("dtype,row", [(torch.bfloat16, (4, 64)), (torch.float32, (3, 5))])
@pytest.mark.parametrize("pinned", [True, False])
def test_download_padded_writes_the_real_rows(dtype, row, pinned):
    """pe_download_padded (copy engines, one copy per sequence) puts the packed
    rows where the device scatter puts them, bit for bit, and leaves the pad
    rows of the host grid as the caller filled them (zero, for
    to_dense_batch's fill; a sentinel here, to see that they are untouched)."""
    lengths = np.array([1, 77, 128, 5, 300, 2], np.int32)
    s = 300
    rng = np.random.default_rng(12)
    n = int(lengths.sum())
    packed = torch.from_numpy(rng.standard_normal((n,) + row).astype(np.float32)).to(dtype)
    packed = packed.to(DEV)
    _, cu, _ = pe.pe_pack_sequences(torch.from_numpy(lengths).to(DEV), s)
    want = pe.pe_scatter_padded(packed, cu, s).cpu()
    host = torch.full((len(lengths), s) + row, 7.0, dtype=dtype)
    if pinned:
        host = host.pin_memory()
    pe.pe_download_padded(packed, lengths, out_host=host)
    torch.cuda.synchronize()
    real = torch.from_numpy(np.arange(s)[None, :] < lengths[:, None])
    assert torch.equal(host[real], want[real])
    assert bool((host[~real] == 7.0).all())


def test_download_rejects_bad_lengths():
    """Lengths outside [1, max_seq_len] are refused before any copy (the packed
    buffer holds sum(L) rows, so the binding's own size check passes)."""
    host = torch.zeros((2, 4, 8), dtype=torch.float32).pin_memory()
    with pytest.raises(pe.PackedAttentionError):
        pe.pe_download_padded(torch.zeros((9, 8), device=DEV), [5, 4], out_host=host)  # 5 > 4
    with pytest.raises(pe.PackedAttentionError):
        pe.pe_download_padded(torch.zeros((4, 8), device=DEV), [0, 4], out_host=host)
