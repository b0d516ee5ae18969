"""Packed rows (several documents per padded row) on the GPU against the
oracle: indexed packing masks and flatten_packed_sequence_metadata (page
"nemo_automodel.components.models.common.packing"), bit-exact, plus the
attention over the documents they describe."""

import math

import numpy as np
import pytest
import torch

import oracle
import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check
from rows_data import packed_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def test_page_example_row(golden):
    g = golden("indexed_packing_mask_example.txt")
    flat, cu, n = pe.pe_pack_document_ids(_dev(np.array([g["row"]], np.int32)))
    assert flat.cpu().tolist() == g["flat_index"] and cu.cpu().tolist() == g["cu_seqlens"]
    flat, cu, n = pe.pe_flatten_packed_metadata(_dev(np.array([g["row_token_indices"]])),
                                                _dev(np.array([g["row_cu_seqlens"]], np.int32)))
    assert flat.cpu().tolist() == g["flat_index"] and cu.cpu().tolist() == g["cu_seqlens"]


@pytest.mark.parametrize("seed,b,s,max_docs,max_doc_len", [
    (0, 6, 40, 5, 12), (1, 1, 9, 3, 4), (2, 64, 16384, 12, 3000), (3, 3000, 64, 4, 30),
    (4, 2049, 7, 7, 1), (5, 17, 1000, 40, 60),
])
@pytest.mark.parametrize("sparse", [False, True])
def test_packed_rows_match_oracle(seed, b, s, max_docs, max_doc_len, sparse):
    ids, tok, rcu = packed_rows(seed, b, s, max_docs, max_doc_len, sparse)
    if not sparse:
        ref_flat, ref_cu = oracle.pack_document_ids(ids)
        flat, cu, n = pe.pe_pack_document_ids(_dev(ids))
        assert n == ref_flat.size
        assert np.array_equal(flat.cpu().numpy(), ref_flat)
        assert np.array_equal(cu.cpu().numpy(), ref_cu)
    ref_flat, ref_cu = oracle.flatten_packed_metadata(tok, rcu, s)
    flat, cu, n = pe.pe_flatten_packed_metadata(_dev(tok), _dev(rcu))
    assert n == ref_flat.size
    assert np.array_equal(flat.cpu().numpy(), ref_flat)
    assert np.array_equal(cu.cpu().numpy(), ref_cu)


def test_empty_rows_and_batch():
    flat, cu, n = pe.pe_pack_document_ids(torch.zeros((5, 8), dtype=torch.int32, device=DEV))
    assert n == 0 and cu.cpu().tolist() == [0]
    flat, cu, n = pe.pe_pack_document_ids(torch.zeros((0, 8), dtype=torch.int32, device=DEV))
    assert n == 0 and cu.cpu().tolist() == [0]
    flat, cu, n = pe.pe_flatten_packed_metadata(
        torch.full((2, 3), -1, dtype=torch.int64, device=DEV),
        torch.tensor([[0, -1], [0, -1]], dtype=torch.int32, device=DEV))
    assert n == 0 and cu.cpu().tolist() == [0]


@pytest.mark.parametrize("row", [[1, 1, 3, 0], [1, 0, 1, 0], [2, 2, 0, 0], [1, 2, 1, 0],
                                 [1, -1, 0, 0], [0, 1, 1, 0]])
def test_malformed_masks_are_rejected(row):
    rows = np.array([[1, 1, 0, 0], row, [1, 2, 2, 2]], np.int32)  # the bad row among good ones
    with pytest.raises(pe.PackedAttentionError) as err:
        pe.pe_pack_document_ids(_dev(rows))
    assert err.value.status == 1          # PE_ERR_INVALID_ARG


@pytest.mark.parametrize("tok,rcu", [
    ([0, 1, 2, -1], [1, 3, -1]), ([0, 1, 2, -1], [0, 2, 2, 3]), ([0, 1, 2, -1], [0, 2, -1, -1]),
    ([0, 1, 2, -1], [0, 3, 4, -1]), ([0, -1, 2, -1], [0, 2, -1, -1]),
    ([0, 1, 2, -1], [0, -1, 3, -1]), ([0, 1, 4, -1], [0, 3, -1, -1]),
])
def test_inconsistent_row_layouts_are_rejected(tok, rcu):
    width = max(len(rcu), 4)
    t = np.array([[0, 1, -1, -1], tok], np.int64)
    r = np.full((2, width), -1, np.int32)
    r[0, :3] = [0, 2, -1]
    r[1, :len(rcu)] = rcu
    with pytest.raises(pe.PackedAttentionError) as err:
        pe.pe_flatten_packed_metadata(_dev(t), _dev(r))
    assert err.value.status == 1


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_attention_over_packed_rows(dtype):
    """Rows of consecutive documents: mask -> flat_index / cu_seqlens -> gather
    -> attention, against the oracle run on the oracle's own conversion."""
    ids, _, _ = packed_rows(7, b=5, s=1024, max_docs=6, max_doc_len=400)
    b, s = ids.shape
    h, d = 4, 64
    rng = np.random.default_rng(8)
    grids = [torch.from_numpy(rng.standard_normal((b, s, h, d)).astype(np.float32)).to(dtype)
             for _ in range(3)]
    flat, cu, n = pe.pe_pack_document_ids(_dev(ids))
    q, k, v = (pe.pe_gather_packed(g.to(DEV), flat, n) for g in grids)
    max_len = int((cu[1:] - cu[:-1]).max())
    out, lse = pe.pe_packed_attention_fwd(q, k, v, cu, max_len, 1 / math.sqrt(d), need_lse=True)
    ref_flat, ref_cu = oracle.pack_document_ids(ids)
    rq, rk, rv = (oracle.gather_rows(g.float().numpy().reshape(b * s, h, d), ref_flat)
                  for g in grids)
    ref, ref_lse = oracle.attention_fwd(rq, rk, rv, ref_cu, max_len, 1 / math.sqrt(d))
    check(out, ref, "fp32" if dtype == torch.float32 else "bf16", "attention over packed rows")
