"""The allocation-free forward entry point against the regular one.

pe_packed_attention_fwd_noalloc serves callers that cannot hand the library a
workspace (a runtime that owns all device memory through its own pool, or a
loop that cannot afford cudaMalloc's implicit synchronisation): its scratch is
a fixed device array inside libpe. This test calls it through the C ABI twice
in a row (so the second call starts from the first call's leftover scratch)
and compares each result with pe_packed_attention_fwd's, within the parity
tolerance the other GPU tests use, and reads the device status of each call
with pe_read_noalloc_status (the status word sits in the library's array,
where the caller cannot address it). One first-token case is large enough
that its partial softmax states do not fit in the array, so the call takes
the documented fallback (one CTA per sequence and head). It lives in its own
file, collected last, and needs nothing that other tests set up.
"""

import ctypes

import numpy as np
import pytest
import torch

import padding_free_packed_gb300 as pe
from padding_free_packed_gb300 import workloads
from parity import check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _noalloc():
    lib = pe.load_library()
    fn = lib.pe_packed_attention_fwd_noalloc
    c = ctypes
    fn.argtypes = [c.c_int, c.c_int32, c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_void_p,
                   c.c_void_p, c.c_void_p, c.c_void_p, c.c_float, c.c_int, c.c_void_p,
                   c.c_void_p, c.c_void_p]
    fn.restype = c.c_int
    return fn


def _status(stream):
    lib = pe.load_library()
    lib.pe_read_noalloc_status.argtypes = [ctypes.c_void_p]
    lib.pe_read_noalloc_status.restype = ctypes.c_int
    return lib.pe_read_noalloc_status(stream)


SHORT = [300, 1, 129, 1000, 64, 257]
# 24 sequences of ~1k tokens with 16 heads x 64: the streaming first-token
# kernel's partial states (two per 64-token chunk, 16 x 66 fp32 each) need
# ~4.4 MiB, more than the 512 KiB array holds.
LONG = [1024 + 37 * i for i in range(24)]


@pytest.mark.parametrize("dtype,d,heads,first_token,lengths",
                         [(torch.bfloat16, 64, 4, False, SHORT),
                          (torch.float32, 64, 4, False, SHORT),
                          (torch.bfloat16, 64, 4, True, SHORT),
                          (torch.bfloat16, 64, 16, True, LONG)])
def test_noalloc_matches_regular_forward_on_two_calls(dtype, d, heads, first_token, lengths):
    fn = _noalloc()
    x = workloads.make_custom(lengths, heads, d, dtype, seed=41)
    s = max(lengths)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).to(DEV)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    if first_token:
        q = q[cu[:-1].long()].contiguous()
    ref, ref_lse = pe.pe_packed_attention_fwd(q, k, v, cu, s, 0.125,
                                              query_is_first_token=first_token, need_lse=True)
    code = pe.binding.PE_BF16 if dtype == torch.bfloat16 else pe.binding.PE_FP32
    tag = "bf16" if dtype == torch.bfloat16 else "fp32"
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = fn(code, len(lengths), k.shape[0], heads, d, s, q.data_ptr(), k.data_ptr(),
                v.data_ptr(), cu.data_ptr(), 0.125, int(first_token), out.data_ptr(),
                lse.data_ptr(), stream)
        assert rc == 0, f"call {call}: status {rc}"
        assert _status(stream) == 0, f"call {call}: device status"
        torch.cuda.synchronize()
        check(out, ref, tag, f"no-alloc call {call}")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=0, atol=1e-4)


def test_noalloc_rejects_batches_beyond_its_scratch():
    fn = _noalloc()
    # Fails in the size check, before any pointer is used or anything launched.
    rc = fn(pe.binding.PE_BF16, 65537, 65537, 1, 64, 1, 16, 16, 16, 16, 0.125, 0, 16, None, None)
    assert rc == 5  # PE_ERR_WORKSPACE
