"""ssd_attention_noalloc against ssd_attention.

The allocation-free entry point serves callers that may not allocate device
memory; it keeps its scratch in a static device array shared by every call.
Two calls in a row check that what the array keeps from one call (the row
descriptor) does not leak into the next.  Collected last so
a stop-at-first-failure run has already run everything else.
"""
import ctypes

import numpy as np
import pytest

from attn_cases import ATTN_TOL, CASES, device_args, make_case

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_existing_entry_point(case):
    import self_speculative_decoding_layer_gb300 as ssd

    lib = ssd.load_library()
    lib.ssd_attention_noalloc.argtypes = [ctypes.POINTER(ssd.AttentionArgsC), ctypes.c_void_p]
    lib.ssd_attention_noalloc.restype = ctypes.c_int
    c = make_case(case, seed=3)
    a, keep, out = device_args(c)
    nbytes = lib.ssd_attention_scratch_bytes(c["rows"], c["hq"], c["hkv"], c["hd"])
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
    ptr = (scratch.data_ptr() + 255) // 256 * 256
    st = torch.cuda.current_stream().cuda_stream
    assert lib.ssd_attention(ctypes.byref(a), ptr, nbytes, st) == 0
    torch.cuda.synchronize()
    ref = out.cpu().numpy().copy()
    assert np.max(np.abs(ref - c["want"])) < ATTN_TOL
    for _ in range(2):
        out.fill_(float("nan"))
        assert lib.ssd_attention_noalloc(ctypes.byref(a), st) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.max(np.abs(got - ref)) < ATTN_TOL


def test_noalloc_rejects_bad_arguments_without_launching():
    import self_speculative_decoding_layer_gb300 as ssd

    lib = ssd.load_library()
    lib.ssd_attention_noalloc.argtypes = [ctypes.POINTER(ssd.AttentionArgsC), ctypes.c_void_p]
    lib.ssd_attention_noalloc.restype = ctypes.c_int
    c = make_case(CASES[0])
    a, keep, out = device_args(c)
    st = torch.cuda.current_stream().cuda_stream
    for field, value in (("rows", 0), ("rows", 65), ("head_dim", 96), ("dtype", 3), ("n_kv_heads", 3)):
        bad = ssd.AttentionArgsC.from_buffer_copy(a)
        setattr(bad, field, value)
        assert lib.ssd_attention_noalloc(ctypes.byref(bad), st) == 1, field
    bad = ssd.AttentionArgsC.from_buffer_copy(a)
    bad.k_cache = a.k_cache + 4  # TMA needs 16-byte aligned tensors
    assert lib.ssd_attention_noalloc(ctypes.byref(bad), st) == 1
    bad = ssd.AttentionArgsC.from_buffer_copy(a)
    bad.prefix = bad.n_pages * 64 + 1  # past the block table
    assert lib.ssd_attention_noalloc(ctypes.byref(bad), st) == 1
