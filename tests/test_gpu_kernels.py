"""Kernel-level GPU parity through the C ABI: attention against the oracle's attention."""
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
def test_attention_matches_oracle(case):
    import self_speculative_decoding_layer_gb300 as ssd

    lib = ssd.load_library()
    c = make_case(case)
    a, keep, out = device_args(c)
    nbytes = lib.ssd_attention_scratch_bytes(c["rows"], c["hq"], c["hkv"], c["hd"])
    assert nbytes > 0
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
    ptr = (scratch.data_ptr() + 255) // 256 * 256
    s = torch.cuda.current_stream()
    for _ in range(2):  # the merge counters re-arm themselves between calls
        assert lib.ssd_attention(ctypes.byref(a), ptr, nbytes, s.cuda_stream) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.max(np.abs(got - c["want"])) < ATTN_TOL


def test_attention_rejects_bad_arguments():
    import self_speculative_decoding_layer_gb300 as ssd

    lib = ssd.load_library()
    c = make_case(CASES[0])
    a, keep, out = device_args(c)
    scratch = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    ptr = (scratch.data_ptr() + 255) // 256 * 256
    s = torch.cuda.current_stream().cuda_stream
    bad = ssd.AttentionArgsC.from_buffer_copy(a)
    bad.head_dim = 96
    assert lib.ssd_attention(ctypes.byref(bad), ptr, 1 << 23, s) == 1
    bad = ssd.AttentionArgsC.from_buffer_copy(a)
    bad.rows = 65
    assert lib.ssd_attention(ctypes.byref(bad), ptr, 1 << 23, s) == 1
    bad = ssd.AttentionArgsC.from_buffer_copy(a)
    bad.prefix = bad.n_pages * 64 + 1
    assert lib.ssd_attention(ctypes.byref(bad), ptr, 1 << 23, s) == 1
    assert lib.ssd_attention(ctypes.byref(a), ptr, 16, s) == 3
