"""The allocation-free entry point (mla_decode_noalloc) against mla_decode.

Some callers cannot allocate device memory on the decode path (their own pool owns every
allocation, or they cannot afford cudaMalloc/cudaFree's device synchronisation); for them
mla_decode_noalloc keeps its scratch in a fixed array inside the library.  This checks,
through the C ABI and on two calls in a row (the second reuses the array the first left
behind), that it returns what mla_decode returns, within the tolerance of the parity tests.
It lives in its own file, collected last, and passes alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

from mla_attention_decode_splitkv_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from mla_attention_decode_splitkv_gb300 import _lib
    return _lib


CASES = [
    (synth.KV_FP8, [700, 1, 1500, 0], 0),       # balanced split (needs batch + SMs - 1 slots)
    (synth.KV_MXFP4, [300, 2049, 17], 3),       # uniform split with combine
    (synth.KV_BF16, [129, 64], 1),              # single split, written directly
]


@pytest.mark.parametrize("kv_dtype,lens,ns", CASES)
def test_noalloc_matches_mla_decode_on_two_calls(lib, kv_dtype, lens, ns):
    inp = synth.make_inputs(len(lens), lens, kv_dtype, seed=321).to("cuda")
    B = inp.batch
    ref = torch.empty((B, 16, 512), dtype=torch.bfloat16, device="cuda")
    rc = lib.mla_decode(inp.q, inp.kv, inp.kv_scale, inp.kv_indptr, ref, B, ns, kv_dtype)
    assert rc == lib.MLA_OK
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy()
    for call in range(2):
        out = torch.full((B, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.mla_decode_noalloc(inp.q, inp.kv, inp.kv_scale, inp.kv_indptr, out, B, ns, kv_dtype)
        assert rc == lib.MLA_OK, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert not np.isnan(got).any(), f"call {call}: output not fully written"
        np.testing.assert_allclose(got, want, atol=ATOL, rtol=RTOL, err_msg=f"call {call}")


def test_noalloc_rejects_work_beyond_its_scratch(lib):
    # 600 sequences x 2 splits needs 1200 partial slots, more than the fixed 512.
    B = 600
    q = torch.zeros((B, 16, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((B, 576), dtype=torch.uint8, device="cuda")
    sc = torch.ones(1, dtype=torch.float32, device="cuda")
    ip = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    out = torch.empty((B, 16, 512), dtype=torch.bfloat16, device="cuda")
    rc = lib.mla_decode_noalloc(q, kv, sc, ip, out, B, 2, synth.KV_FP8)
    assert rc == lib.MLA_ERR_NO_MEMORY
