"""The allocation-free entry point (mla_decode_noalloc) against mla_decode and the oracle.

Some callers cannot allocate device memory on the decode path (their own pool owns every
allocation, or they cannot afford cudaMalloc/cudaFree's device synchronisation); for them
mla_decode_noalloc keeps its scratch in a fixed array inside the library.  This checks,
through the C ABI and on two calls in a row (the second reuses the array the first left
behind), that it returns what mla_decode returns and what the CPU oracle computes, within
the tolerance of the parity tests; that a balanced-mode call needing exactly the array's
slot limit works; that calls alternating between cache encodings leave nothing behind for
each other; and that its status word reads clean.  It lives in its own file, collected
last, and passes alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_attention_decode_splitkv_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2
MAX_SLOTS = 512          # MLA_NOALLOC_MAX_SLOTS in include/mla_decode.h


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from mla_attention_decode_splitkv_gb300 import _lib
    return _lib


def _noalloc(lib, inp, ns):
    B = inp.batch
    out = torch.full((B, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.mla_decode_noalloc(inp.q, inp.kv, inp.kv_scale, inp.kv_indptr, out, B, ns, inp.kv_dtype)
    assert rc == lib.MLA_OK, f"status {rc}"
    torch.cuda.synchronize()
    assert lib.noalloc_status(clear=True) == lib.MLA_OK
    got = out.float().cpu().numpy()
    assert not np.isnan(got).any(), "output not fully written"
    return got


CASES = [
    (synth.KV_FP8, [700, 1, 1500, 0], 0),       # balanced split (needs batch + SMs - 1 slots)
    (synth.KV_MXFP4, [300, 2049, 17], 3),       # uniform split with combine
    (synth.KV_BF16, [129, 64], 1),              # single split, written directly
]


@pytest.mark.parametrize("kv_dtype,lens,ns", CASES)
def test_noalloc_matches_mla_decode_and_oracle_on_two_calls(lib, kv_dtype, lens, ns):
    host = synth.make_inputs(len(lens), lens, kv_dtype, seed=321)
    inp = host.to("cuda")
    B = inp.batch
    ref = torch.empty((B, 16, 512), dtype=torch.bfloat16, device="cuda")
    rc = lib.mla_decode(inp.q, inp.kv, inp.kv_scale, inp.kv_indptr, ref, B, ns, kv_dtype)
    assert rc == lib.MLA_OK
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy()
    exact, _ = oracle.decode(host.q, host.kv, host.kv_scale, host.kv_indptr, kv_dtype)
    for call in range(2):
        got = _noalloc(lib, inp, ns)
        np.testing.assert_allclose(got, want, atol=ATOL, rtol=RTOL, err_msg=f"call {call} vs mla_decode")
        np.testing.assert_allclose(got, exact, atol=ATOL, rtol=RTOL, err_msg=f"call {call} vs oracle")


def test_noalloc_balanced_mode_at_the_slot_limit(lib):
    """batch + SMs - 1 == MLA_NOALLOC_MAX_SLOTS: the largest balanced-mode batch the array
    holds; one more sequence is refused."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = MAX_SLOTS - sms + 1
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.choice([0, 1, 40, 130, 600], size=B)]
    host = synth.make_inputs(B, lens, synth.KV_FP8, seed=77)
    inp = host.to("cuda")
    exact, _ = oracle.decode(host.q, host.kv, host.kv_scale, host.kv_indptr, synth.KV_FP8)
    for call in range(2):
        np.testing.assert_allclose(_noalloc(lib, inp, 0), exact, atol=ATOL, rtol=RTOL, err_msg=f"call {call}")
    big = synth.make_inputs(B + 1, lens + [5], synth.KV_FP8, seed=78).to("cuda")
    out = torch.empty((B + 1, 16, 512), dtype=torch.bfloat16, device="cuda")
    rc = lib.mla_decode_noalloc(big.q, big.kv, big.kv_scale, big.kv_indptr, out, B + 1, 0, synth.KV_FP8)
    assert rc == lib.MLA_ERR_NO_MEMORY


def test_noalloc_calls_alternating_encodings(lib):
    """Consecutive calls switch cache encoding and split mode; each matches the oracle."""
    seq = [(synth.KV_MXFP4, [900, 3, 2000], 0), (synth.KV_FP8, [129, 4000], 5), (synth.KV_BF16, [1000, 1, 77], 0),
           (synth.KV_MXFP4, [64, 65], 2), (synth.KV_FP8, [3000, 0, 10, 2500], 0)]
    prepared = []
    for i, (dt, lens, ns) in enumerate(seq):
        host = synth.make_inputs(len(lens), lens, dt, seed=600 + i)
        exact, _ = oracle.decode(host.q, host.kv, host.kv_scale, host.kv_indptr, dt)
        prepared.append((host.to("cuda"), ns, exact))
    for rnd in range(2):
        for i, (inp, ns, exact) in enumerate(prepared):
            np.testing.assert_allclose(_noalloc(lib, inp, ns), exact, atol=ATOL, rtol=RTOL,
                                       err_msg=f"round {rnd} call {i}")


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
