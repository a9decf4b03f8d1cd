"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every symbol
declared in include/*.h, rejects bad arguments before touching the device, and its
split-count heuristic and workspace sizing follow their documented rules."""
import ctypes
import glob
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mla_attention_decode_splitkv_gb300 import build
    path = build.build()
    from mla_attention_decode_splitkv_gb300 import _lib
    return _lib.load(path)


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(mla_[A-Za-z0-9_]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return sorted(names)


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "mla_decode" in names and len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    from mla_attention_decode_splitkv_gb300 import _lib
    assert set(_lib.EXPORTED) == set(names)


def test_status_strings(lib):
    for code, name in [(0, b"MLA_OK"), (-1, b"MLA_ERR_INVALID_ARG"), (-2, b"MLA_ERR_UNSUPPORTED"),
                       (-3, b"MLA_ERR_CUDA"), (-4, b"MLA_ERR_NO_MEMORY"), (-5, b"MLA_ERR_TIMEOUT")]:
        assert lib.mla_status_string(code) == name
    assert lib.mla_status_string(12345) == b"MLA_UNKNOWN_STATUS"


def _call(lib, q=256, kv=512, scale=1024, ip=2048, out=4096, batch=2, ns=0, dtype=1):
    vp = ctypes.c_void_p
    return lib.mla_decode(vp(q) if q else None, vp(kv) if kv else None, vp(scale) if scale else None,
                          vp(ip) if ip else None, vp(out) if out else None, batch, ns, dtype, None)


def test_argument_checks_precede_any_device_work(lib):
    INV = -1
    assert _call(lib, q=0) == INV
    assert _call(lib, kv=0) == INV
    assert _call(lib, ip=0) == INV
    assert _call(lib, out=0) == INV
    assert _call(lib, batch=0) == INV
    assert _call(lib, batch=-3) == INV
    assert _call(lib, dtype=3) == INV
    assert _call(lib, dtype=-1) == INV
    assert _call(lib, scale=0, dtype=1) == INV          # fp8 needs its scale
    assert _call(lib, scale=0, dtype=2) == INV          # MXFP4 needs its block scales
    assert _call(lib, q=258) == INV                     # q not 16-byte aligned
    assert _call(lib, kv=520) == INV                    # kv not 16-byte aligned
    assert _call(lib, out=4100) == INV                  # out not 8-byte aligned
    assert _call(lib, ns=4097) == INV


def _call_paged(lib, q=256, kv=512, scale=1024, ip=2048, pi=3072, last=3584, ps=64, out=4096, batch=2, ns=0,
                dtype=1):
    vp = ctypes.c_void_p
    a = lambda x: vp(x) if x else None
    return lib.mla_decode_paged(a(q), a(kv), a(scale), a(ip), a(pi), a(last), ps, a(out), batch, ns, dtype, None)


def test_paged_argument_checks_precede_any_device_work(lib):
    INV = -1
    for ps in (0, 3, 6, 12, 48, 96, 256, -64):
        assert _call_paged(lib, ps=ps) == INV          # page size: a power of two in [1, 128]
    assert _call_paged(lib, pi=0) == INV
    assert _call_paged(lib, last=0) == INV
    assert _call_paged(lib, ip=0) == INV
    assert _call_paged(lib, pi=3074) == INV             # page list not 4-byte aligned
    assert _call_paged(lib, last=3586) == INV
    assert _call_paged(lib, q=258) == INV
    assert _call_paged(lib, kv=520) == INV
    assert _call_paged(lib, scale=0, dtype=2) == INV
    assert _call_paged(lib, batch=0) == INV
    assert _call_paged(lib, ns=4097) == INV
    assert _call_paged(lib, dtype=3) == INV


def _call_multi(lib, q=256, qo=128, total_q=3, kv=512, scale=1024, ip=2048, pi=3072, last=3584, ps=64, out=4096,
                batch=2, ns=0, dtype=1):
    vp = ctypes.c_void_p
    a = lambda x: vp(x) if x else None
    return lib.mla_decode_paged_multi(a(q), a(qo), total_q, a(kv), a(scale), a(ip), a(pi), a(last), ps, a(out), batch,
                                      ns, dtype, None)


def test_multi_query_argument_checks_precede_any_device_work(lib):
    INV = -1
    assert _call_multi(lib, qo=0) == INV
    assert _call_multi(lib, qo=130) == INV              # qo_indptr not 4-byte aligned
    assert _call_multi(lib, total_q=0) == INV
    assert _call_multi(lib, batch=0) == INV
    for ps in (0, 3, 48, 256):
        assert _call_multi(lib, ps=ps) == INV
    assert _call_multi(lib, pi=0) == INV
    assert _call_multi(lib, q=258) == INV
    assert _call_multi(lib, ns=4097) == INV
    assert _call_multi(lib, dtype=5) == INV


def test_valid_call_without_a_gpu_fails_cleanly(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    rc = _call(lib, scale=0, dtype=0)
    assert rc in (-2, -3)  # MLA_ERR_UNSUPPORTED or MLA_ERR_CUDA, never a crash
    for ps in (1, 2, 4, 8, 128):
        assert _call_paged(lib, ps=ps) in (-2, -3)
    assert _call_multi(lib) in (-2, -3)


ROW_BYTES = {0: 576 * 2, 1: 576, 2: 288 + 18}          # bf16, fp8, MXFP4 cache rows
PIECE_BYTES = 16 * (512 + 1) * 4                          # fp32 partial output + log-sum-exp of 16 heads
WAVE_BYTES = 222e3                                        # per-wave start-up + drain latency x one SM's HBM share
CROSS_BYTES = 300e3                                       # crossing latency x one SM's HBM share
ROW_RATE = {0: 1.0, 1: 1.0, 2: 0.30}                      # a CTA's rate through the rows / the HBM rate


def _model_splits(batch, L, sms, dtype):
    """The split model as the header states it: cache-row costs c (a piece) and x (a sequence
    crossing), time of the slowest CTA for each uniform split count and for the balanced mode."""
    row = ROW_BYTES[dtype] / ROW_RATE[dtype]
    c, w, x = PIECE_BYTES / row, WAVE_BYTES / row, CROSS_BYTES / row
    L = max(L, 1)
    best_ns, best_t = 1, None
    for ns in range(1, min(4096, -(-L // 128)) + 1):
        waves = -(-batch * ns // sms)
        chunk = -(-(-(-L // ns)) // 128) * 128
        t = waves * (chunk + w + (c if ns > 1 else 0.0)) + (ns * c if ns > 1 else 0.0)
        if best_t is None or t < best_t:
            best_ns, best_t = ns, t
    R = batch * L / sms
    s = math.ceil(R / L) + 1
    p = math.ceil(L / R) + 1
    t_bal = R + w + s * c + (s - 1) * x + p * c
    return 0 if t_bal < best_t else best_ns


def test_split_model_piece_cost_is_the_partial_bytes():
    # c in rows = one piece's bytes over one cached row's bytes
    assert PIECE_BYTES == 32832
    assert abs(PIECE_BYTES / ROW_BYTES[1] - 57.0) < 1e-9


@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_pick_splits_follows_the_documented_model(lib, dtype):
    for batch in (1, 4, 8, 32, 64, 75, 76, 77, 128, 151, 152, 153, 256, 1000):
        for L in (0, 1, 100, 127, 128, 256, 257, 1024, 2048, 2049, 4000, 4096, 8192, 65536):
            for sms in (148, 152):
                assert lib.mla_decode_pick_splits(batch, L, sms, dtype) == _model_splits(batch, L, sms, dtype), \
                    (batch, L, sms)


def test_pick_splits_reproduces_the_measured_choices(lib):
    # GB300 (152 SMs), cold calls, each shape timed at the split counts shown; the model
    # must pick the fastest (or, where two were equal, one of them):
    #   fp8  256 x 4096: balanced 123.6, ns 1 125.6, ns 2 144.0, ns 4 154.3 us
    #   fp8  256 x 8192: balanced 211.6, ns 1 219.8, ns 2 242.3, ns 4 244.4
    #   MXFP4 256 x 8192: balanced 344.7, ns 1 379.5, ns 2 402.1, ns 4 385.7
    #   fp8  64 x 8192: ns 2 72.4, balanced 82.5
    #   MXFP4 (current dequantisation, 0.30 of the HBM rate): 64 x 8192 balanced 99.0, ns 2 101.0;
    #   4 x 8192 ns 16 31.4, ns 8 37.5;  16 x 8192 ns 8 39.6, balanced 45.7, ns 16 51.9;
    #   32 x 8192 ns 4 60.1, balanced 64.2
    #   bf16 64 x 8192: balanced 139.9, ns 2 142.0
    #   fp8  152 x 8192: ns 1 129.7, balanced 131.7, ns 2 139.9
    #   fp8  16 x 8192: ns 8 = ns 9 33.4, balanced 43.7;  4 x 8192: ns 13 = ns 16 25.2, ns 32 27.3
    #   fp8  256 x 1024: ns 1 47.7, balanced 62.1;  256 x 2048: ns 1 70.3, balanced 84.6;
    #   128 x 1024: ns 1 27.3, balanced 45.7
    pick = lambda b, L, dt: lib.mla_decode_pick_splits(b, L, 152, dt)
    assert pick(256, 4096, 1) == 0
    assert pick(256, 8192, 1) == 0
    assert pick(256, 8192, 2) == 0
    assert pick(64, 8192, 1) == 2
    assert pick(64, 8192, 2) == 0
    assert pick(4, 8192, 2) == 16
    assert pick(16, 8192, 2) == 8
    assert pick(32, 8192, 2) == 4
    assert pick(64, 8192, 0) == 0
    assert pick(152, 8192, 1) == 1
    assert pick(16, 8192, 1) in (8, 9)
    assert pick(4, 8192, 1) in (13, 16)
    for L in (1024, 2048):
        assert pick(256, L, 1) == 1
    assert pick(128, 1024, 1) == 1
    assert pick(32, 1024, 1) == 4


def test_pick_splits_rejects_bad_arguments(lib):
    assert lib.mla_decode_pick_splits(0, 10, 152, 1) == -1
    assert lib.mla_decode_pick_splits(4, -1, 152, 1) == -1
    assert lib.mla_decode_pick_splits(4, 10, 0, 1) == -1
    assert lib.mla_decode_pick_splits(4, 10, 152, 7) == -1


def test_workspace_slot_counts(lib):
    assert lib.mla_decode_workspace_slots(64, 1, 152) == 0
    assert lib.mla_decode_workspace_slots(64, 7, 152) == 64 * 7
    assert lib.mla_decode_workspace_slots(64, 0, 152) == 64 + 151
    assert lib.mla_decode_workspace_slots(0, 0, 152) == -1
