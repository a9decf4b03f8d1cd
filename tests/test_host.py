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
    for ps in (0, 1, 2, 4, 12, 48, 96, 256, -64):
        assert _call_paged(lib, ps=ps) == INV          # page size: a power of two in [8, 128]
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
    for ps in (0, 4, 48, 256):
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
    assert _call_paged(lib, ps=128) in (-2, -3)
    assert _call_multi(lib) in (-2, -3)


@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_pick_splits_follows_the_documented_rule(lib, dtype):
    for batch in (1, 4, 32, 64, 75, 76, 77, 128, 151, 152, 153, 256, 1000):
        for L in (0, 1, 100, 127, 128, 256, 257, 1024, 2048, 2049, 4000, 8192, 65536, 10**6):
            for sms in (148, 152):
                ns = min(sms // batch, -(-L // 256), math.isqrt(L // 32))
                want = ns if ns >= 2 else (1 if L <= 2048 else 0)
                assert lib.mla_decode_pick_splits(batch, L, sms, dtype) == want, (batch, L, sms)
    # the workloads: 64 x 8192 -> 2 splits, 32 x 1024 -> 4, 256 x 8192 -> balanced, a ragged
    # batch of 128 (mean length 4096) -> balanced; 256 x 1024 -> 1, 4 x 8192 -> 16
    assert lib.mla_decode_pick_splits(64, 8192, 152, 1) == 2
    assert lib.mla_decode_pick_splits(32, 1024, 152, 1) == 4
    assert lib.mla_decode_pick_splits(256, 8192, 152, 2) == 0
    assert lib.mla_decode_pick_splits(128, 4096, 152, 1) == 0
    assert lib.mla_decode_pick_splits(256, 1024, 152, 1) == 1
    assert lib.mla_decode_pick_splits(4, 8192, 152, 1) == 16


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
