"""Host-side checks of the seeded input generator and its quantisers (no GPU)."""
import math

import numpy as np
import pytest
import torch

from mla_attention_decode_splitkv_gb300 import synth

E4M3_FINITE = [(c, v) for c, v in enumerate(torch.arange(256, dtype=torch.uint8)
                                             .view(torch.float8_e4m3fn).double().tolist())
               if not math.isnan(v)]
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_fp8_quantiser_is_nearest_with_amax_at_448():
    g = torch.Generator().manual_seed(1)
    x = torch.randn((64, 576), generator=g).to(torch.bfloat16)
    codes, scale = synth.quantize_fp8_per_tensor(x)
    assert scale.dtype == torch.float32 and scale.shape == (1,)
    amax = x.float().abs().max()
    assert scale.item() == pytest.approx(amax.item() / 448.0, rel=1e-7)
    i = int(x.float().abs().argmax())
    assert abs(codes.view(-1)[i].view(torch.float8_e4m3fn).float().item()) == 448.0
    y = (x.float() / scale).view(-1).double().tolist()
    vals = np.array([v for _, v in E4M3_FINITE])
    got = codes.view(torch.float8_e4m3fn).double().view(-1).tolist()
    for yi, gi in list(zip(y, got))[:5000]:
        d = np.abs(vals - yi)
        assert abs(gi - yi) <= d.min() + 1e-12


def test_mxfp4_quantiser_scale_rule_rounding_and_nibble_order():
    g = torch.Generator().manual_seed(2)
    x = (torch.randn((16, 576), generator=g) * 3).to(torch.bfloat16)
    x[3, 32:64] = 0                                              # an all-zero block
    packed, scales = synth.quantize_mxfp4(x)
    assert packed.shape == (16, 288) and scales.shape == (16, 18)
    xf = x.double().numpy()
    for r in range(16):
        for blk in range(18):
            amax = np.abs(xf[r, blk * 32:(blk + 1) * 32]).max()
            if amax == 0:
                expect_e = 127
            else:
                m, e = math.frexp(amax / 6.0)
                expect_e = 127 + (e - 1 if m == 0.5 else e)
            assert scales[r, blk].item() == expect_e
            s = math.ldexp(1.0, expect_e - 127)
            for j in range(32):
                d = blk * 32 + j
                byte = packed[r, d // 2].item()
                code = (byte >> 4) if (d & 1) else (byte & 0xF)
                mag = E2M1_GRID[code & 7]
                y = xf[r, d] / s
                dists = [abs(abs(y) - gv) for gv in E2M1_GRID]
                best = min(dists)
                assert abs(mag - abs(y)) <= best + 1e-12
                ties = [i for i, dd in enumerate(dists) if abs(dd - best) <= 1e-12]
                if len(ties) == 2:
                    assert (code & 7) % 2 == 0                  # ties to the even code
                if mag != 0:
                    assert ((code >> 3) & 1) == (1 if y < 0 else 0)


def test_ragged_lengths_deterministic_and_forced_extremes():
    a = synth.ragged_lengths(128, 8192, 1238)
    b = synth.ragged_lengths(128, 8192, 1238)
    assert a == b and len(a) == 128
    assert min(a) == 1 and max(a) == 8192 and all(1 <= n <= 8192 for n in a)
    assert 1 in a and 8192 in a


def test_indptr_and_small_configs():
    inp = synth.make_config(0)
    assert inp.q.shape == (4, 16, 576) and inp.q.dtype == torch.bfloat16
    assert inp.kv.shape == (4096, 576) and inp.kv.dtype == torch.bfloat16
    assert inp.kv_indptr.tolist() == [0, 1024, 2048, 3072, 4096]
    inp1 = synth.make_config(1)
    assert inp1.kv.dtype == torch.uint8 and inp1.kv.shape == (32768, 576)
    assert inp1.kv_scale.shape == (1,) and inp1.kv_bytes() == 32768 * 576
    spec = synth.CONFIGS[4]
    lens = synth.ragged_lengths(spec.batch, 8192, spec.seed)
    ip = synth.indptr_from_lengths(lens)
    assert ip[0] == 0 and ip[-1] == sum(lens) and torch.all(ip[1:] >= ip[:-1])


def test_same_seed_same_inputs():
    a = synth.make_inputs(2, [3, 5], synth.KV_MXFP4, seed=9)
    b = synth.make_inputs(2, [3, 5], synth.KV_MXFP4, seed=9)
    assert torch.equal(a.q, b.q) and torch.equal(a.kv, b.kv) and torch.equal(a.kv_scale, b.kv_scale)


@pytest.mark.parametrize("kv_dtype", [synth.KV_BF16, synth.KV_FP8, synth.KV_MXFP4])
@pytest.mark.parametrize("page_size", [8, 64, 128])
def test_paged_copy_holds_every_row_once_at_its_page_position(kv_dtype, page_size):
    """The page table of to_paged: pages are distinct, in range and not in order; every
    cached row (and its MXFP4 block scales) sits at page_indices[...] * P + t % P; the
    last-page lengths give back the sequence lengths."""
    lens = [1, 0, 200, 64, 129]
    inp = synth.make_inputs(len(lens), lens, kv_dtype, seed=50)
    pg = synth.to_paged(inp, page_size, seed=51)
    ip, pi, last = pg.page_indptr.tolist(), pg.page_indices.tolist(), pg.last_page_len.tolist()
    assert ip[0] == 0 and len(ip) == len(lens) + 1
    used = pi[:ip[-1]]
    assert len(set(used)) == len(used)
    assert all(0 <= x < pg.kv.shape[0] // page_size for x in used)
    assert pg.kv.shape[0] % page_size == 0
    src_ip = inp.kv_indptr.tolist()
    for b, L in enumerate(lens):
        n = ip[b + 1] - ip[b]
        assert n == (L + page_size - 1) // page_size
        assert (n - 1) * page_size + last[b] == L if n else L == 0
        for t in range(L):
            row = pi[ip[b] + t // page_size] * page_size + t % page_size
            assert torch.equal(pg.kv[row], inp.kv[src_ip[b] + t])
            if kv_dtype == synth.KV_MXFP4:
                assert torch.equal(pg.kv_scale[row], inp.kv_scale[src_ip[b] + t])
    if kv_dtype == synth.KV_FP8:
        assert torch.equal(pg.kv_scale, inp.kv_scale)


def test_paged_copy_is_seeded_and_shuffled():
    inp = synth.make_inputs(3, [300, 5, 700], synth.KV_FP8, seed=52)
    a, b, c = (synth.to_paged(inp, 64, seed=s) for s in (53, 53, 54))
    assert torch.equal(a.page_indices, b.page_indices) and torch.equal(a.kv, b.kv)
    assert not torch.equal(a.page_indices, c.page_indices)
    assert a.page_indices.tolist() != sorted(a.page_indices.tolist())


def test_make_queries_rows_and_indptr():
    q, qo = synth.make_queries([2, 0, 3], seed=55)
    assert q.shape == (5, synth.NUM_HEADS, synth.HEAD_DIM) and q.dtype == torch.bfloat16
    assert qo.tolist() == [0, 2, 2, 5] and qo.dtype == torch.int32
    q2, _ = synth.make_queries([2, 0, 3], seed=55)
    assert torch.equal(q, q2)
