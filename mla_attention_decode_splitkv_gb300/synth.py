"""Seeded synthetic inputs for single-token MLA decode.

This module only *makes inputs*: random q and KV caches, their storage encodings
(bf16, fp8-e4m3 with one per-tensor scale, MXFP4 = e2m1 nibbles + e8m0 block scales)
and the int32 ``kv_indptr`` row index (page size 1).  It holds none of the decode
arithmetic (no dequantisation, no attention), so both the CUDA path and the CPU oracle
can consume what it produces without sharing any of the method's code.

The workloads are the leaderboard shapes of the amd-mixed-mla submissions
(batch x kv_len in {4, 32, 64, 256} x {1024, 8192}, 16 query heads over one latent KV
head of width 576); the task's own input generator is not part of the pages, so the
recipe below stands in for it:

* q ~ N(0, 1) in bf16, shape [batch, 16, 576];
* the KV source ~ N(0, 1) in bf16, shape [total_rows, 576];
* fp8: scale = amax / 448 in fp32, code = round-to-nearest-even(x / scale) to e4m3fn,
  saturated to +-448;
* MXFP4: per row, per block of 32 consecutive values, E = 127 + ceil(log2(amax / 6))
  (E = 127 for an all-zero block), element = round-to-nearest-even(x / 2^(E-127)) on the
  e2m1 grid {0, 0.5, 1, 1.5, 2, 3, 4, 6}; element 2i in the low nibble of byte i;
* seeds: ``torch.Generator`` seeded with 1234 + config index.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch

NUM_HEADS = 16
HEAD_DIM = 576
V_DIM = 512
MX_BLOCK = 32
MX_PACKED_BYTES = HEAD_DIM // 2          # 288
MX_SCALES = HEAD_DIM // MX_BLOCK         # 18

KV_BF16, KV_FP8, KV_MXFP4 = 0, 1, 2
DTYPE_NAMES = {KV_BF16: "bf16", KV_FP8: "fp8_e4m3", KV_MXFP4: "mxfp4"}
KV_ROW_BYTES = {KV_BF16: HEAD_DIM * 2, KV_FP8: HEAD_DIM, KV_MXFP4: MX_PACKED_BYTES + MX_SCALES}


@dataclasses.dataclass(frozen=True)
class ConfigSpec:
    name: str
    batch: int
    kv_len: Optional[int]          # None -> ragged
    kv_dtype: int
    num_splits: Optional[int]      # None -> mla_decode_pick_splits (0 = balanced mode)
    seed: int


# The five workloads (index = position in the list); seeds are 1234 + index.
CONFIGS: List[ConfigSpec] = [
    ConfigSpec("bf16_b4_l1024_ns1", 4, 1024, KV_BF16, 1, 1234),
    ConfigSpec("fp8_b32_l1024", 32, 1024, KV_FP8, None, 1235),
    ConfigSpec("fp8_b64_l8192_splitkv", 64, 8192, KV_FP8, None, 1236),
    ConfigSpec("mxfp4_b256_l8192", 256, 8192, KV_MXFP4, None, 1237),
    # A ragged batch runs in the balanced mode: the split model's length hint describes
    # batches of equal lengths.
    ConfigSpec("fp8_ragged_b128_l1to8192", 128, None, KV_FP8, 0, 1238),
]


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor                 # bf16 [batch, 16, 576]
    kv_src: Optional[torch.Tensor]  # bf16 [rows, 576] before quantisation (None if dropped)
    kv: torch.Tensor                # bf16 [rows,576] | uint8 [rows,576] | uint8 [rows,288]
    kv_scale: Optional[torch.Tensor]  # None | fp32 [1] | uint8 [rows, 18]
    kv_indptr: torch.Tensor         # int32 [batch + 1]
    kv_dtype: int
    lens: List[int]

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def rows(self) -> int:
        return int(self.kv.shape[0])

    def kv_bytes(self) -> int:
        """Bytes of KV cache a decode must read (every cached row once)."""
        return self.rows * KV_ROW_BYTES[self.kv_dtype]

    def to(self, device) -> "DecodeInputs":
        mv = lambda t: None if t is None else t.to(device)
        return DecodeInputs(mv(self.q), mv(self.kv_src), mv(self.kv), mv(self.kv_scale),
                            mv(self.kv_indptr), self.kv_dtype, list(self.lens))


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def ragged_lengths(batch: int, max_len: int, seed: int) -> List[int]:
    """Lengths uniform in [1, max_len]; one length 1 and one length max_len are forced at
    two seed-chosen positions."""
    g = _gen("cpu", seed)
    lens = torch.randint(1, max_len + 1, (batch,), generator=g)
    if batch >= 2:
        idx = torch.randperm(batch, generator=g)[:2]
        lens[idx[0]] = 1
        lens[idx[1]] = max_len
    elif batch == 1:
        lens[0] = max_len
    return [int(x) for x in lens]


def indptr_from_lengths(lens: List[int]) -> torch.Tensor:
    ptr = [0]
    for n in lens:
        ptr.append(ptr[-1] + int(n))
    return torch.tensor(ptr, dtype=torch.int32)


def quantize_fp8_per_tensor(x: torch.Tensor):
    """bf16/fp32 tensor -> (uint8 e4m3fn codes, fp32 [1] scale = amax / 448)."""
    xf = x.float()
    amax = xf.abs().max()
    scale = (amax / 448.0).clamp_min(torch.finfo(torch.float32).tiny)
    y = (xf / scale).clamp(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.reshape(1).to(torch.float32)


# e2m1 rounding thresholds on |x| (value grid 0,.5,1,1.5,2,3,4,6; ties go to the even code).
_E2M1_UPPER = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]      # boundaries between codes c and c+1
_E2M1_TIE_UP = [False, True, False, True, False, True, False]  # tie rounds to c+1 (even) ?


def _e2m1_magnitude_code(mag: torch.Tensor) -> torch.Tensor:
    code = torch.zeros_like(mag, dtype=torch.uint8)
    for c, (b, up) in enumerate(zip(_E2M1_UPPER, _E2M1_TIE_UP)):
        above = (mag >= b) if up else (mag > b)
        code = torch.where(above, torch.full_like(code, c + 1), code)
    return code


def quantize_mxfp4(x: torch.Tensor, chunk_rows: int = 1 << 18):
    """[rows, 576] -> (uint8 [rows, 288] packed e2m1, uint8 [rows, 18] e8m0 scales)."""
    rows = x.shape[0]
    packed = torch.empty((rows, MX_PACKED_BYTES), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, MX_SCALES), dtype=torch.uint8, device=x.device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        xb = x[r0:r1].float().reshape(r1 - r0, MX_SCALES, MX_BLOCK)
        amax = xb.abs().amax(dim=-1)                                   # [n, 18]
        ratio = amax / 6.0
        mant, expo = torch.frexp(ratio)                                # ratio = mant * 2^expo, mant in [0.5,1)
        k = torch.where(mant == 0.5, expo - 1, expo)                   # ceil(log2(ratio)) exactly
        k = torch.where(amax > 0, k, torch.zeros_like(k))
        e = (k + 127).clamp(0, 254)
        k = e - 127
        y = xb / torch.ldexp(torch.ones_like(ratio), k.to(torch.float32)).unsqueeze(-1)
        mag = _e2m1_magnitude_code(y.abs())
        sign = ((y < 0) & (mag > 0)).to(torch.uint8) << 3
        code = (mag | sign).reshape(r1 - r0, HEAD_DIM)
        packed[r0:r1] = code[:, 0::2] | (code[:, 1::2] << 4)
        scales[r0:r1] = e.to(torch.uint8)
    return packed, scales


def make_inputs(batch: int, lens, kv_dtype: int, seed: int, device="cpu",
                keep_src: bool = True) -> DecodeInputs:
    """Random q / KV for the given per-sequence lengths, stored as `kv_dtype`."""
    if isinstance(lens, int):
        lens = [lens] * batch
    lens = [int(n) for n in lens]
    assert len(lens) == batch
    indptr = indptr_from_lengths(lens)
    rows = int(indptr[-1])
    g = _gen(device, seed)
    q = torch.randn((batch, NUM_HEADS, HEAD_DIM), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    src = torch.randn((max(rows, 1), HEAD_DIM), generator=g, device=device,
                      dtype=torch.float32).to(torch.bfloat16)[:rows]
    if kv_dtype == KV_BF16:
        kv, scale = src, None
    elif kv_dtype == KV_FP8:
        if rows:
            kv, scale = quantize_fp8_per_tensor(src)
        else:
            kv = torch.zeros((0, HEAD_DIM), dtype=torch.uint8, device=device)
            scale = torch.ones(1, dtype=torch.float32, device=device)
    elif kv_dtype == KV_MXFP4:
        kv, scale = quantize_mxfp4(src)
    else:
        raise ValueError(f"unknown kv dtype {kv_dtype}")
    return DecodeInputs(q, src if keep_src else None, kv, scale, indptr.to(device), kv_dtype, lens)


def make_config(index: int, device="cpu", keep_src: bool = True) -> DecodeInputs:
    spec = CONFIGS[index]
    if spec.kv_len is None:
        lens = ragged_lengths(spec.batch, 8192, spec.seed)
    else:
        lens = [spec.kv_len] * spec.batch
    return make_inputs(spec.batch, lens, spec.kv_dtype, spec.seed, device=device, keep_src=keep_src)



@dataclasses.dataclass
class PagedInputs:
    """A paged copy of a DecodeInputs cache: the same rows, stored in shuffled physical pages."""
    q: torch.Tensor
    kv: torch.Tensor                # [num_pages * page_size, row width] (same encoding as the source)
    kv_scale: Optional[torch.Tensor]  # None | fp32 [1] | uint8 [num_pages * page_size, 18]
    page_indptr: torch.Tensor       # int32 [batch + 1]
    page_indices: torch.Tensor      # int32 [sum of pages]
    last_page_len: torch.Tensor     # int32 [batch]
    page_size: int
    kv_dtype: int
    lens: List[int]

    def to(self, device) -> "PagedInputs":
        mv = lambda t: None if t is None else t.to(device)
        return PagedInputs(mv(self.q), mv(self.kv), mv(self.kv_scale), mv(self.page_indptr), mv(self.page_indices),
                           mv(self.last_page_len), self.page_size, self.kv_dtype, list(self.lens))


def to_paged(inp: DecodeInputs, page_size: int, seed: int, spare_pages: int = 3) -> PagedInputs:
    """Store the rows of `inp` in pages of `page_size` rows at shuffled physical page numbers
    (plus `spare_pages` unused pages).  Rows of a page past a sequence's end, and the spare
    pages, hold other rows of the same cache (valid encodings, so that nothing read there is
    NaN) -- the decode must mask them."""
    g = torch.Generator()
    g.manual_seed(seed)
    ip = inp.kv_indptr.cpu().tolist()
    kv = inp.kv.cpu()
    sc = inp.kv_scale.cpu() if inp.kv_scale is not None else None
    rows = max(int(ip[-1]), 1)
    npages = [(int(ip[b + 1] - ip[b]) + page_size - 1) // page_size for b in range(inp.batch)]
    total = sum(npages) + spare_pages
    perm = torch.randperm(total, generator=g)
    filler = torch.randint(0, rows, (total * page_size,), generator=g)
    kv_pages = kv[filler].clone() if ip[-1] > 0 else torch.zeros((total * page_size,) + tuple(kv.shape[1:]), dtype=kv.dtype)
    sc_pages = None
    if inp.kv_dtype == KV_MXFP4:
        sc_pages = sc[filler].clone() if ip[-1] > 0 else torch.full((total * page_size, MX_SCALES), 127, dtype=torch.uint8)
    elif sc is not None:
        sc_pages = sc.clone()
    indices, indptr, last = [], [0], []
    k = 0
    for b in range(inp.batch):
        L = int(ip[b + 1] - ip[b])
        for j in range(npages[b]):
            pid = int(perm[k]); k += 1
            n = min(page_size, L - j * page_size)
            src = slice(int(ip[b]) + j * page_size, int(ip[b]) + j * page_size + n)
            kv_pages[pid * page_size:pid * page_size + n] = kv[src]
            if inp.kv_dtype == KV_MXFP4:
                sc_pages[pid * page_size:pid * page_size + n] = sc[src]
            indices.append(pid)
        indptr.append(len(indices))
        last.append(L - (npages[b] - 1) * page_size if npages[b] else 0)
    return PagedInputs(inp.q.cpu(), kv_pages, sc_pages, torch.tensor(indptr, dtype=torch.int32),
                       torch.tensor(indices if indices else [0], dtype=torch.int32),
                       torch.tensor(last, dtype=torch.int32), page_size, inp.kv_dtype, list(inp.lens))


def make_queries(q_lens, seed: int, device="cpu"):
    """Several query tokens per sequence: q bf16 [sum(q_lens), 16, 576] ~ N(0, 1) and the
    int32 qo_indptr [len(q_lens) + 1]."""
    q_lens = [int(n) for n in q_lens]
    g = _gen(device, seed)
    q = torch.randn((max(sum(q_lens), 1), NUM_HEADS, HEAD_DIM), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)[:sum(q_lens)]
    return q, indptr_from_lengths(q_lens).to(device)
