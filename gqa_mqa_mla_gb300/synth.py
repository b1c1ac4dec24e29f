"""Seeded synthetic inputs for decode attention over a paged KV cache.

This module only draws random numbers and lays out paged block tables; it
holds none of the attention arithmetic.  Both the CUDA path (through the
tests and the benchmark) and the fp64 oracle consume the tensors it returns
(the oracle through a host copy of the same bytes).

Recipe (see the workload table at the bottom):
  * element values i.i.d. normal N(0, std^2), rounded to the storage dtype;
  * sequence lengths fixed, or uniform integers in [lo, hi] drawn from a CPU
    generator so they are identical on every machine;
  * block table "identity" (sequence b owns physical blocks
    b*max_blocks .. b*max_blocks + max_blocks - 1, i.e. a contiguous cache) or
    "permuted" (a random permutation of all physical blocks in use);
  * table entries past a sequence's last block hold -1 (never dereferenced);
  * cache slots past seq_len inside a sequence's last block hold random
    values by default, or NaN ("nan" tail) to prove they are never used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, dtype: str, std: float, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(TORCH_DTYPES[dtype])


def draw_seq_lens(batch: int, seq_lens, seed: int) -> torch.Tensor:
    """int32 [batch] lengths: an int (all equal), a list, or ("uniform", lo, hi)."""
    if isinstance(seq_lens, int):
        return torch.full((batch,), seq_lens, dtype=torch.int32)
    if isinstance(seq_lens, tuple) and seq_lens and seq_lens[0] == "uniform":
        _, lo, hi = seq_lens
        g = _gen("cpu", seed + 7919)
        return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64).to(torch.int32)
    t = torch.as_tensor(list(seq_lens), dtype=torch.int32)
    assert t.shape == (batch,)
    return t


def make_block_table(seq_lens: torch.Tensor, block_size: int, table: str, seed: int,
                     max_blocks_per_seq: int | None = None, spare_blocks: int = 0):
    """Returns (block_table int32 [B, max_blocks], num_blocks).

    identity: sequence b uses blocks b*max_blocks + k; num_blocks = B*max_blocks.
    permuted: the blocks in use are a random permutation of range(num_blocks),
              num_blocks = total blocks in use + spare_blocks.
    """
    B = seq_lens.shape[0]
    need = [max(0, math.ceil(int(s) / block_size)) for s in seq_lens.tolist()]
    mb = max_blocks_per_seq if max_blocks_per_seq is not None else max(1, max(need))
    assert mb >= max(need)
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    if table == "identity":
        for b in range(B):
            bt[b, : need[b]] = torch.arange(b * mb, b * mb + need[b], dtype=torch.int32)
        return bt, B * mb + spare_blocks
    if table != "permuted":
        raise ValueError(table)
    total = sum(need)
    num_blocks = total + spare_blocks
    g = _gen("cpu", seed + 104729)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    pos = 0
    for b in range(B):
        bt[b, : need[b]] = perm[pos: pos + need[b]]
        pos += need[b]
    return bt, num_blocks


def _fill_tails(cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                block_size: int, value: float) -> None:
    for b, s in enumerate(seq_lens.tolist()):
        if s <= 0 or s % block_size == 0:
            continue
        blk = int(block_table[b, (s - 1) // block_size])
        cache[blk, s % block_size:] = value


@dataclass
class GQAInputs:
    q: torch.Tensor            # [B, h_q, d]
    k_cache: torch.Tensor      # [num_blocks, block_size, h_kv, d]
    v_cache: torch.Tensor      # [num_blocks, block_size, h_kv, d]
    block_table: torch.Tensor  # int32 [B, max_blocks_per_seq]
    seq_lens: torch.Tensor     # int32 [B]
    h_q: int
    h_kv: int
    d_head: int
    block_size: int
    num_blocks: int
    max_seq_len: int
    dtype: str
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]


def gqa_inputs(batch: int, h_q: int, h_kv: int, d_head: int = 128, seq_lens=256,
               block_size: int = 16, dtype: str = "bf16", seed: int = 0, table: str = "permuted",
               q_std: float = 1.0, kv_std: float = 1.0, device="cpu", tail: str = "random",
               spare_blocks: int = 0, max_blocks_per_seq: int | None = None,
               scale: float | None = None) -> GQAInputs:
    sl = draw_seq_lens(batch, seq_lens, seed)
    bt, nb = make_block_table(sl, block_size, table, seed, max_blocks_per_seq, spare_blocks)
    g = _gen(device, seed)
    q = _randn((batch, h_q, d_head), dtype, q_std, g, device)
    k = _randn((nb, block_size, h_kv, d_head), dtype, kv_std, g, device)
    v = _randn((nb, block_size, h_kv, d_head), dtype, kv_std, g, device)
    if tail == "nan":
        _fill_tails(k, bt, sl, block_size, float("nan"))
        _fill_tails(v, bt, sl, block_size, float("nan"))
    elif tail == "zero":
        _fill_tails(k, bt, sl, block_size, 0.0)
        _fill_tails(v, bt, sl, block_size, 0.0)
    dev_bt = bt.to(device)
    dev_sl = sl.to(device)
    return GQAInputs(q=q, k_cache=k, v_cache=v, block_table=dev_bt, seq_lens=dev_sl, h_q=h_q,
                     h_kv=h_kv, d_head=d_head, block_size=block_size, num_blocks=nb,
                     max_seq_len=int(sl.max()) if batch else 0, dtype=dtype,
                     scale=(1.0 / math.sqrt(d_head)) if scale is None else scale)


@dataclass
class GQAFp8Inputs:
    q: torch.Tensor            # [B, h_q, d] fp16 / bf16
    k_codes: torch.Tensor      # uint8 e4m3 codes [num_blocks, block_size, h_kv, d]
    v_codes: torch.Tensor      # uint8 e4m3 codes [num_blocks, block_size, h_kv, d]
    k_scale: torch.Tensor      # float32 [h_kv]: K value = e4m3(code) * k_scale[kv head]
    v_scale: torch.Tensor      # float32 [h_kv]
    block_table: torch.Tensor  # int32 [B, max_blocks_per_seq]
    seq_lens: torch.Tensor     # int32 [B]
    h_q: int
    h_kv: int
    d_head: int
    block_size: int
    num_blocks: int
    max_seq_len: int
    dtype: str                 # of q and out
    scale: float

    @property
    def batch(self) -> int:
        return self.q.shape[0]


def gqa_fp8_inputs(batch: int, h_q: int, h_kv: int, d_head: int = 128, seq_lens=256,
                   block_size: int = 16, dtype: str = "bf16", seed: int = 0,
                   table: str = "permuted", q_std: float = 1.0, device="cpu",
                   tail: str = "random", spare_blocks: int = 0,
                   max_blocks_per_seq: int | None = None, scale: float | None = None,
                   code_std: float = 112.0) -> GQAFp8Inputs:
    """An 8-bit KV cache drawn directly in its storage format: codes are
    N(0, code_std^2) samples rounded to e4m3 by torch (code_std = 112 puts
    four standard deviations at the largest finite value, 448), and every KV
    head gets its own K and V scale drawn uniformly from [0.5, 1.5] / code_std,
    so the cached values are about unit-variance."""
    sl = draw_seq_lens(batch, seq_lens, seed)
    bt, nb = make_block_table(sl, block_size, table, seed, max_blocks_per_seq, spare_blocks)
    g = _gen(device, seed)
    q = _randn((batch, h_q, d_head), dtype, q_std, g, device)
    shape = (nb, block_size, h_kv, d_head)
    # torch maps magnitudes above 448 to the NaN code: clamp to the finite range first.
    k = (torch.randn(shape, generator=g, device=device) * code_std).clamp_(-448.0, 448.0)
    v = (torch.randn(shape, generator=g, device=device) * code_std).clamp_(-448.0, 448.0)
    k, v = k.to(torch.float8_e4m3fn), v.to(torch.float8_e4m3fn)
    k, v = k.view(torch.uint8), v.view(torch.uint8)
    ks = (torch.rand((h_kv,), generator=g, device=device) + 0.5) / code_std
    vs = (torch.rand((h_kv,), generator=g, device=device) + 0.5) / code_std
    if tail == "nan":
        _fill_tails(k, bt, sl, block_size, 0x7F)  # the e4m3 NaN code
        _fill_tails(v, bt, sl, block_size, 0x7F)
    elif tail == "zero":
        _fill_tails(k, bt, sl, block_size, 0)
        _fill_tails(v, bt, sl, block_size, 0)
    return GQAFp8Inputs(q=q, k_codes=k, v_codes=v, k_scale=ks.float(), v_scale=vs.float(),
                        block_table=bt.to(device), seq_lens=sl.to(device), h_q=h_q, h_kv=h_kv,
                        d_head=d_head, block_size=block_size, num_blocks=nb,
                        max_seq_len=int(sl.max()) if batch else 0, dtype=dtype,
                        scale=(1.0 / math.sqrt(d_head)) if scale is None else scale)


MLA_HEADS = 128
MLA_D_C = 512
MLA_D_R = 64


@dataclass
class MLAInputs:
    q_abs: torch.Tensor        # [B, 128, 512]
    q_rope: torch.Tensor       # [B, 128, 64]
    cache: torch.Tensor        # [num_blocks, block_size, 576]
    block_table: torch.Tensor  # int32 [B, max_blocks_per_seq]
    seq_lens: torch.Tensor     # int32 [B]
    block_size: int
    num_blocks: int
    max_seq_len: int
    dtype: str
    scale: float

    @property
    def batch(self) -> int:
        return self.q_abs.shape[0]


def mla_inputs(batch: int, seq_lens=8192, block_size: int = 64, dtype: str = "bf16",
               seed: int = 0, table: str = "permuted", q_std: float = 1.0, c_std: float = 1.0,
               device="cpu", tail: str = "random", spare_blocks: int = 0,
               max_blocks_per_seq: int | None = None, scale: float | None = None) -> MLAInputs:
    sl = draw_seq_lens(batch, seq_lens, seed)
    bt, nb = make_block_table(sl, block_size, table, seed, max_blocks_per_seq, spare_blocks)
    g = _gen(device, seed)
    qa = _randn((batch, MLA_HEADS, MLA_D_C), dtype, q_std, g, device)
    qr = _randn((batch, MLA_HEADS, MLA_D_R), dtype, q_std, g, device)
    c = _randn((nb, block_size, MLA_D_C + MLA_D_R), dtype, c_std, g, device)
    if tail == "nan":
        _fill_tails(c, bt, sl, block_size, float("nan"))
    elif tail == "zero":
        _fill_tails(c, bt, sl, block_size, 0.0)
    return MLAInputs(q_abs=qa, q_rope=qr, cache=c, block_table=bt.to(device),
                     seq_lens=sl.to(device), block_size=block_size, num_blocks=nb,
                     max_seq_len=int(sl.max()) if batch else 0, dtype=dtype,
                     scale=(1.0 / math.sqrt(128 + 64)) if scale is None else scale)


def new_token_rows(batch: int, row_shape, dtype: str = "bf16", seed: int = 0, std: float = 1.0,
                   device="cpu") -> torch.Tensor:
    """[batch, *row_shape] rows of one new token per sequence (its K or V
    heads, or its MLA latent row), N(0, std^2) rounded to the storage dtype."""
    g = _gen(device, seed + 15485863)
    return _randn((batch, *row_shape), dtype, std, g, device)


@dataclass
class MLAAbsorbInputs:
    q_nope: torch.Tensor   # [B, H, d_h]  per-head query (before absorption)
    w_uk: torch.Tensor     # [H, d_c, d_h] W_uk^(i): latent -> key
    o_lat: torch.Tensor    # [B, H, d_c]  softmax-weighted latent (decode output)
    w_uv_t: torch.Tensor   # [H, d_v, d_c] W_uv^(i) transposed: latent -> value
    dtype: str


def mla_absorb_inputs(batch: int, heads: int = MLA_HEADS, d_h: int = 128, d_c: int = MLA_D_C,
                      d_v: int = 128, dtype: str = "bf16", seed: int = 0,
                      device="cpu") -> MLAAbsorbInputs:
    """Random-init up-projection weights (std 1/sqrt(fan-in), so products stay
    about unit-variance) and unit-variance activations."""
    g = _gen(device, seed + 32452843)
    return MLAAbsorbInputs(
        q_nope=_randn((batch, heads, d_h), dtype, 1.0, g, device),
        w_uk=_randn((heads, d_c, d_h), dtype, 1.0 / math.sqrt(d_h), g, device),
        o_lat=_randn((batch, heads, d_c), dtype, 1.0, g, device),
        w_uv_t=_randn((heads, d_v, d_c), dtype, 1.0 / math.sqrt(d_c), g, device),
        dtype=dtype)


def u16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit storage of a fp16/bf16 tensor as a host uint16 numpy array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# Named workloads (single decode layer each), with the shapes of the models
# they are drawn from.  Each entry: (kind, kwargs for gqa_inputs/mla_inputs).
WORKLOADS = {
    # tiny GQA, contiguous cache: B=2, 8 query heads on 2 KV heads, S=256, fp16
    "gqa_tiny_b2_s256": ("gqa", dict(batch=2, h_q=8, h_kv=2, seq_lens=256, block_size=16,
                                     dtype="fp16", table="identity")),
    # Llama-3.1-8B-shaped layer, 32 query heads, MHA / GQA-8kv / MQA
    "llama31_8b_mha_b16": ("gqa", dict(batch=16, h_q=32, h_kv=32, seq_lens=("uniform", 1024, 4096),
                                       block_size=16, dtype="bf16", table="permuted")),
    "llama31_8b_gqa_b16": ("gqa", dict(batch=16, h_q=32, h_kv=8, seq_lens=("uniform", 1024, 4096),
                                       block_size=16, dtype="bf16", table="permuted")),
    "llama31_8b_mqa_b16": ("gqa", dict(batch=16, h_q=32, h_kv=1, seq_lens=("uniform", 1024, 4096),
                                       block_size=16, dtype="bf16", table="permuted")),
    # Llama-3-70B-shaped layer, large batch: 64 query heads on 8 KV heads
    "llama3_70b_b64_s8k": ("gqa", dict(batch=64, h_q=64, h_kv=8, seq_lens=8192, block_size=16,
                                       dtype="bf16", table="permuted", q_std=0.5)),
    # the same 70B-shaped layer over an 8-bit (e4m3) KV cache with per-KV-head scales
    "llama3_70b_b64_s8k_fp8": ("gqa_fp8", dict(batch=64, h_q=64, h_kv=8, seq_lens=8192,
                                               block_size=16, dtype="bf16", table="permuted",
                                               q_std=0.5)),
    # DeepSeek-V2-shaped absorbed MLA layer
    "deepseek_v2_mla_b32_s8k": ("mla", dict(batch=32, seq_lens=8192, block_size=64,
                                            dtype="bf16", table="permuted")),
    # long-context split-KV stress, 70B-shaped heads
    "long_ctx_b1_s128k": ("gqa", dict(batch=1, h_q=64, h_kv=8, seq_lens=131072, block_size=16,
                                      dtype="bf16", table="permuted")),
    "long_ctx_b4_s128k": ("gqa", dict(batch=4, h_q=64, h_kv=8, seq_lens=131072, block_size=16,
                                      dtype="bf16", table="permuted")),
    # wide query groups (tensor-core path): 32 query heads per KV head
    # (70B-shaped heads on 2 KV heads) and 64 (MQA with 64 query heads)
    "wide_g32_b64_s8k": ("gqa", dict(batch=64, h_q=64, h_kv=2, seq_lens=8192, block_size=16,
                                     dtype="bf16", table="permuted", q_std=0.5)),
    "wide_g64_mqa_b128_s8k": ("gqa", dict(batch=128, h_q=64, h_kv=1, seq_lens=8192,
                                          block_size=16, dtype="bf16", table="permuted",
                                          q_std=0.5)),
    # the same MQA layer over an 8-bit (e4m3) KV cache
    "wide_g64_mqa_b128_s8k_fp8": ("gqa_fp8", dict(batch=128, h_q=64, h_kv=1, seq_lens=8192,
                                                  block_size=16, dtype="bf16",
                                                  table="permuted", q_std=0.5)),
}


def workload_inputs(name: str, device="cpu", seed: int = 0, **overrides):
    kind, kw = WORKLOADS[name]
    kw = {**kw, **overrides}
    if kind == "gqa":
        return gqa_inputs(seed=seed, device=device, **kw)
    if kind == "gqa_fp8":
        return gqa_fp8_inputs(seed=seed, device=device, **kw)
    return mla_inputs(seed=seed, device=device, **kw)
