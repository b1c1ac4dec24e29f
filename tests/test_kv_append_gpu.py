"""GPU parity of the decode step's cache write (gqa_kv_append,
gqa_kv_append_fp8kv, mla_kv_append) against the oracle's paged-slot write
and e4m3 quantiser: byte work, so every comparison is bit-exact over the
whole cache."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
import oracle
from gqa_mqa_mla_gb300 import synth

from _parity import compare, gather_rows, oracle_gqa, oracle_gqa_fp8, oracle_mla

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _positions(x, skip=()):
    """Append at each sequence's last position (the inputs are drawn with
    room for it: seq_lens already count the new token); -1 for skips."""
    pos = (x.seq_lens.cpu() - 1).clamp(min=-1)
    for b in skip:
        pos[b] = -1
    return pos.to(torch.int32)


def _u8(t):
    return t.detach().contiguous().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("h_kv", [1, 2, 8, 64])
@pytest.mark.parametrize("block_size", [8, 16, 64, 256])
def test_gqa_append_writes_exactly_the_addressed_slots(dtype, h_kv, block_size):
    lens = [1, 17, block_size, block_size + 1, 3 * block_size, 0, 100]
    x = synth.gqa_inputs(batch=len(lens), h_q=h_kv, h_kv=h_kv, seq_lens=lens,
                         block_size=block_size, dtype=dtype, seed=h_kv + block_size, device=DEV)
    kn = synth.new_token_rows(x.batch, (h_kv, 128), dtype, seed=1, device=DEV)
    vn = synth.new_token_rows(x.batch, (h_kv, 128), dtype, seed=2, device=DEV)
    pos = _positions(x, skip=(6,))
    k0, v0 = synth.u16(x.k_cache), synth.u16(x.v_cache)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    da.gqa_kv_append(kn, vn, pos.to(DEV), x.block_table, x.k_cache, x.v_cache, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    bt = x.block_table.cpu().numpy()
    k_ref, bad_k = oracle.kv_append(k0, synth.u16(kn), pos.numpy(), bt)
    v_ref, bad_v = oracle.kv_append(v0, synth.u16(vn), pos.numpy(), bt)
    assert bad_k == bad_v == {}
    assert np.array_equal(synth.u16(x.k_cache), k_ref)
    assert np.array_equal(synth.u16(x.v_cache), v_ref)


def test_bad_positions_and_block_ids_are_flagged_and_skipped():
    x = synth.gqa_inputs(batch=4, h_q=8, h_kv=2, seq_lens=[20, 20, 20, 20], block_size=16,
                         seed=3, device=DEV)
    kn = synth.new_token_rows(4, (2, 128), "bf16", seed=4, device=DEV)
    vn = synth.new_token_rows(4, (2, 128), "bf16", seed=5, device=DEV)
    bt = x.block_table.clone()
    bt[1, 1] = x.num_blocks + 7           # out-of-range block id at position 19
    pos = torch.tensor([19, 19, 32, 18], dtype=torch.int32)  # 32 is past the 2-block table
    k0, v0 = synth.u16(x.k_cache), synth.u16(x.v_cache)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    da.gqa_kv_append(kn, vn, pos.to(DEV), bt, x.k_cache, x.v_cache, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == da.FLAG_BAD_BLOCK | da.FLAG_BAD_SEQ_LEN
    k_ref, bad = oracle.kv_append(k0, synth.u16(kn), pos.numpy(), bt.cpu().numpy())
    v_ref, _ = oracle.kv_append(v0, synth.u16(vn), pos.numpy(), bt.cpu().numpy())
    assert bad == {1: "bad_block", 2: "bad_position"}
    assert np.array_equal(synth.u16(x.k_cache), k_ref)
    assert np.array_equal(synth.u16(x.v_cache), v_ref)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("h_kv", [1, 8, 16])
@pytest.mark.parametrize("block_size", [16, 64])
def test_fp8_append_quantises_like_the_oracle(dtype, h_kv, block_size):
    lens = [5, 64, 65, 200, 1]
    x = synth.gqa_fp8_inputs(batch=len(lens), h_q=h_kv, h_kv=h_kv, seq_lens=lens,
                             block_size=block_size, dtype=dtype, seed=h_kv * 3 + block_size,
                             device=DEV)
    # about unit variance against scales near 1/112, with a heavy tail that
    # reaches past +-448 * scale (saturation) and values that round to zero
    kn = synth.new_token_rows(x.batch, (h_kv, 128), dtype, seed=6, std=2.0, device=DEV)
    vn = synth.new_token_rows(x.batch, (h_kv, 128), dtype, seed=7, std=2.0, device=DEV)
    kn[0, :, :8] = 1e-5
    kn[1, :, :8] = 60.0
    vn[2, :, :8] = -60.0
    pos = _positions(x)
    k0, v0 = _u8(x.k_codes), _u8(x.v_codes)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    da.gqa_kv_append_fp8kv(kn, vn, x.k_scale, x.v_scale, pos.to(DEV), x.block_table, x.k_codes,
                           x.v_codes, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    bt = x.block_table.cpu().numpy()
    kq = oracle.quant_e4m3(synth.u16(kn), dtype, x.k_scale.cpu().numpy())
    vq = oracle.quant_e4m3(synth.u16(vn), dtype, x.v_scale.cpu().numpy())
    k_ref, _ = oracle.kv_append(k0, kq, pos.numpy(), bt)
    v_ref, _ = oracle.kv_append(v0, vq, pos.numpy(), bt)
    assert np.array_equal(_u8(x.k_codes), k_ref)
    assert np.array_equal(_u8(x.v_codes), v_ref)
    assert (kq == 0x7E).any() or (kq == 0xFE).any()  # saturation was exercised


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_append_rounds_ties_to_even_and_saturates(dtype):
    """Midpoints between adjacent e4m3 values, times power-of-two scales, are
    exact in 16 bits: x / scale hits the tie exactly and must take the even
    code; values past 448 * scale must take 448."""
    h_kv = 2
    x = synth.gqa_fp8_inputs(batch=1, h_q=2, h_kv=h_kv, seq_lens=[9], block_size=16, seed=8,
                             device=DEV)
    scale = torch.tensor([0.25, 2.0], dtype=torch.float32, device=DEV)
    lo = np.arange(0x00, 0x7B, dtype=np.uint8)  # 123 pairs (c, c + 1), both finite
    mids = (oracle.e4m3_to_double(lo) + oracle.e4m3_to_double(lo + 1)) / 2
    mids = np.concatenate([mids, -mids[:3], [512.0, 4096.0]])
    assert mids.shape == (128,)
    row = torch.tensor(mids, dtype=torch.float64)
    kn = torch.stack([row * 0.25, row * 2.0]).to(synth.TORCH_DTYPES[dtype])[None].to(DEV)
    if dtype == "fp16":  # fp16 keeps the tiny midpoints only down to its subnormals
        assert torch.all(torch.isfinite(kn))
    vn = kn.clone()
    pos = torch.tensor([8], dtype=torch.int32)
    da.gqa_kv_append_fp8kv(kn, vn, scale, scale, pos.to(DEV), x.block_table, x.k_codes,
                           x.v_codes)
    torch.cuda.synchronize()
    kq = oracle.quant_e4m3(synth.u16(kn), dtype, scale.cpu().numpy())
    blk = int(x.block_table[0, 0])
    assert np.array_equal(_u8(x.k_codes)[blk, 8], kq[0])
    assert np.array_equal(_u8(x.v_codes)[blk, 8], kq[0])
    # every midpoint times a power of two is exact in 16 bits: all ties, all even
    got = _u8(x.k_codes)[blk, 8, :, :len(lo)]
    assert np.all(got % 2 == 0)
    assert np.all(_u8(x.k_codes)[blk, 8, :, 126:] == 0x7E)  # 512 and 4096 saturate


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("block_size", [8, 16, 64])
def test_mla_append_writes_the_latent_and_rope_key(dtype, block_size):
    lens = [1, block_size, block_size + 1, 300, 0]
    x = synth.mla_inputs(batch=len(lens), seq_lens=lens, block_size=block_size, dtype=dtype,
                         seed=block_size, device=DEV)
    cn = synth.new_token_rows(x.batch, (576,), dtype, seed=9, device=DEV)
    pos = _positions(x)
    c0 = synth.u16(x.cache)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    da.mla_kv_append(cn, pos.to(DEV), x.block_table, x.cache, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    ref, bad = oracle.kv_append(c0, synth.u16(cn), pos.numpy(), x.block_table.cpu().numpy())
    assert bad == {}
    assert np.array_equal(synth.u16(x.cache), ref)


def test_decode_step_append_then_attend_gqa_and_fp8():
    """One decode step end to end: write the new token, then attend over the
    grown sequences; the oracle attends over its own appended cache."""
    lens = [1, 64, 65, 300]
    x = synth.gqa_inputs(batch=4, h_q=16, h_kv=2, seq_lens=lens, block_size=16, seed=10,
                         device=DEV)
    kn = synth.new_token_rows(4, (2, 128), "bf16", seed=11, device=DEV)
    vn = synth.new_token_rows(4, (2, 128), "bf16", seed=12, device=DEV)
    da.gqa_kv_append(kn, vn, _positions(x).to(DEV), x.block_table, x.k_cache, x.v_cache)
    out = da.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale=x.scale,
                        max_seq_len=x.max_seq_len)
    torch.cuda.synchronize()
    ref, _ = oracle_gqa(x)  # reads the cache after the append (copied back to the host)
    compare(gather_rows(out, None), ref, "append+decode")

    f = synth.gqa_fp8_inputs(batch=4, h_q=16, h_kv=2, seq_lens=lens, block_size=16, seed=13,
                             device=DEV)
    kn = synth.new_token_rows(4, (2, 128), "bf16", seed=14, device=DEV)
    vn = synth.new_token_rows(4, (2, 128), "bf16", seed=15, device=DEV)
    da.gqa_kv_append_fp8kv(kn, vn, f.k_scale, f.v_scale, _positions(f).to(DEV), f.block_table,
                           f.k_codes, f.v_codes)
    out = da.gqa_decode_fp8kv(f.q, f.k_codes, f.v_codes, f.k_scale, f.v_scale, f.block_table,
                              f.seq_lens, scale=f.scale, max_seq_len=f.max_seq_len)
    torch.cuda.synchronize()
    ref, _ = oracle_gqa_fp8(f)
    compare(gather_rows(out, None), ref, "fp8 append+decode")


def test_decode_step_append_then_attend_mla():
    x = synth.mla_inputs(batch=3, seq_lens=[1, 64, 200], block_size=64, seed=16, device=DEV)
    cn = synth.new_token_rows(3, (576,), "bf16", seed=17, device=DEV)
    da.mla_kv_append(cn, _positions(x).to(DEV), x.block_table, x.cache)
    out = da.mla_decode(x.q_abs, x.q_rope, x.cache, x.block_table, x.seq_lens, scale=x.scale,
                        max_seq_len=x.max_seq_len)
    torch.cuda.synchronize()
    ref, _ = oracle_mla(x)
    compare(gather_rows(out, None), ref, "mla append+decode")


@pytest.mark.parametrize("name", ["llama3_70b_b64_s8k", "llama3_70b_b64_s8k_fp8",
                                  "deepseek_v2_mla_b32_s8k"])
def test_full_size_layers_change_only_the_appended_slots(name):
    x = synth.workload_inputs(name, device=DEV)
    pos = _positions(x).to(DEV)
    bt = x.block_table
    b = torch.arange(x.batch, device=DEV)
    rows = bt[b, pos.long() // x.block_size].long() * x.block_size + pos.long() % x.block_size
    if name.startswith("deepseek"):
        caches = [x.cache]
        news = [synth.new_token_rows(x.batch, (576,), "bf16", seed=18, device=DEV)]
        before = [c.clone() for c in caches]
        da.mla_kv_append(news[0], pos, bt, x.cache)
        expect = news
    elif name.endswith("fp8"):
        caches = [x.k_codes, x.v_codes]
        news = [synth.new_token_rows(x.batch, (x.h_kv, 128), "bf16", seed=s, device=DEV)
                for s in (19, 20)]
        before = [c.clone() for c in caches]
        da.gqa_kv_append_fp8kv(news[0], news[1], x.k_scale, x.v_scale, pos, bt, *caches)
        expect = [torch.from_numpy(oracle.quant_e4m3(synth.u16(n), "bf16", s.cpu().numpy()))
                  .to(DEV) for n, s in zip(news, (x.k_scale, x.v_scale))]
    else:
        caches = [x.k_cache, x.v_cache]
        news = [synth.new_token_rows(x.batch, (x.h_kv, 128), "bf16", seed=s, device=DEV)
                for s in (21, 22)]
        before = [c.clone() for c in caches]
        da.gqa_kv_append(news[0], news[1], pos, bt, *caches)
        expect = news
    torch.cuda.synchronize()
    for c, c0, e in zip(caches, before, expect):
        flat, flat0 = c.view(-1, *c.shape[2:]), c0.view(-1, *c0.shape[2:])
        assert torch.equal(flat[rows], e.view(flat[rows].shape))
        keep = torch.ones(flat.shape[0], dtype=torch.bool, device=DEV)
        keep[rows] = False
        assert torch.equal(flat[keep], flat0[keep])
