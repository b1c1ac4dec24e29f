"""GPU parity of the sliding-window decode calls (gqa_decode_window over
16-bit caches, gqa_decode_fp8kv_window over e4m3 caches) against the fp64
oracle: the plain GQA definition over each sequence's last `window`
positions ("07 · MHA/MQA/GQA/MLA quick learn", on sliding-window
attention), through the C ABI."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
import oracle
from gqa_mqa_mla_gb300 import synth

from _parity import (compare, gather_rows, oracle_gqa_fp8_window, oracle_gqa_window,
                     sample_rows)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, window, num_splits=0, err_flag=None, block_table=None, k=None, v=None):
    bt = x.block_table if block_table is None else block_table
    if isinstance(x, synth.GQAFp8Inputs):
        out = da.gqa_decode_fp8kv_window(
            x.q, x.k_codes if k is None else k, x.v_codes if v is None else v, x.k_scale,
            x.v_scale, bt, x.seq_lens, window=window, scale=x.scale, max_seq_len=x.max_seq_len,
            num_splits=num_splits, err_flag=err_flag)
    else:
        out = da.gqa_decode_window(x.q, x.k_cache if k is None else k,
                                   x.v_cache if v is None else v, bt, x.seq_lens, window=window,
                                   scale=x.scale, max_seq_len=x.max_seq_len,
                                   num_splits=num_splits, err_flag=err_flag)
    torch.cuda.synchronize()
    return out


def _oracle(x, window, rows, **kw):
    if isinstance(x, synth.GQAFp8Inputs):
        kw = {("k_codes" if a == "k" else "v_codes" if a == "v" else a): t for a, t in kw.items()}
        return oracle_gqa_fp8_window(x, window, rows, **kw)
    kw = {("k_cache" if a == "k" else "v_cache" if a == "v" else a): t for a, t in kw.items()}
    return oracle_gqa_window(x, window, rows, **kw)


def _check(x, window, num_splits=0, n_rows=None, what="", **kw):
    rows = sample_rows(x.batch, x.h_q, n_rows)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(x, window, num_splits, err_flag=flag, **kw)
    assert int(flag.item()) == 0, f"{what}: error flag {int(flag.item())}"
    ref, _ = _oracle(x, window, rows, **kw)
    return compare(gather_rows(out, rows), ref, what)


def _inputs(fp8, **kw):
    return synth.gqa_fp8_inputs(**kw) if fp8 else synth.gqa_inputs(**kw)


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "e4m3"])
@pytest.mark.parametrize("h_q,h_kv", [(8, 8), (8, 2), (32, 8), (32, 1), (64, 8), (48, 2)])
@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_group_sizes_and_splits(fp8, h_q, h_kv, num_splits):
    x = _inputs(fp8, batch=5, h_q=h_q, h_kv=h_kv, seq_lens=[300, 1, 129, 0, 65], block_size=16,
                seed=h_q * 7 + h_kv, device=DEV)
    for w in (1, 17, 64, 65, 200):
        _check(x, w, num_splits, what=f"fp8={fp8} h_q={h_q} h_kv={h_kv} splits={num_splits} w={w}")


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "e4m3"])
@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128, 256])
def test_block_sizes_and_window_boundaries(fp8, block_size):
    lens = [0, 1, 31, 63, 64, 65, 100, 257, 1000]
    x = _inputs(fp8, batch=len(lens), h_q=16, h_kv=2, seq_lens=lens, block_size=block_size,
                seed=block_size + 3, device=DEV)
    for w in (1, 2, 63, 64, 65, 100, 256, 999, 1000, 5000):
        for ns in (1, 2, 0):
            _check(x, w, ns, what=f"fp8={fp8} bs={block_size} w={w} splits={ns}")


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "e4m3"])
@pytest.mark.parametrize("block_size", [16, 64, 128])
def test_recycled_blocks_and_poisoned_tokens_before_the_window(fp8, block_size):
    """Blocks wholly before the window are handed back (-1 in the table and
    NaN in the cache) and the window's first block holds NaN before the
    window starts: nothing of it may reach the output or the error flag."""
    lens = [1000, 777, 64, 65, 3]
    window = 130
    x = _inputs(fp8, batch=len(lens), h_q=32, h_kv=4, seq_lens=lens, block_size=block_size,
                seed=11, device=DEV)
    bt = x.block_table.clone().cpu()
    k = (x.k_codes if fp8 else x.k_cache).clone()
    v = (x.v_codes if fp8 else x.v_cache).clone()
    nan = 0x7F if fp8 else float("nan")
    for b, L in enumerate(lens):
        w0 = oracle.window_start(L, window)
        for t in range(w0):
            blk = int(bt[b, t // block_size])
            k[blk, t % block_size] = nan
            v[blk, t % block_size] = nan
        bt[b, : w0 // block_size] = -1
    bt = bt.to(DEV)
    for ns in (1, 2, 0):
        _check(x, window, ns, what=f"recycled fp8={fp8} bs={block_size} splits={ns}",
               block_table=bt, k=k, v=v)


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "e4m3"])
def test_window_covering_every_sequence_is_bit_identical_to_full_decode(fp8):
    x = _inputs(fp8, batch=4, h_q=16, h_kv=4, seq_lens=[500, 64, 1, 333], block_size=16, seed=5,
                device=DEV)
    for ns in (1, 4, 0):
        if fp8:
            full = da.gqa_decode_fp8kv(x.q, x.k_codes, x.v_codes, x.k_scale, x.v_scale,
                                       x.block_table, x.seq_lens, scale=x.scale,
                                       max_seq_len=x.max_seq_len, num_splits=ns)
        else:
            full = da.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens,
                                 scale=x.scale, max_seq_len=x.max_seq_len, num_splits=ns)
        for w in (500, 10**6):
            win = _run(x, w, ns)
            assert torch.equal(win, full), f"fp8={fp8} splits={ns} w={w}"


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "e4m3"])
def test_sharp_softmax_over_long_sequences(fp8):
    x = _inputs(fp8, batch=3, h_q=32, h_kv=4, seq_lens=("uniform", 2000, 9000), block_size=16,
                seed=9, q_std=4.0, device=DEV)
    for w in (4096, 1500):
        _check(x, w, n_rows=64, what=f"sharp fp8={fp8} w={w}")


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "e4m3"])
def test_llama3_70b_shaped_layer_with_a_4k_window_sampled(fp8):
    x = synth.workload_inputs("llama3_70b_b64_s8k_fp8" if fp8 else "llama3_70b_b64_s8k",
                              device=DEV)
    _check(x, 4096, n_rows=96, what=f"70b w=4096 fp8={fp8}")


def test_invalid_window_is_rejected():
    x = synth.gqa_inputs(batch=1, h_q=8, h_kv=2, seq_lens=[10], block_size=16, device=DEV)
    for w in (0, -5):
        with pytest.raises(da.DecAttnError):
            _run(x, w)


def test_long_context_window_with_the_automatic_plan():
    """B=1 at S=131072 under a 4096-token window: the planner sizes splits
    for the window, not the sequence; sampled rows against the oracle."""
    x = synth.workload_inputs("long_ctx_b1_s128k", device=DEV)
    assert da.gqa_window_plan_splits(1, 64, 8, 131072, 4096, 16) <= \
        da.gqa_plan_splits(1, 64, 8, 4096 + 15)
    _check(x, 4096, n_rows=64, what="S=128k w=4096")
