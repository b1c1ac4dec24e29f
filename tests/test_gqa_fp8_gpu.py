"""GPU parity of gqa_decode_fp8kv (GQA / MHA / MQA over an 8-bit e4m3 KV cache
with per-KV-head scales) against the fp64 oracle (dequantise, then the plain
GQA definition), through the C ABI."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
from gqa_mqa_mla_gb300 import synth

from _parity import compare, gather_rows, oracle_gqa_fp8, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, num_splits=0, err_flag=None, block_table=None, seq_lens=None, k_codes=None):
    out = da.gqa_decode_fp8kv(x.q, x.k_codes if k_codes is None else k_codes, x.v_codes,
                              x.k_scale, x.v_scale,
                              x.block_table if block_table is None else block_table,
                              x.seq_lens if seq_lens is None else seq_lens, scale=x.scale,
                              max_seq_len=x.max_seq_len, num_splits=num_splits, err_flag=err_flag)
    torch.cuda.synchronize()
    return out


def _check(x, num_splits=0, n_rows=None, what=""):
    rows = sample_rows(x.batch, x.h_q, n_rows)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(x, num_splits, err_flag=flag)
    assert int(flag.item()) == 0, f"{what}: error flag {int(flag.item())}"
    ref, _ = oracle_gqa_fp8(x, rows)
    return compare(gather_rows(out, rows), ref, what)


@pytest.mark.parametrize("h_q,h_kv", [(8, 8), (8, 2), (16, 4), (32, 8), (32, 1), (24, 4),
                                      (48, 2), (64, 8), (64, 1)])
@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_group_sizes_and_splits(h_q, h_kv, num_splits):
    x = synth.gqa_fp8_inputs(batch=3, h_q=h_q, h_kv=h_kv, seq_lens=[300, 1, 129], block_size=16,
                             seed=h_q * 5 + h_kv, device=DEV)
    _check(x, num_splits, what=f"h_q={h_q} h_kv={h_kv} splits={num_splits}")


@pytest.mark.parametrize("h_q,h_kv", [(5, 5), (6, 3), (20, 5), (12, 6), (28, 7)])
def test_odd_kv_head_counts(h_q, h_kv):
    """Odd KV-head counts launch without clusters; even ones in clusters of two."""
    x = synth.gqa_fp8_inputs(batch=3, h_q=h_q, h_kv=h_kv, seq_lens=[300, 1, 129], block_size=16,
                             seed=h_q * 13 + h_kv, device=DEV)
    for ns in (1, 3):
        _check(x, ns, what=f"h_q={h_q} h_kv={h_kv} splits={ns}")


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128, 256])
def test_block_sizes_and_ragged_lengths(block_size):
    lens = [0, 1, 31, 63, 64, 65, 100, 257, 1000]
    x = synth.gqa_fp8_inputs(batch=len(lens), h_q=16, h_kv=2, seq_lens=lens,
                             block_size=block_size, seed=block_size, device=DEV)
    for ns in (1, 2, 0):
        _check(x, ns, what=f"bs={block_size} splits={ns}")
    assert torch.all(_run(x)[0] == 0), "seq_len 0 must give a zero row"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_nan_codes_in_tail_slots_are_never_read(dtype):
    x = synth.gqa_fp8_inputs(batch=3, h_q=8, h_kv=1, seq_lens=[37, 100, 5], block_size=64,
                             dtype=dtype, seed=3, tail="nan", device=DEV)
    for ns in (1, 2):
        _check(x, ns, what=f"nan tail {dtype}")
    xm = synth.gqa_fp8_inputs(batch=3, h_q=4, h_kv=4, seq_lens=[37, 100, 5], block_size=16,
                              dtype=dtype, seed=4, tail="nan", device=DEV)
    _check(xm, what=f"nan tail mha {dtype}")


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_sharp_softmax(seed):
    x = synth.gqa_fp8_inputs(batch=2, h_q=32, h_kv=4, seq_lens=("uniform", 200, 3000),
                             block_size=16, seed=seed, q_std=4.0, device=DEV)
    _check(x, what=f"sharp seed={seed}")


def test_llama3_70b_shaped_layer_sampled():
    x = synth.workload_inputs("llama3_70b_b64_s8k_fp8", device=DEV)
    _check(x, n_rows=96, what="70b fp8 b64 s8k")


def test_scales_are_applied_per_kv_head():
    # Doubling one KV head's V scale doubles exactly the outputs of its query
    # heads; K scales change only the heads that read them.
    x = synth.gqa_fp8_inputs(batch=2, h_q=8, h_kv=2, seq_lens=[300, 77], block_size=16, seed=9,
                             device=DEV)
    base = _run(x).float()
    v2 = x.v_scale.clone()
    v2[1] *= 2
    x2 = synth.GQAFp8Inputs(**{**x.__dict__, "v_scale": v2})
    out = _run(x2).float()
    assert torch.equal(out[:, :4], base[:, :4])
    torch.testing.assert_close(out[:, 4:], 2 * base[:, 4:], rtol=1e-2, atol=1e-3)
    k2 = x.k_scale.clone()
    k2[0] *= 3
    x3 = synth.GQAFp8Inputs(**{**x.__dict__, "k_scale": k2})
    out3 = _run(x3).float()
    assert torch.equal(out3[:, 4:], base[:, 4:])
    assert not torch.equal(out3[:, :4], base[:, :4])
    _check(x3, what="k scale x3")


def test_block_permutation_is_bit_exact():
    x = synth.gqa_fp8_inputs(batch=3, h_q=16, h_kv=4, seq_lens=[500, 333, 64], block_size=16,
                             seed=5, table="identity", device=DEV)
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(x.num_blocks, generator=g).to(torch.int32)
    k2 = torch.empty_like(x.k_codes)
    v2 = torch.empty_like(x.v_codes)
    k2[perm.long().to(DEV)] = x.k_codes
    v2[perm.long().to(DEV)] = x.v_codes
    bt2 = x.block_table.clone()
    valid = bt2 >= 0
    bt2[valid] = perm.to(DEV)[bt2[valid].long()]
    x2 = synth.GQAFp8Inputs(**{**x.__dict__, "k_codes": k2, "v_codes": v2, "block_table": bt2})
    for ns in (1, 3):
        o1 = _run(x, ns)
        o2 = _run(x2, ns)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_bad_block_and_bad_seq_len_set_flags_and_zero_rows():
    x = synth.gqa_fp8_inputs(batch=3, h_q=16, h_kv=2, seq_lens=[300, 300, 300], block_size=16,
                             seed=4, device=DEV)
    bt = x.block_table.clone()
    bt[1, 2] = x.num_blocks + 7
    for ns in (1, 2):
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = _run(x, ns, err_flag=flag, block_table=bt)
        assert int(flag.item()) & da.FLAG_BAD_BLOCK
        assert torch.all(out[1] == 0)
        rows = np.array([[b, i] for b in (0, 2) for i in range(16)], np.int32)
        ref, _ = oracle_gqa_fp8(x, rows)
        compare(gather_rows(out, rows), ref, "unaffected rows")
    sl = x.seq_lens.clone()
    sl[2] = -5
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(x, 1, err_flag=flag, seq_lens=sl)
    assert int(flag.item()) & da.FLAG_BAD_SEQ_LEN
    assert torch.all(out[2] == 0)


def test_output_is_deterministic():
    x = synth.gqa_fp8_inputs(batch=4, h_q=32, h_kv=4, seq_lens=("uniform", 500, 3000),
                             block_size=16, seed=2, device=DEV)
    a = _run(x)
    b = _run(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fp8_path_matches_16bit_path_on_the_same_values():
    # The same cache stored as bf16 (every e4m3 value is exact in bf16) with
    # the scales folded in must give nearly the same output through gqa_decode.
    x = synth.gqa_fp8_inputs(batch=2, h_q=32, h_kv=8, seq_lens=[700, 1500], block_size=16,
                             seed=7, device=DEV)
    kv = x.k_codes.view(torch.float8_e4m3fn).float() * x.k_scale[None, None, :, None]
    vv = x.v_codes.view(torch.float8_e4m3fn).float() * x.v_scale[None, None, :, None]
    o16 = da.gqa_decode(x.q, kv.to(torch.bfloat16), vv.to(torch.bfloat16), x.block_table,
                        x.seq_lens, scale=x.scale, max_seq_len=x.max_seq_len)
    o8 = _run(x)
    torch.testing.assert_close(o8.float(), o16.float(), rtol=2e-2, atol=1e-2)


# Groups wider than 16 query heads per KV head run on the tensor-core kernel
# that converts each landed e4m3 tile to f16 in shared memory.

@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("h_q,h_kv", [(64, 2), (40, 2), (64, 1)])
def test_wide_groups_block_sizes_and_ragged_lengths(block_size, h_q, h_kv):
    lens = [0, 1, 63, 64, 65, 257, 1000]
    x = synth.gqa_fp8_inputs(batch=len(lens), h_q=h_q, h_kv=h_kv, seq_lens=lens,
                             block_size=block_size, seed=block_size + h_q, device=DEV)
    for ns in (1, 3, 0):
        _check(x, ns, what=f"wide h_q={h_q} h_kv={h_kv} bs={block_size} splits={ns}")
    assert torch.all(_run(x)[0] == 0), "seq_len 0 must give a zero row"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_wide_groups_nan_tails_and_sharp_softmax(dtype):
    x = synth.gqa_fp8_inputs(batch=3, h_q=32, h_kv=1, seq_lens=[37, 100, 5], block_size=64,
                             dtype=dtype, seed=13, tail="nan", device=DEV)
    for ns in (1, 2):
        _check(x, ns, what=f"wide nan tail {dtype}")
    xs = synth.gqa_fp8_inputs(batch=2, h_q=64, h_kv=2, seq_lens=("uniform", 200, 3000),
                              block_size=16, dtype=dtype, seed=14, q_std=4.0, device=DEV)
    _check(xs, what=f"wide sharp {dtype}")


@pytest.mark.parametrize("num_splits", [1, 3, 40])
def test_wide_groups_bad_block_and_bad_length(num_splits):
    x = synth.gqa_fp8_inputs(batch=5, h_q=64, h_kv=2, seq_lens=[300, 300, 300, 2000, 64],
                             block_size=16, seed=8, device=DEV)
    bt = x.block_table.clone()
    bt[1, 3] = x.num_blocks + 5
    sl = x.seq_lens.clone()
    sl[4] = 10_000
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(x, num_splits, err_flag=flag, block_table=bt, seq_lens=sl)
    assert int(flag.item()) & da.FLAG_BAD_BLOCK
    assert int(flag.item()) & da.FLAG_BAD_SEQ_LEN
    assert torch.all(out[1] == 0) and torch.all(out[4] == 0)
    rows = np.array([[b, i] for b in (0, 2, 3) for i in range(64)], np.int32)
    ref, _ = oracle_gqa_fp8(x, rows)
    compare(gather_rows(out, rows), ref, "unaffected rows")


def test_wide_groups_deterministic_for_every_split_count():
    x = synth.gqa_fp8_inputs(batch=6, h_q=64, h_kv=1, seq_lens=("uniform", 1, 6000),
                             block_size=16, seed=21, device=DEV)
    rows = sample_rows(x.batch, x.h_q, 64)
    ref, _ = oracle_gqa_fp8(x, rows)
    for ns in (1, 2, 9, 64, 256):
        o1 = _run(x, ns)
        o2 = _run(x, ns)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        compare(gather_rows(o1, rows), ref, f"wide splits={ns}")


def test_wide_group_full_size_sampled():
    """32 query heads per KV head at B = 64, S = 8192, planned splits."""
    x = synth.gqa_fp8_inputs(batch=64, h_q=64, h_kv=2, seq_lens=8192, block_size=16,
                             seed=66, device=DEV)
    _check(x, n_rows=64, what="wide fp8 b64 64/2 s8k")


def test_wide_mqa_workload_sampled():
    """The bench's MQA-64 workload over an e4m3 cache at full size."""
    x = synth.workload_inputs("wide_g64_mqa_b128_s8k_fp8", device=DEV)
    _check(x, n_rows=64, what="wide_g64_mqa_b128_s8k_fp8")
