"""GPU parity of gqa_decode (MHA / GQA / MQA) against the fp64 oracle, through
the C ABI."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
from gqa_mqa_mla_gb300 import synth

from _parity import compare, gather_rows, oracle_gqa, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, num_splits=0, err_flag=None, scale=None):
    out = da.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens,
                        scale=x.scale if scale is None else scale, max_seq_len=x.max_seq_len,
                        num_splits=num_splits, err_flag=err_flag)
    torch.cuda.synchronize()
    return out


def _check(x, num_splits=0, n_rows=None, what=""):
    rows = sample_rows(x.batch, x.h_q, n_rows)
    out = _run(x, num_splits)
    ref, _ = oracle_gqa(x, rows)
    return compare(gather_rows(out, rows), ref, what)


@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 4])
def test_tiny_gqa_fp16_contiguous(num_splits):
    x = synth.workload_inputs("gqa_tiny_b2_s256", device=DEV)
    _check(x, num_splits, what=f"tiny splits={num_splits}")


@pytest.mark.parametrize("name", ["llama31_8b_mha_b16", "llama31_8b_gqa_b16", "llama31_8b_mqa_b16"])
def test_llama31_8b_shaped_sweep(name):
    x = synth.workload_inputs(name, device=DEV)
    _check(x, what=name)


def test_llama3_70b_shaped_large_batch_sampled():
    x = synth.workload_inputs("llama3_70b_b64_s8k", device=DEV)
    _check(x, n_rows=96, what="70b b64 s8k")


@pytest.mark.parametrize("name", ["long_ctx_b1_s128k", "long_ctx_b4_s128k"])
@pytest.mark.parametrize("num_splits", [32, 64, 128])
def test_long_context_split_kv(name, num_splits):
    x = synth.workload_inputs(name, device=DEV)
    _check(x, num_splits, n_rows=24, what=f"{name} splits={num_splits}")


@pytest.mark.parametrize("h_q,h_kv", [(8, 8), (8, 4), (12, 4), (16, 4), (20, 4), (24, 4),
                                      (32, 4), (40, 8), (48, 2), (64, 2), (64, 1)])
def test_group_sizes(h_q, h_kv):
    x = synth.gqa_inputs(batch=3, h_q=h_q, h_kv=h_kv, seq_lens=[300, 1, 129], block_size=16,
                         dtype="bf16", seed=h_q * 7 + h_kv, device=DEV)
    _check(x, what=f"h_q={h_q} h_kv={h_kv}")
    _check(x, num_splits=3, what=f"h_q={h_q} h_kv={h_kv} splits=3")


@pytest.mark.parametrize("h_q,h_kv", [(5, 5), (6, 6), (6, 3), (12, 6), (20, 5), (28, 7),
                                      (36, 12), (40, 10)])
def test_kv_head_counts_not_multiples_of_four(h_q, h_kv):
    """KV-head counts that the launch cannot group four to a cluster: the CTAs
    of a (split, sequence) run in clusters of two (even counts) or alone."""
    x = synth.gqa_inputs(batch=3, h_q=h_q, h_kv=h_kv, seq_lens=[300, 1, 129], block_size=16,
                         dtype="bf16", seed=h_q * 11 + h_kv, device=DEV)
    _check(x, what=f"h_q={h_q} h_kv={h_kv}")
    _check(x, num_splits=3, what=f"h_q={h_q} h_kv={h_kv} splits=3")


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("h_kv", [2, 1])
def test_block_sizes_and_ragged_lengths(block_size, h_kv):
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 700]
    x = synth.gqa_inputs(batch=len(lens), h_q=8, h_kv=h_kv, seq_lens=lens, block_size=block_size,
                         dtype="bf16", seed=block_size, device=DEV)
    for ns in (0, 1, 5):
        _check(x, ns, what=f"bs={block_size} h_kv={h_kv} splits={ns}")
    out = _run(x)
    assert torch.all(out[0] == 0), "seq_len 0 must give a zero row"


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("h_kv", [2, 8])
def test_nan_tail_slots_are_never_read(dtype, h_kv):
    x = synth.gqa_inputs(batch=4, h_q=16, h_kv=h_kv, seq_lens=[37, 100, 5, 250], block_size=32,
                         dtype=dtype, seed=3, tail="nan", device=DEV)
    for ns in (1, 2):
        _check(x, ns, what=f"nan tail {dtype} h_kv={h_kv}")


@pytest.mark.parametrize("h_kv", [2, 8, 1])
def test_block_permutation_is_bit_exact(h_kv):
    """The same logical cache placed in different physical blocks gives
    bit-identical output (same split count)."""
    x = synth.gqa_inputs(batch=3, h_q=16, h_kv=h_kv, seq_lens=[500, 333, 64], block_size=16,
                         dtype="bf16", seed=5, table="identity", device=DEV)
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(x.num_blocks, generator=g).to(torch.int32)
    k2 = torch.empty_like(x.k_cache)
    v2 = torch.empty_like(x.v_cache)
    k2[perm.long().to(DEV)] = x.k_cache
    v2[perm.long().to(DEV)] = x.v_cache
    bt2 = x.block_table.clone()
    valid = bt2 >= 0
    bt2[valid] = perm.to(DEV)[bt2[valid].long()]
    for ns in (1, 3):
        o1 = _run(x, ns)
        x2 = synth.GQAInputs(**{**x.__dict__, "k_cache": k2, "v_cache": v2, "block_table": bt2})
        o2 = _run(x2, ns)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_split_counts_agree():
    x = synth.gqa_inputs(batch=2, h_q=64, h_kv=8, seq_lens=[8192, 5000], block_size=16,
                         dtype="bf16", seed=9, device=DEV)
    rows = sample_rows(2, 64, 32)
    ref, _ = oracle_gqa(x, rows)
    outs = []
    for ns in (1, 2, 7, 32, 128):
        o = _run(x, ns)
        compare(gather_rows(o, rows), ref, f"splits={ns}")
        outs.append(o.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-2


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("h_kv", [8, 2])
def test_sharp_softmax(seed, h_kv):
    """Q x 8 makes the softmax peaky, exercising the running-max rescale."""
    x = synth.gqa_inputs(batch=4, h_q=32, h_kv=h_kv, seq_lens=("uniform", 200, 3000),
                         block_size=16, dtype="bf16", seed=seed, q_std=8.0, device=DEV)
    _check(x, what=f"sharp seed={seed}")
    _check(x, num_splits=4, what=f"sharp seed={seed} splits=4")


def test_bad_block_id_sets_flag_and_zeroes_only_that_sequence():
    x = synth.gqa_inputs(batch=3, h_q=8, h_kv=2, seq_lens=[100, 100, 100], block_size=16,
                         dtype="bf16", seed=4, device=DEV)
    bt = x.block_table.clone()
    bt[1, 3] = x.num_blocks + 5  # out of range
    xb = synth.GQAInputs(**{**x.__dict__, "block_table": bt})
    for ns in (1, 2):
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = _run(xb, ns, err_flag=flag)
        assert int(flag.item()) & da.FLAG_BAD_BLOCK
        assert torch.all(out[1] == 0)
        rows = np.array([[b, i] for b in (0, 2) for i in range(8)], np.int32)
        ref, _ = oracle_gqa(x, rows)
        compare(gather_rows(out, rows), ref, "unaffected rows")


def test_bad_seq_len_sets_flag():
    x = synth.gqa_inputs(batch=2, h_q=8, h_kv=8, seq_lens=[64, 64], block_size=16, dtype="bf16",
                         seed=4, device=DEV)
    sl = x.seq_lens.clone()
    sl[0] = 10_000  # beyond max_seq_len
    xb = synth.GQAInputs(**{**x.__dict__, "seq_lens": sl})
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(xb, 1, err_flag=flag)
    assert int(flag.item()) & da.FLAG_BAD_SEQ_LEN
    assert torch.all(out[0] == 0)
    rows = np.array([[1, i] for i in range(8)], np.int32)
    ref, _ = oracle_gqa(x, rows)
    compare(gather_rows(out, rows), ref, "unaffected rows")


def test_clean_run_leaves_flag_zero():
    x = synth.workload_inputs("llama31_8b_gqa_b16", device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    _run(x, err_flag=flag)
    assert int(flag.item()) == 0


def test_output_is_deterministic():
    x = synth.workload_inputs("llama31_8b_gqa_b16", device=DEV)
    a = _run(x)
    b = _run(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------- wide groups
# More than 16 query heads per KV head run on the tcgen05 kernel: ragged and
# empty lengths, many splits (most of them empty for short sequences), bad
# block ids and lengths.

WIDE_LENS = [0, 1, 63, 64, 65, 700, 0, 4097, 130, 2000, 64 * 7 + 5, 3]


@pytest.mark.parametrize("h_q,h_kv", [(32, 1), (64, 1), (64, 2), (48, 2), (40, 2), (68, 4)])
@pytest.mark.parametrize("num_splits", [0, 2, 5, 64])
def test_wide_groups_ragged_and_empty(h_q, h_kv, num_splits):
    if h_q % h_kv or h_q // h_kv > 64:
        pytest.skip("not a supported group")
    x = synth.gqa_inputs(batch=len(WIDE_LENS), h_q=h_q, h_kv=h_kv, seq_lens=WIDE_LENS,
                         block_size=16, dtype="bf16", seed=h_q + h_kv, device=DEV)
    out = _run(x, num_splits)
    rows = sample_rows(x.batch, x.h_q, None)
    ref, _ = oracle_gqa(x, rows)
    compare(gather_rows(out, rows), ref, f"wide h_q={h_q} h_kv={h_kv} splits={num_splits}")
    # empty sequences: zero rows
    for b, n in enumerate(WIDE_LENS):
        if n == 0:
            assert torch.all(out[b] == 0)


@pytest.mark.parametrize("num_splits", [1, 3, 40])
def test_wide_groups_bad_block_and_bad_length(num_splits):
    lens = [300, 300, 300, 2000, 64]
    x = synth.gqa_inputs(batch=5, h_q=64, h_kv=2, seq_lens=lens, block_size=16, dtype="bf16",
                         seed=8, device=DEV)
    bt = x.block_table.clone()
    bt[1, 3] = x.num_blocks + 5  # out of range
    sl = x.seq_lens.clone()
    sl[4] = 10_000  # beyond max_seq_len
    xb = synth.GQAInputs(**{**x.__dict__, "block_table": bt, "seq_lens": sl})
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(xb, num_splits, err_flag=flag)
    assert int(flag.item()) & da.FLAG_BAD_BLOCK
    assert int(flag.item()) & da.FLAG_BAD_SEQ_LEN
    assert torch.all(out[1] == 0) and torch.all(out[4] == 0)
    rows = np.array([[b, i] for b in (0, 2, 3) for i in range(64)], np.int32)
    ref, _ = oracle_gqa(x, rows)
    compare(gather_rows(out, rows), ref, "unaffected rows")


def test_wide_groups_deterministic_for_every_split_count():
    """Two calls give identical bits, and every split count matches the oracle."""
    x = synth.gqa_inputs(batch=6, h_q=64, h_kv=1, seq_lens=("uniform", 1, 6000), block_size=16,
                         dtype="bf16", seed=21, device=DEV)
    rows = sample_rows(x.batch, x.h_q, 64)
    ref, _ = oracle_gqa(x, rows)
    for ns in (1, 2, 9, 64, 256):
        o1 = _run(x, ns)
        o2 = _run(x, ns)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        compare(gather_rows(o1, rows), ref, f"wide splits={ns}")


@pytest.mark.parametrize("name", ["wide_g32_b64_s8k", "wide_g64_mqa_b128_s8k"])
def test_wide_group_workloads_sampled(name):
    """The bench's wide-group workloads at full size and planned splits."""
    x = synth.workload_inputs(name, device=DEV)
    _check(x, n_rows=64, what=name)
