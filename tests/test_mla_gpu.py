"""GPU parity of mla_decode (absorbed MLA, tcgen05/TMEM kernel) against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
from gqa_mqa_mla_gb300 import synth

from _parity import compare, gather_rows, oracle_mla, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, num_splits=0, err_flag=None):
    out = da.mla_decode(x.q_abs, x.q_rope, x.cache, x.block_table, x.seq_lens, scale=x.scale,
                        max_seq_len=x.max_seq_len, num_splits=num_splits, err_flag=err_flag)
    torch.cuda.synchronize()
    return out


def _check(x, num_splits=0, n_rows=None, what=""):
    rows = sample_rows(x.batch, 128, n_rows)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(x, num_splits, flag)
    assert int(flag.item()) == 0, f"{what}: error flag {int(flag.item())}"
    ref, _ = oracle_mla(x, rows)
    return compare(gather_rows(out, rows), ref, what)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 0])
def test_small_mla(num_splits):
    x = synth.mla_inputs(batch=2, seq_lens=[200, 77], block_size=64, seed=1, device=DEV)
    _check(x, num_splits, what=f"small splits={num_splits}")


def test_deepseek_v2_shaped_layer_sampled():
    x = synth.workload_inputs("deepseek_v2_mla_b32_s8k", device=DEV)
    _check(x, n_rows=384, what="deepseek-v2 b32 s8k")
    _check(x, num_splits=1, n_rows=128, what="deepseek-v2 b32 s8k splits=1")


@pytest.mark.parametrize("block_size", [8, 16, 32, 64])
def test_block_sizes_and_ragged_lengths(block_size):
    lens = [0, 1, 31, 32, 33, 63, 64, 65, 100, 257]
    x = synth.mla_inputs(batch=len(lens), seq_lens=lens, block_size=block_size, seed=block_size,
                         device=DEV)
    for ns in (1, 3, 0):
        _check(x, ns, what=f"bs={block_size} splits={ns}")
    assert torch.all(_run(x)[0] == 0), "seq_len 0 must give a zero row"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_nan_tail_slots_are_never_read(dtype):
    x = synth.mla_inputs(batch=3, seq_lens=[37, 100, 5], block_size=64, dtype=dtype, seed=3,
                         tail="nan", device=DEV)
    for ns in (1, 2):
        _check(x, ns, what=f"nan tail {dtype}")


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_sharp_softmax_exercises_rescaling(seed):
    x = synth.mla_inputs(batch=3, seq_lens=("uniform", 300, 2000), block_size=64, seed=seed,
                         q_std=8.0, device=DEV)
    _check(x, what=f"sharp seed={seed}")
    _check(x, num_splits=3, what=f"sharp seed={seed} splits=3")


def test_fp16_inputs():
    x = synth.mla_inputs(batch=4, seq_lens=("uniform", 100, 1500), block_size=32, dtype="fp16",
                         seed=7, device=DEV)
    _check(x, what="fp16")


@pytest.mark.parametrize("block_size", [16, 64])
def test_block_permutation_is_bit_exact(block_size):
    # Block size 64 takes the four-chunk copies, 16 one copy per chunk and block.
    x = synth.mla_inputs(batch=3, seq_lens=[500, 333, 64], block_size=block_size, seed=5,
                         table="identity", device=DEV)
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(x.num_blocks, generator=g).to(torch.int32)
    c2 = torch.empty_like(x.cache)
    c2[perm.long().to(DEV)] = x.cache
    bt2 = x.block_table.clone()
    valid = bt2 >= 0
    bt2[valid] = perm.to(DEV)[bt2[valid].long()]
    x2 = synth.MLAInputs(**{**x.__dict__, "cache": c2, "block_table": bt2})
    for ns in (1, 3):
        o1 = _run(x, ns)
        o2 = _run(x2, ns)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_split_counts_agree():
    x = synth.mla_inputs(batch=2, seq_lens=[4096, 2500], block_size=64, seed=9, device=DEV)
    rows = sample_rows(2, 128, 64)
    ref, _ = oracle_mla(x, rows)
    outs = []
    for ns in (1, 2, 7, 32):
        o = _run(x, ns)
        compare(gather_rows(o, rows), ref, f"splits={ns}")
        outs.append(o.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-2


def test_bad_block_id_sets_flag_and_zeroes_only_that_sequence():
    x = synth.mla_inputs(batch=3, seq_lens=[300, 300, 300], block_size=64, seed=4, device=DEV)
    bt = x.block_table.clone()
    bt[1, 2] = -3
    xb = synth.MLAInputs(**{**x.__dict__, "block_table": bt})
    for ns in (1, 2):
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = _run(xb, ns, err_flag=flag)
        assert int(flag.item()) & da.FLAG_BAD_BLOCK
        assert torch.all(out[1] == 0)
        rows = np.array([[b, i] for b in (0, 2) for i in range(0, 128, 5)], np.int32)
        ref, _ = oracle_mla(x, rows)
        compare(gather_rows(out, rows), ref, "unaffected rows")


def test_bad_seq_len_sets_flag():
    x = synth.mla_inputs(batch=2, seq_lens=[128, 128], block_size=64, seed=4, device=DEV)
    sl = x.seq_lens.clone()
    sl[1] = -1
    xb = synth.MLAInputs(**{**x.__dict__, "seq_lens": sl})
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(xb, 1, err_flag=flag)
    assert int(flag.item()) & da.FLAG_BAD_SEQ_LEN
    assert torch.all(out[1] == 0)
    rows = np.array([[0, i] for i in range(128)], np.int32)
    ref, _ = oracle_mla(x, rows)
    compare(gather_rows(out, rows), ref, "unaffected rows")


def test_output_is_deterministic():
    x = synth.mla_inputs(batch=4, seq_lens=("uniform", 500, 3000), block_size=64, seed=2,
                         device=DEV)
    a = _run(x)
    b = _run(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# The balanced schedule lays all sequences' 64-token tiles end to end and
# cuts them into num_splits equal shares, one per CTA pair.  These cases put
# share boundaries at sequence starts, in the middle of sequences, next to
# empty sequences, and leave pairs with nothing to do.
@pytest.mark.parametrize("num_splits", [1, 2, 3, 5, 9, 17, 64, 0])
def test_balanced_shares_ragged_batch(num_splits):
    lens = [0, 130, 64, 1, 700, 0, 257, 65, 3000, 63]
    x = synth.mla_inputs(batch=len(lens), seq_lens=lens, block_size=16, seed=21, device=DEV)
    _check(x, num_splits, n_rows=640, what=f"ragged shares={num_splits}")
    out = _run(x, num_splits)
    assert torch.all(out[0] == 0) and torch.all(out[5] == 0)


@pytest.mark.parametrize("num_splits", [2, 3, 4, 6, 12])
def test_share_boundaries_on_and_off_sequence_starts(num_splits):
    # 6 sequences of 2 tiles: 3 / 6 / 12 shares start on sequence starts,
    # 4 shares cut sequences in the middle.
    x = synth.mla_inputs(batch=6, seq_lens=[128] * 6, block_size=64, seed=22, device=DEV)
    _check(x, num_splits, n_rows=384, what=f"aligned shares={num_splits}")


def test_more_pairs_than_tiles():
    x = synth.mla_inputs(batch=2, seq_lens=[10, 70], block_size=32, seed=23, device=DEV)
    _check(x, 8, what="8 pairs for 3 tiles")


def test_bad_seq_len_between_cut_sequences():
    x = synth.mla_inputs(batch=4, seq_lens=[500, 400, 300, 200], block_size=64, seed=24,
                         device=DEV)
    sl = x.seq_lens.clone()
    sl[1] = x.max_seq_len + 1
    xb = synth.MLAInputs(**{**x.__dict__, "seq_lens": sl})
    for ns in (3, 7):
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = _run(xb, ns, err_flag=flag)
        assert int(flag.item()) & da.FLAG_BAD_SEQ_LEN
        assert torch.all(out[1] == 0)
        rows = np.array([[b, i] for b in (0, 2, 3) for i in range(0, 128, 3)], np.int32)
        ref, _ = oracle_mla(x, rows)
        compare(gather_rows(out, rows), ref, f"rows around a bad length, shares={ns}")


def test_large_batch_of_short_ragged_sequences():
    """256 sequences of 0..600 tokens: most shares hold many whole sequences
    (segment switches on every CTA pair), some sequences are empty."""
    g = torch.Generator().manual_seed(77)
    lens = torch.randint(0, 601, (256,), generator=g).tolist()
    for b in (3, 100, 200):
        lens[b] = 0
    x = synth.mla_inputs(batch=256, seq_lens=lens, block_size=64, seed=78, device=DEV)
    for ns in (0, 76, 13):
        _check(x, ns, n_rows=512, what=f"B=256 ragged splits={ns}")
    out = _run(x)
    assert torch.all(out[3] == 0) and torch.all(out[200] == 0)


def test_single_long_sequence_over_every_pair():
    """One 65536-token sequence cut across all CTA pairs and merged by the combine."""
    x = synth.mla_inputs(batch=1, seq_lens=[65536], block_size=64, seed=79, device=DEV)
    _check(x, 0, n_rows=128, what="B=1 S=64k auto")
    _check(x, 7, n_rows=64, what="B=1 S=64k 7 pairs")


def test_cost_gaps_leave_pairs_without_tiles():
    """Many one-tile sequences and more pairs than the tile count can feed: the
    per-sequence cost gaps of the schedule give some pairs empty slices, and
    zero-length sequences in between must still be zeroed exactly once."""
    lens = [1, 64, 0, 33, 64, 1, 0, 0, 50, 64, 2, 64, 0, 10, 64, 64, 5, 0, 64, 1] * 2
    x = synth.mla_inputs(batch=len(lens), seq_lens=lens, block_size=64, seed=80, device=DEV)
    for ns in (76, 40, 23, 9):
        _check(x, ns, n_rows=len(lens) * 128, what=f"cost gaps pairs={ns}")
    out = _run(x, 76)
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.all(out[b] == 0)
