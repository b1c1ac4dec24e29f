"""Seeded randomized sweep of mla_decode against the fp64 oracle: batch sizes,
ragged lengths (zero and one-token sequences included), every supported block
size, CTA-pair counts from 1 to one per SM pair (and the planner's), fp16 and
bf16, with NaN in every cache slot past a sequence's end.  The oracle computes
32 random heads of every sequence; the seed fixes every draw, so a failure
names its case."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
from gqa_mqa_mla_gb300 import synth

from _parity import compare, gather_rows, oracle_mla

pytestmark = pytest.mark.gpu

DEV = "cuda"
N_CASES = 32
HEADS_PER_SEQ = 32


def _case(seed):
    rng = np.random.default_rng(5000 + seed)
    batch = int(rng.integers(1, 11))
    bs = int(rng.choice([8, 16, 32, 64]))
    lens = [int(rng.choice([0, 1, rng.integers(2, 70), rng.integers(64, 1500),
                            rng.integers(1500, 4000)])) for _ in range(batch)]
    pairs = int(rng.choice([0, 1, 2, 3, 5, 17, 76]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    heads = np.stack([rng.choice(128, HEADS_PER_SEQ, replace=False) for _ in range(batch)])
    rows = np.array([(b, int(h)) for b in range(batch) for h in heads[b]], dtype=np.int64)
    return dict(batch=batch, bs=bs, lens=lens, pairs=pairs, dtype=dtype), rows


@pytest.mark.parametrize("seed", range(N_CASES))
def test_randomized_mla_case(seed):
    c, rows = _case(seed)
    what = f"seed={seed} {c}"
    # One spare physical block: a batch of empty sequences still has a cache
    # tensor (the ABI requires num_blocks >= 1).
    x = synth.mla_inputs(batch=c["batch"], seq_lens=c["lens"], block_size=c["bs"],
                         dtype=c["dtype"], seed=seed, tail="nan", spare_blocks=1, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = da.mla_decode(x.q_abs, x.q_rope, x.cache, x.block_table, x.seq_lens, scale=x.scale,
                        max_seq_len=x.max_seq_len, num_splits=c["pairs"], err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0, what
    ref, _ = oracle_mla(x, rows)
    compare(gather_rows(out, rows), ref, what)
