"""Seeded randomized sweep of the GQA decode calls against the fp64 oracle:
query/KV head counts, block sizes, ragged lengths (zero included), split
counts, sliding windows, 16-bit and e4m3 caches, fp16 and bf16.  Each case is
small; the seed fixes every draw, so a failure names its case."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
from gqa_mqa_mla_gb300 import synth

from _parity import (compare, gather_rows, oracle_gqa, oracle_gqa_fp8, oracle_gqa_fp8_window,
                     oracle_gqa_window)

pytestmark = pytest.mark.gpu

DEV = "cuda"
N_CASES = 48


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    h_kv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 24, 32, 48, 64]))
    batch = int(rng.integers(1, 7))
    bs = int(rng.choice([8, 16, 32, 64, 128, 256]))
    lens = [int(rng.choice([0, rng.integers(1, 70), rng.integers(64, 900)])) for _ in range(batch)]
    fp8 = bool(rng.integers(0, 2))
    dtype = str(rng.choice(["bf16", "fp16"]))
    splits = int(rng.choice([0, 1, 2, 3, 7]))
    window = int(rng.choice([0, 1, 33, 64, 200])) or None
    return dict(h_kv=h_kv, h_q=h_kv * group, batch=batch, bs=bs, lens=lens, fp8=fp8,
                dtype=dtype, splits=splits, window=window)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_randomized_case(seed):
    c = _case(seed)
    what = f"seed={seed} {c}"
    # One spare physical block: a batch of empty sequences still has a cache
    # tensor (the ABI requires num_blocks >= 1).
    kw = dict(batch=c["batch"], h_q=c["h_q"], h_kv=c["h_kv"], seq_lens=c["lens"],
              block_size=c["bs"], dtype=c["dtype"], seed=seed, tail="nan", spare_blocks=1,
              device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    if c["fp8"]:
        x = synth.gqa_fp8_inputs(**kw)
        out = da.gqa_decode_fp8kv(x.q, x.k_codes, x.v_codes, x.k_scale, x.v_scale,
                                  x.block_table, x.seq_lens, scale=x.scale,
                                  max_seq_len=x.max_seq_len, num_splits=c["splits"],
                                  err_flag=flag, window=c["window"])
        ref, _ = (oracle_gqa_fp8(x) if c["window"] is None
                  else oracle_gqa_fp8_window(x, c["window"]))
    else:
        x = synth.gqa_inputs(**kw)
        out = da.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens,
                            scale=x.scale, max_seq_len=x.max_seq_len,
                            num_splits=c["splits"], err_flag=flag, window=c["window"])
        ref, _ = oracle_gqa(x) if c["window"] is None else oracle_gqa_window(x, c["window"])
    torch.cuda.synchronize()
    assert int(flag.item()) == 0, what
    compare(gather_rows(out, None), ref, what)
