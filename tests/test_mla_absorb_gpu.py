"""GPU parity of MLA's absorption GEMMs (mla_absorb_q: the query times
W_uk^(i)^T per head; mla_unabsorb_out: the latent output times W_uv^(i) per
head) against the fp64 oracle, and of the whole absorbed decode chain
(absorb, attend over the latent cache, un-absorb) against explicit per-head
reconstruction ("MQA, GQA, and MLA", section 5)."""
import numpy as np
import pytest
import torch

import gqa_mqa_mla_gb300 as da
import oracle
from gqa_mqa_mla_gb300 import synth

from _parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _flat(t):
    return t.float().cpu().numpy().reshape(-1, t.shape[-1])


def _check_pair(x, what):
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    qa = da.mla_absorb_q(x.q_nope, x.w_uk, err_flag=flag)
    out = da.mla_unabsorb_out(x.o_lat, x.w_uv_t, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0, what
    ref_q = oracle.mla_absorb_q(synth.u16(x.q_nope), synth.u16(x.w_uk), dtype=x.dtype)
    ref_o = oracle.mla_unabsorb_out(synth.u16(x.o_lat), synth.u16(x.w_uv_t), dtype=x.dtype)
    compare(_flat(qa), ref_q.reshape(-1, ref_q.shape[-1]), what + " absorb")
    compare(_flat(out), ref_o.reshape(-1, ref_o.shape[-1]), what + " unabsorb")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("batch", [1, 3, 16, 32, 100, 256, 300, 1000])
def test_deepseek_shapes_over_batch_sizes(dtype, batch):
    x = synth.mla_absorb_inputs(batch, dtype=dtype, seed=batch, device=DEV)
    _check_pair(x, f"{dtype} B={batch}")


@pytest.mark.parametrize("heads,d_h,d_c,d_v", [(1, 128, 512, 128), (2, 64, 256, 128),
                                               (16, 192, 384, 256), (128, 128, 128, 128)])
def test_other_widths_and_head_counts(heads, d_h, d_c, d_v):
    x = synth.mla_absorb_inputs(37, heads=heads, d_h=d_h, d_c=d_c, d_v=d_v, seed=heads + d_h,
                                device=DEV)
    _check_pair(x, f"H={heads} d_h={d_h} d_c={d_c} d_v={d_v}")


def test_each_head_uses_its_own_weight():
    """Zeroing one head's weight zeroes exactly that head's outputs."""
    x = synth.mla_absorb_inputs(8, heads=4, seed=3, device=DEV)
    x.w_uk[2].zero_()
    x.w_uv_t[1].zero_()
    qa = da.mla_absorb_q(x.q_nope, x.w_uk)
    out = da.mla_unabsorb_out(x.o_lat, x.w_uv_t)
    torch.cuda.synchronize()
    assert torch.all(qa[:, 2] == 0)
    assert torch.count_nonzero(qa[:, [0, 1, 3]]) > 0.99 * qa[:, [0, 1, 3]].numel()
    assert torch.all(out[:, 1] == 0)
    assert torch.count_nonzero(out[:, [0, 2, 3]]) > 0.99 * out[:, [0, 2, 3]].numel()


def test_absorb_attend_unabsorb_chain_matches_explicit_reconstruction():
    """q_nope -> mla_absorb_q -> mla_decode -> mla_unabsorb_out on the GPU
    against the oracle's reconstruct-then-attend, per sequence."""
    B, S = 3, 200
    x = synth.mla_absorb_inputs(B, seed=5, device=DEV)
    m = synth.mla_inputs(batch=B, seq_lens=[S, 1, 77], block_size=64, seed=6, device=DEV)
    qa = da.mla_absorb_q(x.q_nope, x.w_uk)
    lat = da.mla_decode(qa, m.q_rope, m.cache, m.block_table, m.seq_lens, scale=m.scale,
                        max_seq_len=m.max_seq_len)
    out = da.mla_unabsorb_out(lat, x.w_uv_t)
    torch.cuda.synchronize()
    cache = oracle.bf16_to_double(synth.u16(m.cache))
    bt = m.block_table.cpu().numpy()
    w_uk = oracle.bf16_to_double(synth.u16(x.w_uk))
    w_uv = np.swapaxes(oracle.bf16_to_double(synth.u16(x.w_uv_t)), 1, 2).copy()
    q_nope = oracle.bf16_to_double(synth.u16(x.q_nope))
    q_rope = oracle.bf16_to_double(synth.u16(m.q_rope))
    got = out.float().cpu().numpy()
    for b, L in enumerate(m.seq_lens.tolist()):
        rows = [cache[bt[b, t // 64], t % 64] for t in range(L)]
        c = np.stack([r[:512] for r in rows])
        kr = np.stack([r[512:] for r in rows])
        ref, _ = oracle.mla_explicit(q_nope[b], q_rope[b], c, kr, w_uk, w_uv, scale=m.scale)
        compare(got[b], ref, f"chain b={b}", max_abs=3e-2, mean_abs=3e-3, rel_rms=2e-2)


@pytest.mark.parametrize("batch", [256, 300])
def test_narrow_contraction_with_a_wide_batch_tile(batch):
    """K = 64 (one ring stage) with 256-row batch tiles: the output staging
    area is larger than the ring and must not run into the barriers."""
    x = synth.mla_absorb_inputs(batch, heads=4, d_h=64, d_c=256, d_v=128, seed=batch,
                                device=DEV)
    qa = da.mla_absorb_q(x.q_nope, x.w_uk)
    torch.cuda.synchronize()
    ref = oracle.mla_absorb_q(synth.u16(x.q_nope), synth.u16(x.w_uk), dtype=x.dtype)
    compare(_flat(qa), ref.reshape(-1, ref.shape[-1]), f"K=64 B={batch}")
