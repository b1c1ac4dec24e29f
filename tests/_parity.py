"""Shared helpers for the GPU parity tests: run the C-ABI path, run the fp64
oracle on the same bytes, compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gqa_mqa_mla_gb300 import synth

# Tolerances for fp16/bf16 inputs with fp32 accumulation (outputs rounded to
# the 16-bit type): max |gpu - oracle| and mean |gpu - oracle| over the
# compared elements, plus a relative-RMS bound (error RMS / oracle RMS) that
# stays meaningful when the outputs themselves are small (long flat softmax).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
REL_RMS = 1e-2


def sample_rows(batch: int, heads: int, n: int | None, seed: int = 0):
    """All (b, i) pairs, or n of them drawn without replacement (always
    including the first and the last row)."""
    total = batch * heads
    if n is None or n >= total:
        return None
    rng = np.random.default_rng(seed + 12345)
    idx = np.unique(np.concatenate([[0, total - 1], rng.choice(total, n - 2, replace=False)]))
    return np.stack([idx // heads, idx % heads], axis=1).astype(np.int32)


def oracle_gqa(x: synth.GQAInputs, rows=None, scale=None):
    return oracle.gqa_decode(synth.u16(x.q), synth.u16(x.k_cache), synth.u16(x.v_cache),
                             x.block_table.cpu().numpy(), x.seq_lens.cpu().numpy(), dtype=x.dtype,
                             scale=x.scale if scale is None else scale, rows=rows)


def oracle_gqa_fp8(x: synth.GQAFp8Inputs, rows=None, scale=None):
    return oracle.gqa_decode_fp8kv(synth.u16(x.q), x.k_codes.cpu().numpy(), x.v_codes.cpu().numpy(),
                                   x.k_scale.cpu().double().numpy(), x.v_scale.cpu().double().numpy(),
                                   x.block_table.cpu().numpy(), x.seq_lens.cpu().numpy(),
                                   q_dtype=x.dtype, scale=x.scale if scale is None else scale,
                                   rows=rows)


def oracle_gqa_window(x: synth.GQAInputs, window: int, rows=None, block_table=None,
                      k_cache=None, v_cache=None):
    bt = x.block_table if block_table is None else block_table
    return oracle.gqa_decode_window(synth.u16(x.q), synth.u16(x.k_cache if k_cache is None else k_cache),
                                    synth.u16(x.v_cache if v_cache is None else v_cache),
                                    bt.cpu().numpy(), x.seq_lens.cpu().numpy(), dtype=x.dtype,
                                    scale=x.scale, window=window, rows=rows)


def oracle_gqa_fp8_window(x: synth.GQAFp8Inputs, window: int, rows=None, block_table=None,
                          k_codes=None, v_codes=None):
    bt = x.block_table if block_table is None else block_table
    kc = x.k_codes if k_codes is None else k_codes
    vc = x.v_codes if v_codes is None else v_codes
    return oracle.gqa_decode_fp8kv_window(synth.u16(x.q), kc.cpu().numpy(), vc.cpu().numpy(),
                                          x.k_scale.cpu().double().numpy(),
                                          x.v_scale.cpu().double().numpy(), bt.cpu().numpy(),
                                          x.seq_lens.cpu().numpy(), q_dtype=x.dtype,
                                          scale=x.scale, window=window, rows=rows)


def oracle_mla(x: synth.MLAInputs, rows=None):
    return oracle.mla_decode(synth.u16(x.q_abs), synth.u16(x.q_rope), synth.u16(x.cache),
                             x.block_table.cpu().numpy(), x.seq_lens.cpu().numpy(), dtype=x.dtype,
                             scale=x.scale, rows=rows)


def gather_rows(out: torch.Tensor, rows) -> np.ndarray:
    o = out.float().cpu().numpy()
    if rows is None:
        return o.reshape(-1, o.shape[-1])
    return o[rows[:, 0], rows[:, 1]]


def compare(got: np.ndarray, ref: np.ndarray, what: str = "", max_abs=MAX_ABS, mean_abs=MEAN_ABS,
            rel_rms=REL_RMS) -> dict:
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    err = np.abs(got - ref)
    rms_ref = float(np.sqrt(np.mean(ref * ref)))
    stats = {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
             "rel_rms": float(np.sqrt(np.mean(err * err)) / rms_ref) if rms_ref > 0 else 0.0}
    assert stats["max_abs"] <= max_abs, f"{what}: {stats}"
    assert stats["mean_abs"] <= mean_abs, f"{what}: {stats}"
    if rms_ref > 0:
        assert stats["rel_rms"] <= rel_rms, f"{what}: {stats}"
    return stats
