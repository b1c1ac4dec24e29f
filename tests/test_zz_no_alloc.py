"""gqa_decode_noalloc: the allocation-free variant of gqa_decode, whose
split-KV scratch is a fixed device array inside the library (for hosts that
cannot call cudaMalloc around a decode call).  Called through the C ABI and
compared with gqa_decode on the same inputs.  Both run the same split plan
through the same kernels, so the outputs must be bit-identical; the calls
alternate between two shapes so that partials left in the shared scratch by
the previous call would show."""
import ctypes

import pytest
import torch

from gqa_mqa_mla_gb300 import binding, synth

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


def _noalloc(x, out, num_splits=0):
    lib = binding.lib()
    fn = lib.gqa_decode_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, P, I, I, I, F, ctypes.POINTER(binding.Launch)]
    fn.restype = I
    L = binding.make_launch(x.batch, x.num_blocks, x.block_size, x.block_table.shape[1],
                            x.max_seq_len, num_splits, binding._DT[x.q.dtype], None, 0, None,
                            torch.cuda.current_stream().cuda_stream)
    return fn(x.q.data_ptr(), x.k_cache.data_ptr(), x.v_cache.data_ptr(),
              x.block_table.data_ptr(), x.seq_lens.data_ptr(), out.data_ptr(), x.h_q, x.h_kv,
              x.d_head, x.scale, ctypes.byref(L))


def _case(batch, seq_len, seed):
    x = synth.gqa_inputs(batch=batch, h_q=64, h_kv=8, seq_lens=seq_len, block_size=16,
                         dtype="bf16", seed=seed, device="cuda")
    splits = binding.gqa_plan_splits(x.batch, x.h_q, x.h_kv, x.max_seq_len)
    assert splits > 1, "the case must use the split-KV scratch"
    assert binding.gqa_workspace_size(x.batch, x.h_q, splits) <= SCRATCH_BYTES
    ref = binding.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens,
                             scale=x.scale, max_seq_len=x.max_seq_len)
    return x, ref


def test_noalloc_matches_gqa_decode_bit_for_bit():
    cases = [_case(1, 32768, 21), _case(4, 8192, 23)]
    torch.cuda.synchronize()
    for _ in range(2):
        for x, ref in cases:
            out = torch.full_like(x.q, float("nan"))
            assert _noalloc(x, out) == binding.DECATTN_OK
            torch.cuda.synchronize()
            assert torch.equal(out, ref)


def test_noalloc_runs_many_requested_splits_on_short_sequences():
    # 64 splits requested on one-tile sequences run as one split (no scratch),
    # although 64 real splits would need far more than the scratch holds.
    x = synth.gqa_inputs(batch=64, h_q=64, h_kv=8, seq_lens=64, block_size=16, dtype="bf16",
                         seed=24, device="cuda")
    assert binding.gqa_workspace_size(x.batch, x.h_q, 64) > SCRATCH_BYTES
    ref = binding.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens,
                             scale=x.scale, max_seq_len=x.max_seq_len, num_splits=1)
    out = torch.full_like(x.q, float("nan"))
    assert _noalloc(x, out, num_splits=64) == binding.DECATTN_OK
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_noalloc_rejects_plans_beyond_its_scratch():
    x = synth.gqa_inputs(batch=8, h_q=64, h_kv=8, seq_lens=8192, block_size=16, dtype="bf16",
                         seed=22, device="cuda")
    need = binding.gqa_workspace_size(x.batch, x.h_q, 64)
    assert need > SCRATCH_BYTES
    out = torch.zeros_like(x.q)
    assert _noalloc(x, out, num_splits=64) == binding.DECATTN_ERR_WORKSPACE
