"""The failure path of every pipeline wait, on the GPU and without a fault:
the library's bounded mbarrier waits run against barriers that nothing ever
completes (decattn_selftest_wait_timeout), give up, set the error flag and let
the CTA leave; the CUDA context stays usable."""
import pytest
import torch

import gqa_mqa_mla_gb300 as da
from gqa_mqa_mla_gb300 import binding, synth

from _parity import compare, gather_rows, oracle_gqa

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("limit_us", [200, 1000, 5000])
def test_bounded_waits_give_up_and_set_the_timeout_flag(limit_us):
    flag, res = binding.selftest_wait_timeout(limit_us)
    assert flag == da.FLAG_TIMEOUT
    assert res[0] == 1, "the waiting thread must give up"
    assert res[4] == 1, "the plain bounded wait must give up too"
    assert res[1] == 1, "a thread watching the abort word must leave with it"
    assert limit_us <= res[2] < limit_us + 100000, res
    assert res[3] < 100 * limit_us, res  # left on the abort word, not on its own 1000x limit


def test_context_is_usable_after_the_waits_gave_up():
    binding.selftest_wait_timeout(500)
    x = synth.workload_inputs("gqa_tiny_b2_s256", device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = da.gqa_decode(x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens, scale=x.scale,
                        max_seq_len=x.max_seq_len, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    ref, _ = oracle_gqa(x)
    compare(gather_rows(out, None), ref, "after selftest")
