"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/decattn.h declares, and its host-side argument checks return
the documented statuses before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

import oracle
from gqa_mqa_mla_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decattn.h")

FAKE = 0x100000  # an aligned address that is never dereferenced by the host checks


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"gqa_decode", "mla_decode", "decattn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in decattn.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.decattn_version() >= 100
    for st in (0, -1, -2, -3, -4, 7):
        assert binding.status_string(st)


GOLDEN = os.path.join(ROOT, "tests", "golden", "cache_sizes.txt")


def test_library_cache_size_formulas_match_the_oracle_and_pages(lib):
    with open(GOLDEN) as f:
        rows = [l.split("|")[0].split() for l in f if l.strip() and not l.startswith("#")]
    for tok in rows:
        kind = tok[1]
        n_layers, a, b, nbytes = (int(x) for x in tok[2:6])
        if kind == "kv":
            assert binding.kv_bytes_per_token(n_layers, a, b, nbytes) == \
                oracle.kv_bytes_per_token(n_layers, a, b, nbytes)
        else:
            assert binding.mla_bytes_per_token(n_layers, a, b, nbytes) == \
                oracle.mla_bytes_per_token(n_layers, a, b, nbytes)
    assert binding.kv_bytes_per_token(80, 64, 128, 2) == 2_621_440
    assert binding.mla_bytes_per_token(1, 512, 64, 1) == 576
    assert binding.kv_bytes_per_token(-1, 1, 1, 1) < 0


def test_workspace_sizes(lib):
    assert binding.gqa_workspace_size(4, 32, 1) == 0
    ws = binding.gqa_workspace_size(4, 32, 8)
    assert ws >= 4 * 32 * 8 * 128 * 4 + 4 * 32 * 8 * 4
    assert binding.mla_workspace_size(2, 3) >= 2 * 128 * 3 * 512 * 4 + 2 * 128 * 3 * 4
    assert binding.gqa_workspace_size(4, 32, 0) == 0
    assert binding.gqa_workspace_size(4, 32, binding.MAX_SPLITS + 1) == 0


def test_planner_is_bounded_and_spreads_long_sequences(lib):
    for B, h_q, h_kv, S in [(1, 64, 8, 131072), (4, 64, 8, 131072), (64, 64, 8, 8192),
                            (16, 32, 32, 4096), (2, 8, 2, 256), (1, 8, 8, 0)]:
        ns = binding.gqa_plan_splits(B, h_q, h_kv, S, num_sms=152)
        assert 1 <= ns <= binding.MAX_SPLITS
        assert ns <= max(1, -(-S // 64))
    # one short-batch long sequence must be split across many CTAs
    assert binding.gqa_plan_splits(1, 64, 8, 131072, num_sms=152) >= 16
    assert 1 <= binding.mla_plan_splits(32, 8192, num_sms=152) <= binding.MAX_SPLITS
    assert binding.mla_plan_splits(1, 65536, num_sms=152) >= 16


def test_fp8_planner_fills_one_wave_of_four_ctas_per_sm_up_to_8_heads_per_kv_head(lib):
    # 512 (sequence, KV head) units of the 70B-shaped layer fit the 608 slots
    # of four CTAs per SM: one split; 128 units: four splits (0.84 of a wave).
    assert binding.gqa_fp8_plan_splits(64, 64, 8, 8192, num_sms=152) == 1
    assert binding.gqa_fp8_plan_splits(16, 64, 8, 8192, num_sms=152) == 4
    # wider groups keep two CTAs per SM and about two waves
    assert binding.gqa_fp8_plan_splits(64, 128, 8, 8192, num_sms=152) == 1
    assert binding.gqa_fp8_plan_splits(16, 256, 8, 8192, num_sms=152) == 2


def _launch(**kw):
    d = dict(batch=2, num_blocks=64, block_size=16, max_blocks_per_seq=16, max_seq_len=256,
             num_splits=1, dtype=binding.DECATTN_BF16, workspace=None, workspace_bytes=0,
             err_flag=None, stream=None)
    d.update(kw)
    return binding.Launch(**d)


def _gqa(lib, L, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, out=FAKE, h_q=8, h_kv=2, d=128,
         scale=0.088):
    return lib.gqa_decode(q, k, v, bt, sl, out, h_q, h_kv, d, scale,
                          None if L is None else ctypes.byref(L))


def _mla(lib, L, qa=FAKE, qr=FAKE, c=FAKE, bt=FAKE, sl=FAKE, out=FAKE, scale=0.07):
    return lib.mla_decode(qa, qr, c, bt, sl, out, scale, None if L is None else ctypes.byref(L))


@pytest.mark.parametrize("case,expect", [
    (dict(L=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(q=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(k=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(out=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(h_q=9, h_kv=2), binding.DECATTN_ERR_INVALID_ARG),
    (dict(h_kv=0), binding.DECATTN_ERR_INVALID_ARG),
    (dict(d=64), binding.DECATTN_ERR_UNSUPPORTED),
    (dict(h_q=256, h_kv=2), binding.DECATTN_ERR_UNSUPPORTED),
    (dict(q=FAKE + 2), binding.DECATTN_ERR_INVALID_ARG),
    (dict(bt=FAKE + 2), binding.DECATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(batch=0)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(dtype=5)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(block_size=12)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(block_size=4)), binding.DECATTN_ERR_UNSUPPORTED),
    (dict(L=dict(max_seq_len=257)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(num_splits=-1)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(num_splits=binding.MAX_SPLITS + 1)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(num_splits=4)), binding.DECATTN_ERR_WORKSPACE),
    (dict(L=dict(num_splits=4, workspace=FAKE, workspace_bytes=100)),
     binding.DECATTN_ERR_WORKSPACE),
    (dict(L=dict(workspace=FAKE + 4)), binding.DECATTN_ERR_INVALID_ARG),
])
def test_gqa_host_checks(lib, case, expect):
    case = dict(case)
    L = case.pop("L", {})
    L = None if L is None else _launch(**L)
    assert _gqa(lib, L, **case) == expect


def _gqa_noalloc(lib, L, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, out=FAKE, h_q=8, h_kv=2,
                 d=128, scale=0.088):
    fn = lib.gqa_decode_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, P, I, I, I, F, ctypes.POINTER(binding.Launch)]
    fn.restype = I
    return fn(q, k, v, bt, sl, out, h_q, h_kv, d, scale, None if L is None else ctypes.byref(L))


# The no-allocation variant runs gqa_decode's argument checks before its
# scratch-size check, so every bad argument gets gqa_decode's status.
@pytest.mark.parametrize("case,expect", [
    (dict(L=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(q=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(h_q=9, h_kv=2), binding.DECATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(num_splits=-1)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(max_seq_len=257)), binding.DECATTN_ERR_INVALID_ARG),
    # a plan far beyond the 8 MiB scratch, with an unsupported head size:
    # the head size decides the status
    (dict(d=64, h_q=64, h_kv=8, L=dict(batch=64, max_seq_len=8192, max_blocks_per_seq=512,
                                       num_blocks=1 << 15, num_splits=64)),
     binding.DECATTN_ERR_UNSUPPORTED),
    (dict(h_q=256, h_kv=2, L=dict(batch=64, max_seq_len=8192, max_blocks_per_seq=512,
                                  num_blocks=1 << 15, num_splits=64)),
     binding.DECATTN_ERR_UNSUPPORTED),
    # the same plan with valid arguments needs 135 MB of scratch
    (dict(h_q=64, h_kv=8, L=dict(batch=64, max_seq_len=8192, max_blocks_per_seq=512,
                                 num_blocks=1 << 15, num_splits=64)),
     binding.DECATTN_ERR_WORKSPACE),
])
def test_gqa_noalloc_host_checks(lib, case, expect):
    case = dict(case)
    L = case.pop("L", {})
    L = None if L is None else _launch(**L)
    assert _gqa_noalloc(lib, L, **case) == expect


# This call passes every host check, so on a machine with a GPU it would
# launch the kernel on the fake addresses: it runs only where no GPU is
# visible (the GPU side of the same plan, on real buffers, is
# test_zz_no_alloc.py::test_noalloc_runs_many_requested_splits_on_short_sequences).
@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake device addresses")
def test_gqa_noalloc_sizes_scratch_by_the_splits_it_runs(lib):
    # 64 splits requested on one-tile sequences run as a single split, which
    # needs no scratch: the call must not be refused for scratch (with no GPU
    # it reaches the device lookup and reports a CUDA status instead).
    L = _launch(batch=64, max_seq_len=64, max_blocks_per_seq=4, num_blocks=256, num_splits=64)
    st = _gqa_noalloc(lib, L, h_q=64, h_kv=8)
    assert st != binding.DECATTN_ERR_WORKSPACE
    assert binding.gqa_workspace_size(64, 64, 64) > 8 << 20


@pytest.mark.parametrize("case,expect", [
    (dict(L=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(qa=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(c=FAKE + 8), binding.DECATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(block_size=128, max_blocks_per_seq=4)), binding.DECATTN_ERR_UNSUPPORTED),
    (dict(L=dict(max_seq_len=10**6)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(num_splits=2)), binding.DECATTN_ERR_WORKSPACE),
])
def test_mla_host_checks(lib, case, expect):
    case = dict(case)
    L = case.pop("L", {})
    L = None if L is None else _launch(**L)
    assert _mla(lib, L, **case) == expect


def _gqa_window(lib, L, window, fp8=False):
    if fp8:
        return lib.gqa_decode_fp8kv_window(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 2, 128,
                                           0.088, window, ctypes.byref(L))
    return lib.gqa_decode_window(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 2, 128, 0.088, window,
                                 ctypes.byref(L))


@pytest.mark.parametrize("fp8", [False, True])
def test_window_host_checks(lib, fp8):
    for w in (0, -1, -(2**31)):
        assert _gqa_window(lib, _launch(), w, fp8) == binding.DECATTN_ERR_INVALID_ARG
    # the shared checks still come first for a valid window
    assert _gqa_window(lib, _launch(batch=0), 5, fp8) == binding.DECATTN_ERR_INVALID_ARG
    assert _gqa_window(lib, _launch(dtype=7), 5, fp8) == binding.DECATTN_ERR_INVALID_ARG
    # a window long enough for 4 splits still needs the workspace for them
    assert _gqa_window(lib, _launch(num_splits=4), 300, fp8) == binding.DECATTN_ERR_WORKSPACE


def test_window_planner_plans_for_the_window_not_the_sequence(lib):
    for B, h_q, h_kv, S, W, bs in [(1, 64, 8, 131072, 4096, 16), (4, 32, 8, 65536, 1024, 128),
                                   (2, 8, 1, 8192, 1, 16), (64, 64, 8, 8192, 4096, 16),
                                   (3, 16, 2, 100, 4096, 16)]:
        span = min(S, W + min(bs, 64) - 1)
        for kv_bytes, plan in ((2, binding.gqa_plan_splits), (1, binding.gqa_fp8_plan_splits)):
            got = binding.gqa_window_plan_splits(B, h_q, h_kv, S, W, bs, kv_bytes, num_sms=152)
            assert got == plan(B, h_q, h_kv, span, num_sms=152)
    # a 4k window over a 128k sequence is planned like a 4k sequence, not like 128k
    assert binding.gqa_window_plan_splits(1, 64, 8, 131072, 4096, 16, num_sms=152) < \
        binding.gqa_plan_splits(1, 64, 8, 131072, num_sms=152)
    for bad in [dict(window=0), dict(block_size=24), dict(kv_bytes=4)]:
        a = dict(batch=2, h_q=8, h_kv=2, max_seq_len=100, window=10, block_size=16, kv_bytes=2)
        a.update(bad)
        with pytest.raises(binding.DecAttnError):
            binding.gqa_window_plan_splits(a["batch"], a["h_q"], a["h_kv"], a["max_seq_len"],
                                           a["window"], a["block_size"], a["kv_bytes"],
                                           num_sms=152)


def _append(lib, kind, L, **kw):
    a = dict(k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, pos=FAKE, bt=FAKE, kc=FAKE, vc=FAKE, h_kv=2, d=128)
    a.update(kw)
    Lp = None if L is None else ctypes.byref(L)
    if kind == "gqa":
        return lib.gqa_kv_append(a["k"], a["v"], a["pos"], a["bt"], a["kc"], a["vc"], a["h_kv"],
                                 a["d"], Lp)
    if kind == "fp8":
        return lib.gqa_kv_append_fp8kv(a["k"], a["v"], a["ks"], a["vs"], a["pos"], a["bt"],
                                       a["kc"], a["vc"], a["h_kv"], a["d"], Lp)
    return lib.mla_kv_append(a["k"], a["pos"], a["bt"], a["kc"], Lp)


@pytest.mark.parametrize("kind", ["gqa", "fp8", "mla"])
@pytest.mark.parametrize("case,expect", [
    (dict(L=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(k=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(pos=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(kc=FAKE + 8), binding.DECATTN_ERR_INVALID_ARG),
    (dict(pos=FAKE + 2), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(batch=0)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(dtype=3)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(block_size=12)), binding.DECATTN_ERR_INVALID_ARG),
    (dict(L=dict(block_size=4)), binding.DECATTN_ERR_UNSUPPORTED),
    (dict(L=dict(err_flag=FAKE + 1)), binding.DECATTN_ERR_INVALID_ARG),
])
def test_kv_append_host_checks(lib, kind, case, expect):
    case = dict(case)
    L = case.pop("L", {})
    L = None if L is None else _launch(**L)
    assert _append(lib, kind, L, **case) == expect


def test_kv_append_kind_specific_checks(lib):
    L = _launch()
    assert _append(lib, "gqa", L, v=None) == binding.DECATTN_ERR_INVALID_ARG
    assert _append(lib, "gqa", L, d=64) == binding.DECATTN_ERR_UNSUPPORTED
    assert _append(lib, "gqa", L, h_kv=0) == binding.DECATTN_ERR_INVALID_ARG
    assert _append(lib, "fp8", L, ks=None) == binding.DECATTN_ERR_INVALID_ARG
    assert _append(lib, "fp8", L, vs=FAKE + 2) == binding.DECATTN_ERR_INVALID_ARG
    assert _append(lib, "mla", _launch(block_size=128)) == binding.DECATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("fn", ["mla_absorb_q", "mla_unabsorb_out"])
@pytest.mark.parametrize("args,expect", [
    (dict(x=None), binding.DECATTN_ERR_INVALID_ARG),
    (dict(w=FAKE + 8), binding.DECATTN_ERR_INVALID_ARG),
    (dict(y=FAKE + 1), binding.DECATTN_ERR_INVALID_ARG),
    (dict(batch=0), binding.DECATTN_ERR_INVALID_ARG),
    (dict(heads=0), binding.DECATTN_ERR_INVALID_ARG),
    (dict(dtype=9), binding.DECATTN_ERR_INVALID_ARG),
    (dict(err=FAKE + 2), binding.DECATTN_ERR_INVALID_ARG),
])
def test_absorption_gemm_host_checks(lib, fn, args, expect):
    a = dict(x=FAKE, w=FAKE, y=FAKE, batch=4, heads=128, kdim=128, mdim=512,
             dtype=binding.DECATTN_BF16, err=None)
    if fn == "mla_unabsorb_out":
        a.update(kdim=512, mdim=128)
    a.update(args)
    # argument order: (x, w, y, batch, heads, contracted width, output width, ...)
    assert getattr(lib, fn)(a["x"], a["w"], a["y"], a["batch"], a["heads"], a["kdim"],
                            a["mdim"], a["dtype"], a["err"], None) == expect


def test_absorption_gemm_shape_limits(lib):
    bf = binding.DECATTN_BF16
    # output width must be a multiple of 128, contracted width of 64
    assert lib.mla_absorb_q(FAKE, FAKE, FAKE, 4, 8, 128, 500, bf, None, None) == \
        binding.DECATTN_ERR_UNSUPPORTED
    assert lib.mla_absorb_q(FAKE, FAKE, FAKE, 4, 8, 100, 512, bf, None, None) == \
        binding.DECATTN_ERR_UNSUPPORTED
    assert lib.mla_unabsorb_out(FAKE, FAKE, FAKE, 4, 8, 512, 96, bf, None, None) == \
        binding.DECATTN_ERR_UNSUPPORTED


def test_selftest_argument_checks(lib):
    for args in [(None, FAKE, 100), (FAKE, None, 100), (FAKE + 2, FAKE, 100), (FAKE, FAKE, 0),
                 (FAKE, FAKE, 100001)]:
        assert lib.decattn_selftest_wait_timeout(args[0], args[1], args[2], None) == \
            binding.DECATTN_ERR_INVALID_ARG
