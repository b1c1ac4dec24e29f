"""Pins for the fp64 oracle, against what the pages and the mathematics fix.

Each test is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong index, a wrong sign, a transposed operand, a wrong softmax base or
scale) fails at least one of them.  None of them compares the oracle with a
retyped copy of its own formula.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
UNITS = {"B": 1, "KiB": 2**10, "MiB": 2**20, "GiB": 2**30, "MB": 1e6, "GB": 1e9}


def _f64_cache(rng, shape):
    return rng.standard_normal(shape)


def _paged(x_seq, block_size, table):
    """Scatter a contiguous [S, ...] sequence into blocks named by table (test helper)."""
    S = x_seq.shape[0]
    nb = int(max(table)) + 1
    out = np.full((nb, block_size) + x_seq.shape[1:], np.nan)
    for t in range(S):
        out[table[t // block_size], t % block_size] = x_seq[t]
    return out


# ---------------------------------------------------------------- element decoding

def test_half_decoding_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.half_to_double(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoding_matches_torch_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_double(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- cache-size formulas

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "cache_sizes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            body, cite = line.split("|", 1)
            tok = body.split()
            rows.append((tok[0], tok[1], [int(x) for x in tok[2:8]], float(tok[8]), tok[9],
                         float(tok[10]), cite.strip()))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_cache_size_formulas_match_printed_values(row):
    name, kind, (n_layers, a, b, nbytes, tokens, batch), printed, unit, tol, cite = row
    if kind == "kv":
        per_token = oracle.kv_bytes_per_token(n_layers, a, b, nbytes)
    else:
        per_token = oracle.mla_bytes_per_token(n_layers, a, b, nbytes)
    total = per_token * tokens * batch
    value = total / UNITS[unit]
    if tol == 0:
        assert value == printed, (name, value, printed, cite)
    else:
        assert abs(value - printed) <= tol * printed + 1e-12, (name, value, printed, cite)


def test_mla_vs_mha_ratio_and_gqa_equivalent_heads():
    # 576 vs 32768 elements per token per layer: "roughly a 57x difference",
    # "approximately 2.25 GQA KV heads" (576 / (2 x 128)).
    mla = oracle.mla_bytes_per_token(1, 512, 64, 1)
    mha = oracle.kv_bytes_per_token(1, 128, 128, 1)
    assert round(mha / mla) == 57
    assert mla / oracle.kv_bytes_per_token(1, 1, 128, 1) == 2.25


def test_convexity_of_the_kv_head_dial():
    # 32 -> 8 KV heads removes 75% of the cache, 8 -> 1 removes about 22 points more.
    full = oracle.kv_bytes_per_token(32, 32, 128, 2)
    g8 = oracle.kv_bytes_per_token(32, 8, 128, 2)
    g1 = oracle.kv_bytes_per_token(32, 1, 128, 2)
    assert (full - g8) / full == 0.75
    assert round(100 * (g8 - g1) / full) == 22


# ---------------------------------------------------------------- GQA decode pins

def _gqa(q, k, v, bt, sl, scale, **kw):
    return oracle.gqa_decode(q, k, v, bt, sl, dtype="f64", scale=scale, **kw)


def test_paged_gather_equals_contiguous_sequence():
    """Scattering a contiguous sequence into permuted blocks must not change anything."""
    rng = np.random.default_rng(1)
    S, bs, h_kv, d, h_q = 37, 4, 2, 8, 4
    kseq = rng.standard_normal((S, h_kv, d))
    vseq = rng.standard_normal((S, h_kv, d))
    q = rng.standard_normal((1, h_q, d))
    nblk = math.ceil(S / bs)
    # contiguous: identity table over a [nblk, bs] layout
    ident = np.arange(nblk, dtype=np.int32)
    kc = _paged(kseq, bs, ident)
    vc = _paged(vseq, bs, ident)
    kc[np.isnan(kc)] = 0.0
    vc[np.isnan(vc)] = 0.0
    o1, l1 = _gqa(q, kc, vc, ident[None], np.array([S], np.int32), 0.3)
    # permuted blocks, with spare never-referenced blocks full of NaN
    perm = rng.permutation(nblk + 5)[:nblk].astype(np.int32)
    kp = _paged(kseq, bs, perm)
    vp = _paged(vseq, bs, perm)
    o2, l2 = _gqa(q, kp, vp, perm[None], np.array([S], np.int32), 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_cache_row_inverse_of_scatter():
    table = np.array([[5, 2, 7]], dtype=np.int32)
    # token 9 with block_size 4 sits in logical block 2 -> physical 7, slot 1
    assert oracle.cache_row(table, 4, 8, 0, 9) == 7 * 4 + 1
    assert oracle.cache_row(table, 4, 8, 0, 0) == 5 * 4
    assert oracle.cache_row(np.array([[9]], np.int32), 4, 8, 0, 0) == -1


@pytest.mark.parametrize("h_q,h_kv", [(8, 2), (8, 1), (8, 8), (12, 3)])
def test_gqa_equals_mha_on_repeat_interleaved_kv(h_q, h_kv):
    """Indexing KV head i // (h_q/h_kv) equals MHA on K/V with each head repeated."""
    rng = np.random.default_rng(2)
    S, bs, d = 19, 4, 16
    nb = math.ceil(S / bs)
    k = rng.standard_normal((nb, bs, h_kv, d))
    v = rng.standard_normal((nb, bs, h_kv, d))
    q = rng.standard_normal((2, h_q, d))
    bt = np.stack([np.arange(nb), np.arange(nb)[::-1]]).astype(np.int32)
    sl = np.array([S, S - 6], np.int32)
    o_g, l_g = _gqa(q, k, v, bt, sl, 0.25)
    rep = h_q // h_kv
    k_rep = np.repeat(k, rep, axis=2)  # repeat_interleave along the head axis
    v_rep = np.repeat(v, rep, axis=2)
    o_m, l_m = _gqa(q, k_rep, v_rep, bt, sl, 0.25)
    assert np.array_equal(o_g, o_m) and np.array_equal(l_g, l_m)
    if 1 < h_kv < h_q:
        # sensitivity: the interleaved-modulo mapping (head i -> i % h_kv) is different
        o_bad, _ = _gqa(q, np.tile(k, (1, 1, rep, 1)), np.tile(v, (1, 1, rep, 1)), bt, sl, 0.25)
        assert not np.allclose(o_bad, o_g)


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((2, 4, 2, 8))
    v = rng.standard_normal((2, 4, 2, 8))
    q = rng.standard_normal((1, 4, 8))
    bt = np.array([[1, 0]], np.int32)
    out, lse = _gqa(q, k, v, bt, np.array([1], np.int32), 0.5)
    for i in range(4):
        j = i // 2
        assert np.array_equal(out[i], v[1, 0, j])
        assert lse[i] == pytest.approx(0.5 * float(q[0, i] @ k[1, 0, j]), abs=1e-14)


def test_zero_query_gives_mean_of_values_and_log_length():
    rng = np.random.default_rng(4)
    S, bs = 23, 8
    k = rng.standard_normal((3, bs, 1, 8))
    v = rng.standard_normal((3, bs, 1, 8))
    q = np.zeros((1, 2, 8))
    bt = np.array([[2, 0, 1]], np.int32)
    out, lse = _gqa(q, k, v, bt, np.array([S], np.int32), 1.0)
    vals = np.stack([v[bt[0, t // bs], t % bs, 0] for t in range(S)])
    for i in range(2):
        np.testing.assert_allclose(out[i], vals.mean(axis=0), rtol=0, atol=1e-14)
        assert lse[i] == pytest.approx(math.log(S), abs=1e-14)


def test_equal_keys_give_mean_and_constant_values_are_reproduced():
    rng = np.random.default_rng(5)
    S = 9
    kvec = rng.standard_normal(8)
    k = np.broadcast_to(kvec, (S, 1, 1, 8)).copy().reshape(S, 1, 1, 8)
    v = rng.standard_normal((S, 1, 1, 8))
    q = rng.standard_normal((1, 1, 8))
    bt = np.arange(S, dtype=np.int32)[None]
    out, lse = _gqa(q, k, v, bt, np.array([S], np.int32), 0.7)
    np.testing.assert_allclose(out[0], v[:, 0, 0].mean(axis=0), atol=1e-14)
    assert lse[0] == pytest.approx(0.7 * float(q[0, 0] @ kvec) + math.log(S), abs=1e-13)
    # constant values: the probabilities sum to one
    k2 = rng.standard_normal((S, 1, 1, 8))
    vc = np.full((S, 1, 1, 8), -1.75)
    out2, _ = _gqa(q, k2, vc, bt, np.array([S], np.int32), 0.7)
    np.testing.assert_allclose(out2[0], -1.75, atol=1e-14)


def test_two_tokens_closed_form():
    # q = e0, k0 = 2 e0, k1 = 0, scale 1/2 -> s0 = 1, s1 = 0
    # p0 = e/(1+e), p1 = 1/(1+e); v0 = e0, v1 = e1.
    d = 4
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    k = np.zeros((2, 1, 1, d)); k[0, 0, 0, 0] = 2.0
    v = np.zeros((2, 1, 1, d)); v[0, 0, 0, 0] = 1.0; v[1, 0, 0, 1] = 1.0
    bt = np.array([[0, 1]], np.int32)
    out, lse = _gqa(q, k, v, bt, np.array([2], np.int32), 0.5)
    e = math.e
    assert out[0, 0] == pytest.approx(e / (1 + e), abs=1e-15)
    assert out[0, 1] == pytest.approx(1 / (1 + e), abs=1e-15)
    assert out[0, 2] == 0.0 and out[0, 3] == 0.0
    assert lse[0] == pytest.approx(math.log(1 + e), abs=1e-15)


def test_softmax_weights_follow_exponential_of_scaled_scores():
    # one-hot query and keys: s_t = scale * c_t; one-hot values read p back.
    S, d = 6, 8
    c = np.array([0.0, 3.0, -2.0, 1.5, 3.0, -7.0])
    q = np.zeros((1, 1, d)); q[0, 0, 2] = 1.0
    k = np.zeros((S, 1, 1, d)); k[:, 0, 0, 2] = c
    v = np.zeros((S, 1, 1, d))
    for t in range(S):
        v[t, 0, 0, t] = 1.0
    scale = 0.8
    bt = np.arange(S, dtype=np.int32)[None]
    out, lse = _gqa(q, k, v, bt, np.array([S], np.int32), scale)
    z = math.fsum(math.exp(scale * x) for x in c)
    for t in range(S):
        assert out[0, t] == pytest.approx(math.exp(scale * c[t]) / z, rel=1e-14)
    assert lse[0] == pytest.approx(math.log(z), abs=1e-14)


def test_large_scores_select_the_argmax_value():
    rng = np.random.default_rng(6)
    S, d = 12, 16
    k = rng.standard_normal((S, 1, 1, d)) * 0.01
    k[7, 0, 0] = 0.0
    k[7, 0, 0, 3] = 1.0
    q = np.zeros((1, 1, d)); q[0, 0, 3] = 1.0
    v = rng.standard_normal((S, 1, 1, d))
    bt = np.arange(S, dtype=np.int32)[None]
    out, _ = _gqa(q, k, v, bt, np.array([S], np.int32), 60.0)
    np.testing.assert_allclose(out[0], v[7, 0, 0], atol=1e-20 + 1e-12)


@pytest.mark.parametrize("split", [0, 1, 5, 16, 31, 32])
def test_lse_merge_of_halves_equals_whole(split):
    rng = np.random.default_rng(7)
    S, bs, d, h_q = 32, 4, 8, 4
    k = rng.standard_normal((8, bs, 2, d)) * 2
    v = rng.standard_normal((8, bs, 2, d))
    q = rng.standard_normal((1, h_q, d))
    bt = rng.permutation(8).astype(np.int32)[None]
    sl = np.array([S], np.int32)
    whole, lw = _gqa(q, k, v, bt, sl, 0.9)
    a, la = _gqa(q, k, v, bt, sl, 0.9, t_begin=0, t_end=split)
    b, lb = _gqa(q, k, v, bt, sl, 0.9, t_begin=split, t_end=-1)
    for i in range(h_q):
        m, lm = oracle.lse_merge(np.stack([a[i], b[i]]), np.array([la[i], lb[i]]))
        np.testing.assert_allclose(m, whole[i], atol=1e-13)
        assert lm == pytest.approx(lw[i], abs=1e-13)


def test_token_order_does_not_matter():
    rng = np.random.default_rng(8)
    S, d = 15, 8
    kseq = rng.standard_normal((S, 1, 1, d))
    vseq = rng.standard_normal((S, 1, 1, d))
    q = rng.standard_normal((1, 2, d))
    perm = rng.permutation(S)
    bt = np.arange(S, dtype=np.int32)[None]
    o1, l1 = _gqa(q, kseq, vseq, bt, np.array([S], np.int32), 0.6)
    o2, l2 = _gqa(q, kseq[perm], vseq[perm], bt, np.array([S], np.int32), 0.6)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


def test_empty_sequence_and_bad_block():
    k = np.ones((2, 4, 1, 8))
    q = np.ones((2, 1, 8))
    bt = np.array([[0, 1], [1, 5]], np.int32)
    out, lse = _gqa(q, k, k, bt, np.array([0, 4], np.int32), 1.0)
    assert np.all(out[0] == 0.0) and lse[0] == -math.inf
    with pytest.raises(ValueError):
        _gqa(q, k, k, bt, np.array([0, 6], np.int32), 1.0)  # token 4 reads block id 5 >= 2


def test_oracle_reads_16bit_storage_like_its_decoded_values():
    rng = np.random.default_rng(9)
    kf = rng.standard_normal((3, 4, 2, 8)).astype(np.float16)
    vf = rng.standard_normal((3, 4, 2, 8)).astype(np.float16)
    qf = rng.standard_normal((1, 4, 8)).astype(np.float16)
    bt = np.array([[2, 0, 1]], np.int32)
    sl = np.array([11], np.int32)
    o16, l16 = oracle.gqa_decode(qf.view(np.uint16), kf.view(np.uint16), vf.view(np.uint16), bt,
                                 sl, dtype="fp16", scale=0.4)
    o64, l64 = _gqa(qf.astype(np.float64), kf.astype(np.float64), vf.astype(np.float64), bt, sl,
                    0.4)
    assert np.array_equal(o16, o64) and np.array_equal(l16, l64)


# ---------------------------------------------------------------- MLA pins

def test_absorbed_mla_matches_explicit_reconstruction():
    """Reconstruct-then-attend equals the absorbed form (the pages' MLA exercise)."""
    rng = np.random.default_rng(10)
    h, d_c, d_h, d_r, d_v, S = 4, 32, 16, 8, 16, 7
    q_nope = rng.standard_normal((h, d_h))
    q_rope = rng.standard_normal((h, d_r))
    c = rng.standard_normal((S, d_c))
    kr = rng.standard_normal((S, d_r))
    w_uk = rng.standard_normal((h, d_c, d_h)) / math.sqrt(d_c)
    w_uv = rng.standard_normal((h, d_c, d_v)) / math.sqrt(d_c)
    scale = 1.0 / math.sqrt(d_h + d_r)
    out_x, scores_x = oracle.mla_explicit(q_nope, q_rope, c, kr, w_uk, w_uv, scale=scale)
    # absorbed: q_abs^(i) = W_uk^(i) q_nope^(i) (a d_c vector); cache = [c | kr]
    q_abs = np.einsum("iae,ie->ia", w_uk, q_nope)[None]
    cache = np.concatenate([c, kr], axis=1)[:, None, :]  # block_size 1
    bt = np.arange(S, dtype=np.int32)[None]
    lat, lse = oracle.mla_decode(q_abs, q_rope[None], cache, bt, np.array([S], np.int32),
                                 dtype="f64", scale=scale)
    out_a = np.einsum("ia,iav->iv", lat, w_uv)
    np.testing.assert_allclose(out_a, out_x, rtol=1e-10, atol=1e-12)
    m = scores_x.max(axis=1)
    lse_x = m + np.log(np.exp(scores_x - m[:, None]).sum(axis=1))
    np.testing.assert_allclose(lse, lse_x, rtol=1e-10)


def test_mla_without_rope_is_mqa_with_latent_as_key_and_value():
    rng = np.random.default_rng(11)
    H, d_c, S, bs = 6, 16, 21, 4
    nb = math.ceil(S / bs) + 2
    lat = rng.standard_normal((nb, bs, d_c))
    cache = np.concatenate([lat, rng.standard_normal((nb, bs, 4))], axis=2)
    q_abs = rng.standard_normal((1, H, d_c))
    q_rope = np.zeros((1, H, 4))
    bt = rng.permutation(nb)[: math.ceil(S / bs)].astype(np.int32)[None]
    sl = np.array([S], np.int32)
    o_mla, l_mla = oracle.mla_decode(q_abs, q_rope, cache, bt, sl, dtype="f64", scale=0.3)
    o_mqa, l_mqa = _gqa(q_abs, lat[:, :, None, :], lat[:, :, None, :], bt, sl, 0.3)
    np.testing.assert_allclose(o_mla, o_mqa, atol=1e-14)
    np.testing.assert_allclose(l_mla, l_mqa, atol=1e-14)


def test_mla_rope_part_closed_form():
    # q_abs = 0; q_rope = a e0; kr_0 = e0, kr_1 = 0 -> s0 = scale a, s1 = 0
    d_c, d_r = 8, 4
    a, scale = 3.0, 0.5
    q_abs = np.zeros((1, 1, d_c))
    q_rope = np.zeros((1, 1, d_r)); q_rope[0, 0, 0] = a
    cache = np.zeros((2, 1, d_c + d_r))
    cache[0, 0, :d_c] = np.arange(1, d_c + 1)
    cache[1, 0, :d_c] = -1.0
    cache[0, 0, d_c] = 1.0
    bt = np.array([[0, 1]], np.int32)
    out, lse = oracle.mla_decode(q_abs, q_rope, cache, bt, np.array([2], np.int32), dtype="f64",
                                 scale=scale)
    p0 = 1.0 / (1.0 + math.exp(-scale * a))
    np.testing.assert_allclose(out[0], p0 * np.arange(1, d_c + 1) + (1 - p0) * -1.0, atol=1e-14)
    assert lse[0] == pytest.approx(math.log(math.exp(scale * a) + 1.0), abs=1e-14)


def test_mla_latent_part_closed_form():
    # q_abs = e3; latent of token 0 = 2 e3 + 5 e0, of token 1 = 0; rope ignored (q_rope = 0)
    d_c, d_r = 8, 4
    q_abs = np.zeros((1, 1, d_c)); q_abs[0, 0, 3] = 1.0
    q_rope = np.zeros((1, 1, d_r))
    cache = np.zeros((2, 2, d_c + d_r))
    cache[1, 0, 3] = 2.0; cache[1, 0, 0] = 5.0
    cache[1, 0, d_c:] = 100.0  # rope key: multiplied by a zero query
    bt = np.array([[1]], np.int32)
    out, _ = oracle.mla_decode(q_abs, q_rope, cache, bt, np.array([2], np.int32), dtype="f64",
                               scale=1.0)
    p0 = math.exp(2.0) / (math.exp(2.0) + 1.0)
    expect = np.zeros(d_c); expect[3] = 2.0 * p0; expect[0] = 5.0 * p0
    np.testing.assert_allclose(out[0], expect, atol=1e-14)


# ---------------------------------------------------------------- 8-bit (e4m3) KV cache

def test_e4m3_decoding_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_double(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # 0x7f, 0xff
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_closed_form_codes():
    # sign | 4-bit exponent (bias 7) | 3-bit fraction; exponent 0 is subnormal.
    cases = {0x00: 0.0, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x08: 2.0**-6, 0x38: 1.0,
             0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    got = oracle.e4m3_to_double(np.array(list(cases), np.uint8))
    assert list(got) == list(cases.values())
    assert math.copysign(1.0, oracle.e4m3_to_double(np.array([0x80], np.uint8))[0]) == -1.0
    # monotone over the positive finite codes
    pos = oracle.e4m3_to_double(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


def test_dequant_uses_the_scale_of_each_kv_head():
    rows, h_kv, d = 3, 4, 5
    codes = np.full((rows, h_kv, d), 0x38, np.uint8)  # every code is 1.0
    scales = np.array([0.5, 2.0, 3.0, -1.25])
    out = oracle.dequant_e4m3(codes, scales)
    for j in range(h_kv):
        assert np.all(out[:, j, :] == scales[j])


def _fp8_case(rng, B=2, h_q=8, h_kv=2, d=16, S=(23, 9), bs=4):
    nblk = [math.ceil(s / bs) for s in S]
    table = np.full((B, max(nblk)), -1, np.int32)
    perm = rng.permutation(sum(nblk) + 2).astype(np.int32)
    k = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[k:k + nblk[b]]
        k += nblk[b]
    nb = int(perm.max()) + 1
    # finite e4m3 codes of moderate magnitude (|value| <= 8)
    mags = np.array([c for c in range(0x60) if c != 0x7F], np.uint8)
    kc = rng.choice(mags, size=(nb, bs, h_kv, d)) | (rng.integers(0, 2, (nb, bs, h_kv, d)) << 7).astype(np.uint8)
    vc = rng.choice(mags, size=(nb, bs, h_kv, d)) | (rng.integers(0, 2, (nb, bs, h_kv, d)) << 7).astype(np.uint8)
    q = torch.from_numpy(rng.standard_normal((B, h_q, d))).to(torch.bfloat16)
    qbits = q.view(torch.int16).numpy().view(np.uint16)
    return qbits, kc.astype(np.uint8), vc.astype(np.uint8), table, np.array(S, np.int32)


def test_fp8kv_with_unit_scales_equals_the_16bit_path():
    # Every e4m3 value is exactly representable in bfloat16, so the same cache
    # stored as bf16 bits must give exactly the same fp64 result.
    rng = np.random.default_rng(11)
    q, kc, vc, bt, sl = _fp8_case(rng)
    to_bf16 = lambda c: torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    ones = np.ones(kc.shape[2])
    o1, l1 = oracle.gqa_decode_fp8kv(q, kc, vc, ones, ones, bt, sl, q_dtype="bf16", scale=0.2)
    o2, l2 = oracle.gqa_decode(q, to_bf16(kc), to_bf16(vc), bt, sl, dtype="bf16", scale=0.2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8kv_scales_act_on_scores_and_values_per_kv_head():
    # V's scale multiplies the output of the heads that read that KV head; K's
    # scale is the same as scaling those heads' queries.
    rng = np.random.default_rng(12)
    q, kc, vc, bt, sl = _fp8_case(rng, h_q=8, h_kv=2)
    ks = np.array([0.75, 1.5])
    vs = np.array([0.25, 4.0])
    ones = np.ones(2)
    o, lse = oracle.gqa_decode_fp8kv(q, kc, vc, ks, vs, bt, sl, q_dtype="bf16", scale=0.2)
    q64 = oracle.bf16_to_double(q)
    G = q.shape[1] // 2
    qs = q64 * np.repeat(ks, G)[None, :, None]
    o_ref, lse_ref = oracle.gqa_decode(qs, oracle.dequant_e4m3(kc, ones), oracle.dequant_e4m3(vc, ones),
                                       bt, sl, dtype="f64", scale=0.2)
    heads = np.tile(np.arange(q.shape[1]), q.shape[0])
    np.testing.assert_allclose(o, o_ref * vs[heads // G][:, None], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- sliding-window decode

def _window_case(seed, lens, bs=4, h_q=4, h_kv=2, d=8):
    rng = np.random.default_rng(seed)
    B = len(lens)
    per = max(math.ceil(max(lens) / bs), 1)
    nb = B * per + 3
    k = rng.standard_normal((nb, bs, h_kv, d)) * 1.5
    v = rng.standard_normal((nb, bs, h_kv, d))
    q = rng.standard_normal((B, h_q, d))
    bt = rng.permutation(nb)[:B * per].reshape(B, per).astype(np.int32)
    return q, k, v, bt, np.array(lens, np.int32)


def test_window_start_reading():
    # the window holds the newest `window` positions, the query's own included
    assert oracle.window_start(10, 3) == 7
    assert oracle.window_start(10, 10) == 0
    assert oracle.window_start(10, 11) == 0
    assert oracle.window_start(0, 1) == 0
    assert oracle.window_start(5, 1) == 4


def test_window_covering_every_sequence_is_full_attention():
    q, k, v, bt, sl = _window_case(20, [13, 1, 0, 9])
    full, lf = _gqa(q, k, v, bt, sl, 0.4)
    for w in (13, 14, 1000):
        o, l = oracle.gqa_decode_window(q, k, v, bt, sl, dtype="f64", scale=0.4, window=w)
        assert np.array_equal(o, full) and np.array_equal(l, lf)


def test_window_of_one_returns_the_newest_value():
    q, k, v, bt, sl = _window_case(21, [13, 1, 7])
    o, l = oracle.gqa_decode_window(q, k, v, bt, sl, dtype="f64", scale=0.4, window=1)
    bs, group = k.shape[1], q.shape[1] // k.shape[2]
    for b, L in enumerate(sl):
        t = L - 1
        blk, slot = bt[b, t // bs], t % bs
        for i in range(q.shape[1]):
            r = b * q.shape[1] + i
            assert np.array_equal(o[r], v[blk, slot, i // group])
            assert l[r] == pytest.approx(0.4 * float(q[b, i] @ k[blk, slot, i // group]), abs=1e-13)


@pytest.mark.parametrize("window", [2, 3, 4, 5, 8, 11])
def test_window_equals_full_attention_on_the_last_tokens_copied_out(window):
    """Copy each sequence's last `window` tokens into a fresh contiguous cache
    and attend to all of them: the windowed result must be the same, and one
    token more or fewer must not be."""
    q, k, v, bt, sl = _window_case(22, [13, 6, 12, 4, 5])
    bs = k.shape[1]
    o, l = oracle.gqa_decode_window(q, k, v, bt, sl, dtype="f64", scale=0.7, window=window)

    def copied(b, n):
        L = int(sl[b])
        pos = list(range(max(0, L - n), L))
        kk = np.stack([k[bt[b, t // bs], t % bs] for t in pos])[None]  # one block of len(pos)
        vv = np.stack([v[bt[b, t // bs], t % bs] for t in pos])[None]
        return _gqa(q[b:b + 1], kk, vv, np.zeros((1, 1), np.int32),
                    np.array([len(pos)], np.int32), 0.7)

    h_q = q.shape[1]
    for b in range(len(sl)):
        ref_o, ref_l = copied(b, window)
        got = slice(b * h_q, (b + 1) * h_q)
        np.testing.assert_allclose(o[got], ref_o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l[got], ref_l, rtol=0, atol=1e-13)
        if sl[b] > window:  # sensitivity: an off-by-one window is a different result
            assert not np.allclose(o[got], copied(b, window + 1)[0])
            assert not np.allclose(o[got], copied(b, window - 1)[0])


def test_growing_the_window_by_one_admits_exactly_the_next_older_token():
    """out_{W+1} and lse_{W+1} follow from out_W, lse_W and the one token at
    position L - W - 1 by the closed-form softmax update."""
    q, k, v, bt, sl = _window_case(23, [13, 9])
    bs, h_q, group = k.shape[1], q.shape[1], q.shape[1] // k.shape[2]
    scale = 0.6
    for w in (1, 3, 6):
        o1, l1 = oracle.gqa_decode_window(q, k, v, bt, sl, dtype="f64", scale=scale, window=w)
        o2, l2 = oracle.gqa_decode_window(q, k, v, bt, sl, dtype="f64", scale=scale, window=w + 1)
        for b, L in enumerate(sl):
            t = L - w - 1
            blk, slot = bt[b, t // bs], t % bs
            for i in range(h_q):
                r = b * h_q + i
                s = scale * float(q[b, i] @ k[blk, slot, i // group])
                lse = np.logaddexp(l1[r], s)
                assert l2[r] == pytest.approx(lse, abs=1e-12)
                expect = math.exp(l1[r] - lse) * o1[r] + math.exp(s - lse) * v[blk, slot, i // group]
                np.testing.assert_allclose(o2[r], expect, rtol=0, atol=1e-12)


def test_blocks_before_the_window_are_never_read():
    """Blocks wholly before the window may be recycled: invalid ids there and
    NaN in the window's first block before its start change nothing."""
    q, k, v, bt, sl = _window_case(24, [13, 11], bs=4)
    w = 6
    ref, lref = oracle.gqa_decode_window(q, k, v, bt, sl, dtype="f64", scale=0.5, window=w)
    bt2, k2, v2 = bt.copy(), k.copy(), v.copy()
    for b, L in enumerate(sl):
        w0 = oracle.window_start(L, w)
        for t in range(w0):
            blk = bt[b, t // 4]
            k2[blk, t % 4] = np.nan
            v2[blk, t % 4] = np.nan
        bt2[b, :w0 // 4] = -1  # blocks wholly before the window
    o, l = oracle.gqa_decode_window(q, k2, v2, bt2, sl, dtype="f64", scale=0.5, window=w)
    assert np.array_equal(o, ref) and np.array_equal(l, lref)
    with pytest.raises(ValueError):  # but a bad id inside the window is still an error
        bt3 = bt.copy()
        bt3[0, (int(sl[0]) - 1) // 4] = 99
        oracle.gqa_decode_window(q, k, v, bt3, sl, dtype="f64", scale=0.5, window=w)


def test_fp8kv_window_reduces_to_the_full_fp8_path_and_to_one_value():
    rng = np.random.default_rng(25)
    nb, bs, h_kv, d, h_q = 6, 4, 2, 8, 4
    codes_k = rng.integers(0, 256, (nb, bs, h_kv, d), dtype=np.uint8)
    codes_v = rng.integers(0, 256, (nb, bs, h_kv, d), dtype=np.uint8)
    codes_k[(codes_k & 0x7F) == 0x7F] = 0x10  # no NaN codes
    codes_v[(codes_v & 0x7F) == 0x7F] = 0x20
    ks, vs = np.array([0.01, 0.02]), np.array([0.5, 0.25])
    q = torch.randn(2, h_q, d, generator=torch.Generator().manual_seed(5)).to(torch.float16)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    bt = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    sl = np.array([11, 7], np.int32)
    full = oracle.gqa_decode_fp8kv(qb, codes_k, codes_v, ks, vs, bt, sl, q_dtype="fp16", scale=0.3)
    win = oracle.gqa_decode_fp8kv_window(qb, codes_k, codes_v, ks, vs, bt, sl, q_dtype="fp16",
                                         scale=0.3, window=11)
    assert np.array_equal(full[0], win[0])
    one, _ = oracle.gqa_decode_fp8kv_window(qb, codes_k, codes_v, ks, vs, bt, sl, q_dtype="fp16",
                                            scale=0.3, window=1)
    for b, L in enumerate(sl):
        t = L - 1
        for i in range(h_q):
            j = i // 2
            expect = oracle.e4m3_to_double(codes_v[bt[b, t // bs], t % bs, j]) * vs[j]
            assert np.array_equal(one[b * h_q + i], expect)


# ---------------------------------------------------------------- e4m3 encoding and KV append

def test_e4m3_encoding_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    values = oracle.e4m3_to_double(codes).astype(np.float32)  # exact in fp32
    assert np.array_equal(oracle.e4m3_from_float32(values), codes)  # -0 keeps its sign too


def test_e4m3_encoding_matches_torch_rounding_inside_the_range():
    """torch's float8_e4m3fn cast rounds to nearest even; inside +-448 it must agree."""
    g = torch.Generator().manual_seed(17)
    y = torch.cat([torch.randn(200000, generator=g) * s for s in (0.01, 1.0, 30.0, 150.0)])
    y = y.clamp(-448, 448)
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_from_float32(y.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encoding_ties_saturation_and_specials():
    f = lambda v: int(oracle.e4m3_from_float32([v])[0])
    # ties go to the even code: between 2^-6 (0x08) and 1.125 * 2^-6 (0x09) -> 0x08,
    # between 0x09 and 0x0A (1.25 * 2^-6) -> 0x0A
    assert f(2.0**-6 * 1.0625) == 0x08
    assert f(2.0**-6 * 1.1875) == 0x0A
    assert f(2.0**-6 * 1.0625 * (1 + 2**-20)) == 0x09  # just above the tie
    # below half the smallest subnormal (2^-9) is zero; the half itself ties to 0x00
    assert f(2.0**-10) == 0x00 and f(2.0**-10 * 1.001) == 0x01 and f(-(2.0**-11)) == 0x80
    # saturation at 448 in place of overflow; infinities saturate; NaN stays NaN
    assert f(449.0) == 0x7E and f(464.0) == 0x7E and f(1e30) == 0x7E and f(-1e30) == 0xFE
    assert f(float("inf")) == 0x7E and f(float("-inf")) == 0xFE and f(float("nan")) == 0x7F
    # largest step: 416 (0x7D) .. 448 (0x7E); 432 is the tie -> even code 0x7E
    assert f(430.0) == 0x7D and f(432.0) == 0x7E and f(433.0) == 0x7E


def test_quantisation_divides_by_each_kv_heads_scale():
    rng = np.random.default_rng(31)
    codes = rng.integers(0, 0x7E, (3, 2, 16), dtype=np.uint8)  # positive finite codes
    scale = np.array([0.5, 0.03125], dtype=np.float32)  # powers of two: products exact
    vals = oracle.e4m3_to_double(codes) * scale[None, :, None]
    bits = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    bits = bits.numpy().view(np.uint16)
    back = oracle.bf16_to_double(bits)
    assert np.array_equal(back, vals)  # every value is exact in bf16
    assert np.array_equal(oracle.quant_e4m3(bits, "bf16", scale), codes)
    # swapping the heads' scales moves every code of the two heads
    wrong = oracle.quant_e4m3(bits, "bf16", scale[::-1].copy())
    assert np.all(wrong[:, 0][codes[:, 0] > 0x10] != codes[:, 0][codes[:, 0] > 0x10])


def test_kv_append_writes_exactly_one_slot_per_sequence():
    rng = np.random.default_rng(32)
    nb, bs, h_kv, d = 9, 4, 2, 8
    cache = rng.standard_normal((nb, bs, h_kv, d))
    bt = np.array([[3, 7, -1], [0, 5, 8], [1, 2, 4], [6, -1, -1]], np.int32)
    new = rng.standard_normal((4, h_kv, d))
    pos = np.array([5, 8, -1, 4], np.int64)  # seq 1 starts block 2; seq 2 skips; seq 3 has no block
    out, bad = oracle.kv_append(cache, new, pos, bt)
    assert bad == {3: "bad_block"}
    assert np.array_equal(out[7, 1], new[0])      # position 5 = block 1 (id 7), slot 1
    assert np.array_equal(out[8, 0], new[1])      # position 8 = block 2 (id 8), slot 0
    changed = np.any(out != cache, axis=(2, 3))
    assert changed.sum() == 2 and changed[7, 1] and changed[8, 0]
    _, bad = oracle.kv_append(cache, new, np.array([12, -5, -5, -5]), bt)
    assert bad == {0: "bad_position"}              # past the table's 3 blocks
    # read back through the decode path's gather: token 5 of sequence 0 is the new row
    row = oracle.cache_row(bt, bs, nb, 0, 5)
    assert np.array_equal(out.reshape(nb * bs, h_kv, d)[row], new[0])


def test_appending_then_attending_equals_attending_over_the_longer_sequence():
    """Append the next token then decode over L + 1 tokens = decode over a
    contiguous copy of the L + 1 tokens."""
    rng = np.random.default_rng(33)
    bs, h_kv, d, h_q, L = 4, 2, 8, 4, 10
    nb = 5
    k = rng.standard_normal((nb, bs, h_kv, d))
    v = rng.standard_normal((nb, bs, h_kv, d))
    bt = np.array([[4, 0, 2]], np.int32)
    kn, vn = rng.standard_normal((1, h_kv, d)), rng.standard_normal((1, h_kv, d))
    k2, _ = oracle.kv_append(k, kn, [L], bt)
    v2, _ = oracle.kv_append(v, vn, [L], bt)
    q = rng.standard_normal((1, h_q, d))
    o, l = _gqa(q, k2, v2, bt, np.array([L + 1], np.int32), 0.3)
    seq_k = np.stack([k[bt[0, t // bs], t % bs] for t in range(L)] + [kn[0]])[None]
    seq_v = np.stack([v[bt[0, t // bs], t % bs] for t in range(L)] + [vn[0]])[None]
    o_ref, l_ref = _gqa(q, seq_k, seq_v, np.zeros((1, 1), np.int32), np.array([L + 1], np.int32),
                        0.3)
    assert np.array_equal(o, o_ref) and np.array_equal(l, l_ref)


# ---------------------------------------------------------------- MLA absorption GEMMs

def test_absorption_gemms_match_brute_force_loops():
    rng = np.random.default_rng(40)
    B, H, d_h, d_c, d_v = 2, 3, 4, 5, 6
    q = rng.standard_normal((B, H, d_h))
    w_uk = rng.standard_normal((H, d_c, d_h))
    o = rng.standard_normal((B, H, d_c))
    w_uv_t = rng.standard_normal((H, d_v, d_c))
    qa = oracle.mla_absorb_q(q, w_uk, dtype="f64")
    out = oracle.mla_unabsorb_out(o, w_uv_t, dtype="f64")
    for b in range(B):
        for i in range(H):
            for a in range(d_c):  # q_abs_i = q_i W_uk^(i)^T, W_uk^(i) = w_uk[i] (d_c x d_h)
                assert qa[b, i, a] == pytest.approx(sum(q[b, i, e] * w_uk[i, a, e]
                                                        for e in range(d_h)), abs=1e-13)
            for v in range(d_v):  # out_i = o_i W_uv^(i), W_uv^(i) = w_uv_t[i]^T (d_c x d_v)
                assert out[b, i, v] == pytest.approx(sum(o[b, i, a] * w_uv_t[i, v, a]
                                                         for a in range(d_c)), abs=1e-13)


def test_absorb_attend_unabsorb_equals_explicit_reconstruction_per_sequence():
    """Absorb the query, attend over the latent cache, apply W_uv: the same as
    reconstructing every head's K and V from the latent and attending to them
    (the pages' reconstruct-or-absorb question), for a batch of sequences."""
    rng = np.random.default_rng(41)
    B, H, d_c, d_h, d_r, d_v, S = 2, 4, 32, 16, 8, 16, 9
    q_nope = rng.standard_normal((B, H, d_h))
    q_rope = rng.standard_normal((B, H, d_r))
    c = rng.standard_normal((B, S, d_c))
    kr = rng.standard_normal((B, S, d_r))
    w_uk = rng.standard_normal((H, d_c, d_h)) / math.sqrt(d_c)
    w_uv = rng.standard_normal((H, d_c, d_v)) / math.sqrt(d_c)
    scale = 1.0 / math.sqrt(d_h + d_r)
    q_abs = oracle.mla_absorb_q(q_nope, w_uk, dtype="f64")
    cache = np.concatenate([c, kr], axis=2).reshape(B * S, 1, d_c + d_r)  # block_size 1
    bt = np.arange(B * S, dtype=np.int32).reshape(B, S)
    lat, _ = oracle.mla_decode(q_abs, q_rope, cache, bt, np.full(B, S, np.int32), dtype="f64",
                               scale=scale)
    out = oracle.mla_unabsorb_out(lat.reshape(B, H, d_c), np.swapaxes(w_uv, 1, 2).copy(),
                                  dtype="f64")
    for b in range(B):
        ref, _ = oracle.mla_explicit(q_nope[b], q_rope[b], c[b], kr[b], w_uk, w_uv, scale=scale)
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)
    # sensitivity: W_uk^(i) used untransposed (square case) or heads shifted is different
    sq = rng.standard_normal((H, d_h, d_h))
    assert not np.allclose(oracle.mla_absorb_q(q_nope, sq, dtype="f64"),
                           oracle.mla_absorb_q(q_nope, np.swapaxes(sq, 1, 2).copy(), dtype="f64"))
    assert not np.allclose(q_abs, oracle.mla_absorb_q(q_nope, np.roll(w_uk, 1, axis=0),
                                                      dtype="f64"))


def test_absorption_reads_16bit_weights_like_their_decoded_values():
    rng = np.random.default_rng(42)
    q = rng.standard_normal((2, 3, 8)).astype(np.float16)
    w = rng.standard_normal((3, 5, 8)).astype(np.float16)
    got = oracle.mla_absorb_q(q.view(np.uint16), w.view(np.uint16), dtype="fp16")
    ref = oracle.mla_absorb_q(q.astype(np.float64), w.astype(np.float64), dtype="f64")
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- library cross-checks

def _sdpa(q, k, v, scale):
    """torch's scaled_dot_product_attention in fp64 on the CPU (a library
    routine independent of the oracle): q [H, 1, d], k/v [H, S, d]."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None]
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v),
                                                            scale=scale)[0].numpy()


@pytest.mark.parametrize("h_q,h_kv,S", [(4, 4, 1), (4, 2, 3), (8, 1, 8), (6, 3, 7), (8, 2, 8)])
def test_gqa_decode_matches_torch_sdpa_on_tiny_cases(h_q, h_kv, S):
    rng = np.random.default_rng(50 + S)
    bs, d = 4, 16
    nb = math.ceil(S / bs) + 2
    k = rng.standard_normal((nb, bs, h_kv, d))
    v = rng.standard_normal((nb, bs, h_kv, d))
    q = rng.standard_normal((1, h_q, d))
    bt = rng.permutation(nb)[:math.ceil(S / bs)].astype(np.int32)[None]
    out, lse = _gqa(q, k, v, bt, np.array([S], np.int32), 0.37)
    kseq = np.stack([k[bt[0, t // bs], t % bs] for t in range(S)])  # [S, h_kv, d]
    vseq = np.stack([v[bt[0, t // bs], t % bs] for t in range(S)])
    g = h_q // h_kv
    kk = np.repeat(kseq.transpose(1, 0, 2), g, axis=0)  # [h_q, S, d], head i -> KV head i // g
    vv = np.repeat(vseq.transpose(1, 0, 2), g, axis=0)
    ref = _sdpa(q[0][:, None, :], kk, vv, 0.37)[:, 0, :]
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


def test_mla_decode_matches_torch_sdpa_on_a_tiny_case():
    """Absorbed MLA is attention with the 576-d cache row as key (the query
    being q_abs and q_rope side by side) and its first 512 entries as value."""
    rng = np.random.default_rng(60)
    H, d_c, d_r, S = 4, 32, 8, 7
    q_abs = rng.standard_normal((1, H, d_c))
    q_rope = rng.standard_normal((1, H, d_r))
    cache = rng.standard_normal((S, 1, d_c + d_r))
    bt = np.arange(S, dtype=np.int32)[None]
    out, _ = oracle.mla_decode(q_abs, q_rope, cache, bt, np.array([S], np.int32), dtype="f64",
                               scale=0.2)
    qcat = np.concatenate([q_abs[0], q_rope[0]], axis=1)[:, None, :]  # [H, 1, d_c + d_r]
    keys = np.repeat(cache[:, 0][None], H, axis=0)                      # [H, S, d_c + d_r]
    vals = keys[..., :d_c]
    ref = _sdpa(qcat, keys, np.ascontiguousarray(vals), 0.2)[:, 0, :]
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


def test_softmax_weights_sum_to_one():
    """out = sum_t p_t v_t with sum_t p_t = 1: appending a constant column c to
    every value row must give exactly c in that output column (up to rounding)."""
    rng = np.random.default_rng(61)
    S, bs, d = 37, 8, 8
    nb = math.ceil(S / bs)
    k = rng.standard_normal((nb, bs, 2, d)) * 3
    v = rng.standard_normal((nb, bs, 2, d))
    v[..., -1] = 1.0  # the last value column is constant
    q = rng.standard_normal((2, 4, d))
    bt = np.stack([np.arange(nb), np.arange(nb)[::-1]]).astype(np.int32)
    out, _ = _gqa(q, k, v, bt, np.array([S, 20], np.int32), 0.9)
    np.testing.assert_allclose(out[:, -1], 1.0, rtol=0, atol=1e-12)
