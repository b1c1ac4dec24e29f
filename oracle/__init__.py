"""fp64 CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the benchmark's CPU-baseline leg, never by the product library.  It
shares no code with the CUDA path.  The arithmetic lives in
``decattn_oracle.c`` (plain loops, double precision); this module compiles it
with gcc on first use and marshals numpy arrays through ctypes.

Array conventions (numpy, C-contiguous):
  16-bit element tensors are passed as ``uint16`` arrays holding the raw bits,
  with ``dtype`` naming the format ("fp16" or "bf16"); fp64 tensors as
  ``float64`` with dtype "f64".  Index tensors are ``int32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decattn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_DTYPES = {"fp16": 0, "bf16": 1, "f64": 2}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-std=c11", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            I64 = ctypes.c_int64
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = D
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = D
            lib.oracle_decode_array.argtypes = [P, I, I64, P]
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = D
            lib.oracle_dequant_e4m3.argtypes = [P, I64, I, I, P, P]
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_float_array.argtypes = [P, I64, P]
            lib.oracle_e4m3_from_float_array.restype = None
            lib.oracle_quant_e4m3.argtypes = [P, I, I64, I, I, P, P]
            lib.oracle_quant_e4m3.restype = None
            lib.oracle_decode_array.restype = None
            lib.oracle_cache_row.argtypes = [P, I, I, I, I, I]
            lib.oracle_cache_row.restype = I64
            lib.oracle_gqa_decode.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, D, P, I, I, I,
                                              P, P]
            lib.oracle_gqa_decode.restype = I
            lib.oracle_mla_decode.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, D, P, I, I, I,
                                              P, P]
            lib.oracle_mla_decode.restype = I
            lib.oracle_mla_explicit.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, D, P, P]
            lib.oracle_mla_explicit.restype = I
            lib.oracle_lse_merge.argtypes = [I, I, P, P, P, P]
            lib.oracle_lse_merge.restype = None
            lib.oracle_kv_bytes_per_token.argtypes = [I, I, I, I]
            lib.oracle_kv_bytes_per_token.restype = I64
            lib.oracle_mla_bytes_per_token.argtypes = [I, I, I, I]
            lib.oracle_mla_bytes_per_token.restype = I64
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _elems(a: np.ndarray, dtype: str) -> np.ndarray:
    want = np.float64 if dtype == "f64" else np.uint16
    if a.dtype != want:
        raise TypeError(f"oracle: expected {np.dtype(want).name} storage for dtype {dtype}, "
                        f"got {a.dtype}")
    return np.ascontiguousarray(a)


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    return r, r.shape[0]


def half_to_double(bits: np.ndarray) -> np.ndarray:
    """Decode raw IEEE binary16 bit patterns to float64."""
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    dst = np.empty(src.shape, dtype=np.float64)
    _load().oracle_decode_array(_ptr(src), 0, src.size, _ptr(dst))
    return dst


def bf16_to_double(bits: np.ndarray) -> np.ndarray:
    """Decode raw bfloat16 bit patterns to float64."""
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    dst = np.empty(src.shape, dtype=np.float64)
    _load().oracle_decode_array(_ptr(src), 1, src.size, _ptr(dst))
    return dst


def e4m3_to_double(codes: np.ndarray) -> np.ndarray:
    """Decode raw e4m3 codes (uint8) to float64."""
    src = np.ascontiguousarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.oracle_e4m3_to_double(int(c)) for c in src.reshape(-1)],
                    dtype=np.float64).reshape(src.shape)


def dequant_e4m3(codes: np.ndarray, scales) -> np.ndarray:
    """Dequantise an e4m3 cache [..., h_kv, d] with one scale per KV head."""
    src = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(np.asarray(scales, dtype=np.float64).reshape(-1))
    h_kv, d = src.shape[-2], src.shape[-1]
    assert sc.shape == (h_kv,)
    out = np.empty(src.shape, dtype=np.float64)
    _load().oracle_dequant_e4m3(_ptr(src), src.size // (h_kv * d), h_kv, d, _ptr(sc), _ptr(out))
    return out


def gqa_decode_fp8kv(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, *,
                     q_dtype: str, scale: float, rows=None, t_begin: int = 0, t_end: int = -1):
    """GQA decode over an e4m3 KV cache in fp64: dequantise K and V with their
    per-KV-head scales, then the plain GQA definition (gqa_decode).

    q [B, h_q, d] fp16/bf16 bits; k_codes, v_codes [num_blocks, block_size,
    h_kv, d] uint8; k_scale, v_scale [h_kv].
    """
    q64 = half_to_double(q) if q_dtype == "fp16" else bf16_to_double(q)
    return gqa_decode(q64, dequant_e4m3(k_codes, k_scale), dequant_e4m3(v_codes, v_scale),
                      block_table, seq_lens, dtype="f64", scale=scale, rows=rows,
                      t_begin=t_begin, t_end=t_end)


def e4m3_from_float32(y) -> np.ndarray:
    """e4m3 codes of float32 values: nearest finite value, ties to the even
    code, saturating at +-448, sign kept (oracle_e4m3_from_float)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    _load().oracle_e4m3_from_float_array(_ptr(y), y.size, _ptr(out))
    return out


def quant_e4m3(x_bits, dtype: str, scales) -> np.ndarray:
    """Quantise 16-bit values [..., h_kv, d] (raw bits) to e4m3 codes with one
    fp32 scale per KV head: code = e4m3(fp32(x) / scale[j])."""
    x = _elems(x_bits, dtype)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    h_kv, d = x.shape[-2], x.shape[-1]
    assert s.shape == (h_kv,)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_quant_e4m3(_ptr(x), _DTYPES[dtype], x.size // (h_kv * d), h_kv, d, _ptr(s),
                              _ptr(out))
    return out


def kv_append(cache, new_rows, positions, block_table):
    """Decode-step append: sequence b's new token row (new_rows[b], any shape
    matching one cache slot) is written to slot positions[b] % block_size of
    block block_table[b][positions[b] // block_size] of a copy of `cache`
    [num_blocks, block_size, ...].  A negative position skips the sequence; a
    position past the table or a block id outside [0, num_blocks) skips it
    and is reported.  Returns (new cache, {b: "bad_position" | "bad_block"})."""
    out = np.array(cache, copy=True)
    nb, bs = out.shape[0], out.shape[1]
    bt = np.asarray(block_table, dtype=np.int32)
    bad = {}
    for b, pos in enumerate(np.asarray(positions, dtype=np.int64).tolist()):
        if pos < 0:
            continue
        if pos // bs >= bt.shape[1]:
            bad[b] = "bad_position"
            continue
        blk = int(bt[b, pos // bs])
        if blk < 0 or blk >= nb:
            bad[b] = "bad_block"
            continue
        out[blk, pos % bs] = new_rows[b]
    return out, bad


def cache_row(block_table: np.ndarray, block_size: int, num_blocks: int, b: int, t: int) -> int:
    """Physical row (block * block_size + slot) of token t of sequence b, or -1."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    return int(_load().oracle_cache_row(_ptr(bt), bt.shape[1], block_size, num_blocks, b, t))


def gqa_decode(q, k_cache, v_cache, block_table, seq_lens, *, dtype: str, scale: float,
               rows=None, t_begin: int = 0, t_end: int = -1):
    """GQA/MHA/MQA decode in fp64.

    q [B, h_q, d]; k_cache, v_cache [num_blocks, block_size, h_kv, d];
    block_table [B, max_blocks_per_seq] int32; seq_lens [B] int32.
    rows: optional list of (b, i) pairs; default every (b, i), b-major.
    Returns (out [n_rows, d] float64, lse [n_rows] float64 natural log).
    """
    q = _elems(q, dtype)
    k_cache = _elems(k_cache, dtype)
    v_cache = _elems(v_cache, dtype)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, h_q, d = q.shape
    nb, bs, h_kv, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape and bt.shape[0] == B and sl.shape == (B,)
    r, n_rows = _rows(rows)
    n = n_rows if r is not None else B * h_q
    out = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    st = _load().oracle_gqa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _DTYPES[dtype],
                                   _ptr(bt), _ptr(sl), B, h_q, h_kv, d, nb, bs, bt.shape[1],
                                   float(scale), _ptr(r), n_rows, t_begin, t_end, _ptr(out),
                                   _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_gqa_decode failed with status {st}")
    return out, lse


def window_start(seq_len: int, window: int) -> int:
    """First position a query attends to under a sliding window of `window`
    tokens ("07 · MHA/MQA/GQA/MLA quick learn", on what sliding-window
    attention does differently: each token sees only the last W tokens).  The
    decode query is the sequence's newest token, already in the cache at
    position seq_len - 1, so the window is [seq_len - window, seq_len),
    clipped at 0."""
    return max(0, int(seq_len) - int(window))


def gqa_decode_window(q, k_cache, v_cache, block_table, seq_lens, *, dtype: str, scale: float,
                      window: int, rows=None):
    """Sliding-window GQA decode in fp64: the plain GQA definition
    (gqa_decode) over positions [window_start(L_b, window), L_b) of each
    sequence b.  Same arguments and results as gqa_decode."""
    if window < 1:
        raise ValueError("window must be >= 1")
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, h_q = np.shape(q)[0], np.shape(q)[1]
    if rows is None:
        rows = np.stack(np.meshgrid(np.arange(B), np.arange(h_q), indexing="ij"), -1).reshape(-1, 2)
    rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
    d = np.shape(q)[2]
    out = np.empty((rows.shape[0], d), dtype=np.float64)
    lse = np.empty((rows.shape[0],), dtype=np.float64)
    for b in np.unique(rows[:, 0]):
        sel = np.nonzero(rows[:, 0] == b)[0]
        o, l = gqa_decode(q, k_cache, v_cache, block_table, sl, dtype=dtype, scale=scale,
                          rows=rows[sel], t_begin=window_start(sl[b], window), t_end=-1)
        out[sel], lse[sel] = o, l
    return out, lse


def gqa_decode_fp8kv_window(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, *,
                            q_dtype: str, scale: float, window: int, rows=None):
    """Sliding-window decode over an e4m3 KV cache: dequantise (as in
    gqa_decode_fp8kv), then gqa_decode_window."""
    q64 = half_to_double(q) if q_dtype == "fp16" else bf16_to_double(q)
    return gqa_decode_window(q64, dequant_e4m3(k_codes, k_scale), dequant_e4m3(v_codes, v_scale),
                             block_table, seq_lens, dtype="f64", scale=scale, window=window,
                             rows=rows)


def mla_decode(q_abs, q_rope, cache, block_table, seq_lens, *, dtype: str, scale: float,
               rows=None, t_begin: int = 0, t_end: int = -1):
    """Absorbed MLA decode in fp64.

    q_abs [B, H, d_c]; q_rope [B, H, d_r]; cache [num_blocks, block_size, d_c + d_r].
    Returns (out [n_rows, d_c], lse [n_rows]).
    """
    q_abs = _elems(q_abs, dtype)
    q_rope = _elems(q_rope, dtype)
    cache = _elems(cache, dtype)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H, d_c = q_abs.shape
    d_r = q_rope.shape[2]
    nb, bs, width = cache.shape
    assert width == d_c + d_r and q_rope.shape[:2] == (B, H)
    r, n_rows = _rows(rows)
    n = n_rows if r is not None else B * H
    out = np.empty((n, d_c), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    st = _load().oracle_mla_decode(_ptr(q_abs), _ptr(q_rope), _ptr(cache), _DTYPES[dtype],
                                   _ptr(bt), _ptr(sl), B, H, d_c, d_r, nb, bs, bt.shape[1],
                                   float(scale), _ptr(r), n_rows, t_begin, t_end, _ptr(out),
                                   _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_mla_decode failed with status {st}")
    return out, lse


def mla_explicit(q_nope, q_rope, c, k_rope, w_uk, w_uv, *, scale: float):
    """Explicit per-head reconstruction MLA for one sequence (all fp64).

    q_nope [h, d_h], q_rope [h, d_r], c [S, d_c], k_rope [S, d_r],
    w_uk [h, d_c, d_h], w_uv [h, d_c, d_v].  Returns (out [h, d_v], scores [h, S]).
    """
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (q_nope, q_rope, c, k_rope, w_uk, w_uv)]
    q_nope, q_rope, c, k_rope, w_uk, w_uv = arrs
    h, d_h = q_nope.shape
    S, d_c = c.shape
    d_r = q_rope.shape[1]
    d_v = w_uv.shape[2]
    out = np.empty((h, d_v), dtype=np.float64)
    scores = np.empty((h, S), dtype=np.float64)
    st = _load().oracle_mla_explicit(*[_ptr(a) for a in arrs], S, h, d_c, d_h, d_r, d_v,
                                     float(scale), _ptr(out), _ptr(scores))
    if st != 0:
        raise ValueError(f"oracle_mla_explicit failed with status {st}")
    return out, scores


def mla_absorb_q(q_nope, w_uk, *, dtype: str) -> np.ndarray:
    """The query-side absorption ("MQA, GQA, and MLA", section 5: q_i . k_i =
    x (W_q^(i) W_uk^(i)^T) c^T, so the per-head query times W_uk^(i)^T scores
    directly against the cached latent): q_abs[b, i, :] = q_nope[b, i, :]
    W_uk^(i)^T in fp64.

    q_nope [B, H, d_h]; w_uk [H, d_c, d_h] with w_uk[i] = W_uk^(i) (k_i = c
    W_uk^(i)).  Returns [B, H, d_c] float64.
    """
    q = _elems(q_nope, dtype)
    w = _elems(w_uk, dtype)
    if dtype != "f64":
        q, w = _to_f64(q, dtype), _to_f64(w, dtype)
    return np.einsum("bie,ice->bic", q, w)


def mla_unabsorb_out(o_lat, w_uv_t, *, dtype: str) -> np.ndarray:
    """The value-side step after the latent attention: the head's output is
    its softmax-weighted latent times W_uv^(i) (v_i = c W_uv^(i), so
    sum_t p_t v_{i,t} = (sum_t p_t c_t) W_uv^(i)): out[b, i, :] =
    o_lat[b, i, :] W_uv^(i) in fp64.

    o_lat [B, H, d_c]; w_uv_t [H, d_v, d_c] with w_uv_t[i] = W_uv^(i)^T.
    Returns [B, H, d_v] float64.
    """
    o = _elems(o_lat, dtype)
    w = _elems(w_uv_t, dtype)
    if dtype != "f64":
        o, w = _to_f64(o, dtype), _to_f64(w, dtype)
    return np.einsum("bic,ivc->biv", o, w)


def _to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    return half_to_double(bits) if dtype == "fp16" else bf16_to_double(bits)


def lse_merge(o_parts, lse_parts):
    """Merge partial (o, lse) over disjoint token ranges. o_parts [n, d], lse_parts [n]."""
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    l = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o.shape
    out = np.empty((d,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    _load().oracle_lse_merge(n, d, _ptr(o), _ptr(l), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def kv_bytes_per_token(n_layers: int, n_kv: int, d_head: int, bytes_per_elem: int) -> int:
    return int(_load().oracle_kv_bytes_per_token(n_layers, n_kv, d_head, bytes_per_elem))


def mla_bytes_per_token(n_layers: int, d_c: int, d_r: int, bytes_per_elem: int) -> int:
    return int(_load().oracle_mla_bytes_per_token(n_layers, d_c, d_r, bytes_per_elem))


def num_threads() -> int:
    """OpenMP threads the oracle will use (OMP_NUM_THREADS, else the usable cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1
