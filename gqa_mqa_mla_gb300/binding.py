"""ctypes binding of libdecattn (include/decattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the current
stream.  If the shared library is missing the calls raise; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DECATTN_OK = 0
DECATTN_ERR_INVALID_ARG = -1
DECATTN_ERR_UNSUPPORTED = -2
DECATTN_ERR_WORKSPACE = -3
DECATTN_ERR_CUDA = -4
DECATTN_FP16 = 0
DECATTN_BF16 = 1
FLAG_BAD_BLOCK = 1
FLAG_BAD_SEQ_LEN = 2
FLAG_TIMEOUT = 4
MAX_SPLITS = 256

MLA_HEADS, MLA_D_C, MLA_D_R = 128, 512, 64

_DT = {torch.float16: DECATTN_FP16, torch.bfloat16: DECATTN_BF16}


class DecAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


class Launch(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_blocks", ctypes.c_int),
        ("block_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("max_seq_len", ctypes.c_int),
        ("num_splits", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("err_flag", ctypes.c_void_p),
        ("stream", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libdecattn.so (built by gqa_mqa_mla_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m gqa_mqa_mla_gb300.build` (no fallback exists)")
            L = ctypes.CDLL(path)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            S, I64 = ctypes.c_size_t, ctypes.c_int64
            LP = ctypes.POINTER(Launch)
            L.gqa_decode.argtypes = [P, P, P, P, P, P, I, I, I, F, LP]
            L.gqa_decode.restype = I
            L.gqa_decode_fp8kv.argtypes = [P, P, P, P, P, P, P, P, I, I, I, F, LP]
            L.gqa_decode_fp8kv.restype = I
            L.gqa_decode_window.argtypes = [P, P, P, P, P, P, I, I, I, F, I, LP]
            L.gqa_decode_window.restype = I
            L.gqa_decode_fp8kv_window.argtypes = [P, P, P, P, P, P, P, P, I, I, I, F, I, LP]
            L.gqa_decode_fp8kv_window.restype = I
            L.gqa_decode_window_plan_splits.argtypes = [I, I, I, I, I, I, I, I, I]
            L.gqa_decode_window_plan_splits.restype = I
            L.gqa_kv_append.argtypes = [P, P, P, P, P, P, I, I, LP]
            L.gqa_kv_append.restype = I
            L.gqa_kv_append_fp8kv.argtypes = [P, P, P, P, P, P, P, P, I, I, LP]
            L.gqa_kv_append_fp8kv.restype = I
            L.mla_kv_append.argtypes = [P, P, P, P, LP]
            L.mla_kv_append.restype = I
            L.mla_absorb_q.argtypes = [P, P, P, I, I, I, I, I, P, P]
            L.mla_absorb_q.restype = I
            L.mla_unabsorb_out.argtypes = [P, P, P, I, I, I, I, I, P, P]
            L.mla_unabsorb_out.restype = I
            L.mla_decode.argtypes = [P, P, P, P, P, P, F, LP]
            L.mla_decode.restype = I
            L.gqa_decode_plan_splits.argtypes = [I, I, I, I, I, I]
            L.gqa_decode_plan_splits.restype = I
            L.gqa_decode_fp8kv_plan_splits.argtypes = [I, I, I, I, I, I]
            L.gqa_decode_fp8kv_plan_splits.restype = I
            L.mla_decode_plan_splits.argtypes = [I, I, I]
            L.mla_decode_plan_splits.restype = I
            L.gqa_decode_workspace_size.argtypes = [I, I, I, I]
            L.gqa_decode_workspace_size.restype = S
            L.mla_decode_workspace_size.argtypes = [I, I]
            L.mla_decode_workspace_size.restype = S
            L.decattn_kv_bytes_per_token.argtypes = [I, I, I, I]
            L.decattn_kv_bytes_per_token.restype = I64
            L.decattn_mla_bytes_per_token.argtypes = [I, I, I, I]
            L.decattn_mla_bytes_per_token.restype = I64
            L.decattn_status_string.argtypes = [I]
            L.decattn_status_string.restype = ctypes.c_char_p
            L.decattn_selftest_wait_timeout.argtypes = [P, P, I, P]
            L.decattn_selftest_wait_timeout.restype = I
            L.decattn_version.argtypes = []
            L.decattn_version.restype = I
            _lib = L
    return _lib


def selftest_wait_timeout(limit_us: int = 1000, device="cuda"):
    """Run the bounded-wait self test; returns (err_flag, result list of 5 ints)."""
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    res = torch.full((5,), -1, dtype=torch.int32, device=device)
    st = lib().decattn_selftest_wait_timeout(flag.data_ptr(), res.data_ptr(), int(limit_us),
                                              _stream_handle(None))
    if st != DECATTN_OK:
        raise DecAttnError("decattn_selftest_wait_timeout", st)
    torch.cuda.synchronize()
    return int(flag.item()), res.cpu().tolist()


def status_string(status: int) -> str:
    return lib().decattn_status_string(int(status)).decode()


def kv_bytes_per_token(n_layers: int, n_kv: int, d_head: int, bytes_per_elem: int) -> int:
    return int(lib().decattn_kv_bytes_per_token(n_layers, n_kv, d_head, bytes_per_elem))


def mla_bytes_per_token(n_layers: int, d_c: int, d_rope: int, bytes_per_elem: int) -> int:
    return int(lib().decattn_mla_bytes_per_token(n_layers, d_c, d_rope, bytes_per_elem))


def gqa_plan_splits(batch: int, h_q: int, h_kv: int, max_seq_len: int, d_head: int = 128,
                    num_sms: int = 0) -> int:
    r = lib().gqa_decode_plan_splits(batch, h_q, h_kv, d_head, max_seq_len, num_sms)
    if r < 0:
        raise DecAttnError("gqa_decode_plan_splits", r)
    return r


def gqa_fp8_plan_splits(batch: int, h_q: int, h_kv: int, max_seq_len: int, d_head: int = 128,
                        num_sms: int = 0) -> int:
    r = lib().gqa_decode_fp8kv_plan_splits(batch, h_q, h_kv, d_head, max_seq_len, num_sms)
    if r < 0:
        raise DecAttnError("gqa_decode_fp8kv_plan_splits", r)
    return r


def gqa_window_plan_splits(batch: int, h_q: int, h_kv: int, max_seq_len: int, window: int,
                           block_size: int, kv_bytes: int = 2, d_head: int = 128,
                           num_sms: int = 0) -> int:
    r = lib().gqa_decode_window_plan_splits(batch, h_q, h_kv, d_head, max_seq_len, window,
                                            block_size, kv_bytes, num_sms)
    if r < 0:
        raise DecAttnError("gqa_decode_window_plan_splits", r)
    return r


def mla_plan_splits(batch: int, max_seq_len: int, num_sms: int = 0) -> int:
    r = lib().mla_decode_plan_splits(batch, max_seq_len, num_sms)
    if r < 0:
        raise DecAttnError("mla_decode_plan_splits", r)
    return r


def gqa_workspace_size(batch: int, h_q: int, num_splits: int, d_head: int = 128) -> int:
    return int(lib().gqa_decode_workspace_size(batch, h_q, d_head, num_splits))


def mla_workspace_size(batch: int, num_splits: int) -> int:
    return int(lib().mla_decode_workspace_size(batch, num_splits))


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_launch(batch, num_blocks, block_size, max_blocks_per_seq, max_seq_len, num_splits,
                dtype, workspace=None, workspace_bytes=0, err_flag=None, stream=None) -> Launch:
    return Launch(batch, num_blocks, block_size, max_blocks_per_seq, max_seq_len, num_splits,
                  dtype, workspace, workspace_bytes, err_flag, stream)


def gqa_decode(q, k_cache, v_cache, block_table, seq_lens, *, scale: float, max_seq_len: int,
               out=None, num_splits: int = 0, workspace=None, err_flag=None, stream=None,
               window: int | None = None):
    """MHA/GQA/MQA decode through the C ABI; returns out [B, h_q, d].

    q [B, h_q, d]; k_cache/v_cache [num_blocks, block_size, h_kv, d];
    block_table int32 [B, max_blocks]; seq_lens int32 [B]; max_seq_len a host
    upper bound of seq_lens.  workspace: optional uint8 CUDA tensor (sized by
    gqa_workspace_size); allocated here when needed and not given.  window:
    attend only to each sequence's last `window` tokens (gqa_decode_window).
    """
    _check(q, "q", ndim=3)
    _check(k_cache, "k_cache", q.dtype, 4)
    _check(v_cache, "v_cache", q.dtype, 4)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    if q.dtype not in _DT:
        raise TypeError("q must be float16 or bfloat16")
    B, h_q, d = q.shape
    nb, bs, h_kv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache / v_cache shape mismatch")
    if h_kv < 1 or h_q % h_kv != 0:
        raise ValueError(f"h_q={h_q} is not a multiple of h_kv={h_kv}")
    if out is None:
        out = torch.empty_like(q)
    if num_splits:
        ns = num_splits
    elif window is None:
        ns = gqa_plan_splits(B, h_q, h_kv, max_seq_len, d)
    else:
        ns = gqa_window_plan_splits(B, h_q, h_kv, max_seq_len, window, bs, 2, d)
    need = gqa_workspace_size(B, h_q, ns, d)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    L = make_launch(B, nb, bs, block_table.shape[1], max_seq_len, ns, _DT[q.dtype],
                    _ptr(workspace), 0 if workspace is None else workspace.numel(),
                    _ptr(err_flag), _stream_handle(stream))
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
            seq_lens.data_ptr(), out.data_ptr(), h_q, h_kv, d, float(scale))
    if window is None:
        name, st = "gqa_decode", lib().gqa_decode(*args, ctypes.byref(L))
    else:
        name = "gqa_decode_window"
        st = lib().gqa_decode_window(*args, int(window), ctypes.byref(L))
    if st != DECATTN_OK:
        raise DecAttnError(name, st)
    return out


def gqa_decode_window(q, k_cache, v_cache, block_table, seq_lens, *, window: int, **kw):
    """gqa_decode restricted to each sequence's last `window` tokens."""
    return gqa_decode(q, k_cache, v_cache, block_table, seq_lens, window=window, **kw)


def gqa_decode_fp8kv(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, *,
                     scale: float, max_seq_len: int, out=None, num_splits: int = 0,
                     workspace=None, err_flag=None, stream=None, window: int | None = None):
    """GQA decode over an 8-bit (e4m3) KV cache through the C ABI; returns out.

    q [B, h_q, d] fp16/bf16; k_codes/v_codes uint8 (or float8_e4m3fn)
    [num_blocks, block_size, h_kv, d]; k_scale/v_scale float32 [h_kv] (the
    value of KV head j is e4m3(code) * scale[j]); the rest as gqa_decode
    (window: gqa_decode_fp8kv_window).
    """
    _check(q, "q", ndim=3)
    if q.dtype not in _DT:
        raise TypeError("q must be float16 or bfloat16")
    if k_codes.dtype == torch.float8_e4m3fn:
        k_codes = k_codes.view(torch.uint8)
    if v_codes.dtype == torch.float8_e4m3fn:
        v_codes = v_codes.view(torch.uint8)
    _check(k_codes, "k_codes", torch.uint8, 4)
    _check(v_codes, "v_codes", torch.uint8, 4)
    _check(k_scale, "k_scale", torch.float32, 1)
    _check(v_scale, "v_scale", torch.float32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    B, h_q, d = q.shape
    nb, bs, h_kv, d2 = k_codes.shape
    if d2 != d or v_codes.shape != k_codes.shape:
        raise ValueError("k_codes / v_codes shape mismatch")
    if k_scale.shape != (h_kv,) or v_scale.shape != (h_kv,):
        raise ValueError("k_scale / v_scale must be [h_kv]")
    if h_kv < 1 or h_q % h_kv != 0:
        raise ValueError(f"h_q={h_q} is not a multiple of h_kv={h_kv}")
    if out is None:
        out = torch.empty_like(q)
    if num_splits:
        ns = num_splits
    elif window is None:
        ns = gqa_fp8_plan_splits(B, h_q, h_kv, max_seq_len, d)
    else:
        ns = gqa_window_plan_splits(B, h_q, h_kv, max_seq_len, window, bs, 1, d)
    need = gqa_workspace_size(B, h_q, ns, d)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    L = make_launch(B, nb, bs, block_table.shape[1], max_seq_len, ns, _DT[q.dtype],
                    _ptr(workspace), 0 if workspace is None else workspace.numel(),
                    _ptr(err_flag), _stream_handle(stream))
    args = (q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(), k_scale.data_ptr(),
            v_scale.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
            h_q, h_kv, d, float(scale))
    if window is None:
        name, st = "gqa_decode_fp8kv", lib().gqa_decode_fp8kv(*args, ctypes.byref(L))
    else:
        name = "gqa_decode_fp8kv_window"
        st = lib().gqa_decode_fp8kv_window(*args, int(window), ctypes.byref(L))
    if st != DECATTN_OK:
        raise DecAttnError(name, st)
    return out


def gqa_decode_fp8kv_window(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, *,
                            window: int, **kw):
    """gqa_decode_fp8kv restricted to each sequence's last `window` tokens."""
    return gqa_decode_fp8kv(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens,
                            window=window, **kw)


def _append_launch(new, cache, block_table, dtype, err_flag, stream) -> Launch:
    return make_launch(new.shape[0], cache.shape[0], cache.shape[1], block_table.shape[1], 0, 1,
                       _DT[dtype], None, 0, _ptr(err_flag), _stream_handle(stream))


def gqa_kv_append(k_new, v_new, positions, block_table, k_cache, v_cache, *, err_flag=None,
                  stream=None):
    """Write each sequence's new K/V rows [B, h_kv, d] into slot positions[b]
    of its paged 16-bit cache (in place); a negative position skips."""
    _check(k_new, "k_new", ndim=3)
    _check(v_new, "v_new", k_new.dtype, 3)
    _check(k_cache, "k_cache", k_new.dtype, 4)
    _check(v_cache, "v_cache", k_new.dtype, 4)
    _check(positions, "positions", torch.int32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    if k_new.dtype not in _DT:
        raise TypeError("k_new must be float16 or bfloat16")
    B, h_kv, d = k_new.shape
    if v_new.shape != k_new.shape or k_cache.shape[2:] != (h_kv, d) or \
            v_cache.shape != k_cache.shape or positions.shape != (B,) or block_table.shape[0] != B:
        raise ValueError("kv_append: shape mismatch")
    L = _append_launch(k_new, k_cache, block_table, k_new.dtype, err_flag, stream)
    st = lib().gqa_kv_append(k_new.data_ptr(), v_new.data_ptr(), positions.data_ptr(),
                             block_table.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), h_kv,
                             d, ctypes.byref(L))
    if st != DECATTN_OK:
        raise DecAttnError("gqa_kv_append", st)


def gqa_kv_append_fp8kv(k_new, v_new, k_scale, v_scale, positions, block_table, k_codes, v_codes,
                        *, err_flag=None, stream=None):
    """Quantise each sequence's new K/V rows [B, h_kv, d] (fp16/bf16) to e4m3
    codes with the per-KV-head scales and write them into slot positions[b]
    of the 8-bit cache (uint8 or float8_e4m3fn, in place)."""
    if k_codes.dtype == torch.float8_e4m3fn:
        k_codes = k_codes.view(torch.uint8)
    if v_codes.dtype == torch.float8_e4m3fn:
        v_codes = v_codes.view(torch.uint8)
    _check(k_new, "k_new", ndim=3)
    _check(v_new, "v_new", k_new.dtype, 3)
    _check(k_scale, "k_scale", torch.float32, 1)
    _check(v_scale, "v_scale", torch.float32, 1)
    _check(k_codes, "k_codes", torch.uint8, 4)
    _check(v_codes, "v_codes", torch.uint8, 4)
    _check(positions, "positions", torch.int32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    if k_new.dtype not in _DT:
        raise TypeError("k_new must be float16 or bfloat16")
    B, h_kv, d = k_new.shape
    if v_new.shape != k_new.shape or k_codes.shape[2:] != (h_kv, d) or \
            v_codes.shape != k_codes.shape or positions.shape != (B,) or \
            block_table.shape[0] != B or k_scale.shape != (h_kv,) or v_scale.shape != (h_kv,):
        raise ValueError("kv_append_fp8kv: shape mismatch")
    L = _append_launch(k_new, k_codes, block_table, k_new.dtype, err_flag, stream)
    st = lib().gqa_kv_append_fp8kv(k_new.data_ptr(), v_new.data_ptr(), k_scale.data_ptr(),
                                   v_scale.data_ptr(), positions.data_ptr(),
                                   block_table.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(),
                                   h_kv, d, ctypes.byref(L))
    if st != DECATTN_OK:
        raise DecAttnError("gqa_kv_append_fp8kv", st)


def mla_kv_append(latent_new, positions, block_table, latent_cache, *, err_flag=None,
                  stream=None):
    """Write each sequence's new latent row [B, 576] (c_t then the RoPE key)
    into slot positions[b] of the paged latent cache (in place)."""
    _check(latent_new, "latent_new", ndim=2)
    _check(latent_cache, "latent_cache", latent_new.dtype, 3)
    _check(positions, "positions", torch.int32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    if latent_new.dtype not in _DT:
        raise TypeError("latent_new must be float16 or bfloat16")
    B = latent_new.shape[0]
    if latent_new.shape[1] != 576 or latent_cache.shape[2] != 576 or positions.shape != (B,) or \
            block_table.shape[0] != B:
        raise ValueError("mla_kv_append: shape mismatch")
    L = _append_launch(latent_new, latent_cache, block_table, latent_new.dtype, err_flag, stream)
    st = lib().mla_kv_append(latent_new.data_ptr(), positions.data_ptr(), block_table.data_ptr(),
                             latent_cache.data_ptr(), ctypes.byref(L))
    if st != DECATTN_OK:
        raise DecAttnError("mla_kv_append", st)


def mla_absorb_q(q_nope, w_uk, *, out=None, err_flag=None, stream=None):
    """q_abs[b, i, :] = q_nope[b, i, :] W_uk^(i)^T through the C ABI.

    q_nope [B, H, d_h]; w_uk [H, d_c, d_h] (w_uk[i] = W_uk^(i)); returns
    q_abs [B, H, d_c], mla_decode's absorbed query.
    """
    _check(q_nope, "q_nope", ndim=3)
    _check(w_uk, "w_uk", q_nope.dtype, 3)
    if q_nope.dtype not in _DT:
        raise TypeError("q_nope must be float16 or bfloat16")
    B, H, d_h = q_nope.shape
    if w_uk.shape[0] != H or w_uk.shape[2] != d_h:
        raise ValueError("w_uk must be [H, d_c, d_h]")
    d_c = w_uk.shape[1]
    if out is None:
        out = torch.empty((B, H, d_c), dtype=q_nope.dtype, device=q_nope.device)
    _check(out, "out", q_nope.dtype, 3)
    st = lib().mla_absorb_q(q_nope.data_ptr(), w_uk.data_ptr(), out.data_ptr(), B, H, d_h, d_c,
                            _DT[q_nope.dtype], _ptr(err_flag), _stream_handle(stream))
    if st != DECATTN_OK:
        raise DecAttnError("mla_absorb_q", st)
    return out


def mla_unabsorb_out(o_lat, w_uv_t, *, out=None, err_flag=None, stream=None):
    """out[b, i, :] = o_lat[b, i, :] W_uv^(i) through the C ABI.

    o_lat [B, H, d_c] (mla_decode's output); w_uv_t [H, d_v, d_c] (w_uv_t[i]
    = W_uv^(i) transposed); returns [B, H, d_v].
    """
    _check(o_lat, "o_lat", ndim=3)
    _check(w_uv_t, "w_uv_t", o_lat.dtype, 3)
    if o_lat.dtype not in _DT:
        raise TypeError("o_lat must be float16 or bfloat16")
    B, H, d_c = o_lat.shape
    if w_uv_t.shape[0] != H or w_uv_t.shape[2] != d_c:
        raise ValueError("w_uv_t must be [H, d_v, d_c]")
    d_v = w_uv_t.shape[1]
    if out is None:
        out = torch.empty((B, H, d_v), dtype=o_lat.dtype, device=o_lat.device)
    _check(out, "out", o_lat.dtype, 3)
    st = lib().mla_unabsorb_out(o_lat.data_ptr(), w_uv_t.data_ptr(), out.data_ptr(), B, H, d_c,
                                d_v, _DT[o_lat.dtype], _ptr(err_flag), _stream_handle(stream))
    if st != DECATTN_OK:
        raise DecAttnError("mla_unabsorb_out", st)
    return out


def mla_decode(q_absorbed, q_rope, latent_cache, block_table, seq_lens, *, scale: float,
               max_seq_len: int, out=None, num_splits: int = 0, workspace=None, err_flag=None,
               stream=None):
    """Absorbed MLA decode through the C ABI; returns out [B, 128, 512]."""
    _check(q_absorbed, "q_absorbed", ndim=3)
    _check(q_rope, "q_rope", q_absorbed.dtype, 3)
    _check(latent_cache, "latent_cache", q_absorbed.dtype, 3)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    if q_absorbed.dtype not in _DT:
        raise TypeError("q_absorbed must be float16 or bfloat16")
    B = q_absorbed.shape[0]
    if q_absorbed.shape != (B, MLA_HEADS, MLA_D_C) or q_rope.shape != (B, MLA_HEADS, MLA_D_R):
        raise ValueError("q_absorbed must be [B,128,512] and q_rope [B,128,64]")
    nb, bs, width = latent_cache.shape
    if width != MLA_D_C + MLA_D_R:
        raise ValueError("latent_cache must be [num_blocks, block_size, 576]")
    if out is None:
        out = torch.empty_like(q_absorbed)
    ns = num_splits if num_splits else mla_plan_splits(B, max_seq_len)
    need = mla_workspace_size(B, ns)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_absorbed.device)
    L = make_launch(B, nb, bs, block_table.shape[1], max_seq_len, ns, _DT[q_absorbed.dtype],
                    _ptr(workspace), 0 if workspace is None else workspace.numel(),
                    _ptr(err_flag), _stream_handle(stream))
    st = lib().mla_decode(q_absorbed.data_ptr(), q_rope.data_ptr(), latent_cache.data_ptr(),
                          block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                          float(scale), ctypes.byref(L))
    if st != DECATTN_OK:
        raise DecAttnError("mla_decode", st)
    return out
