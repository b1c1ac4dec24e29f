"""libdecattn: GB300-native single-token decode attention over a paged KV cache.

MHA / GQA / MQA (``gqa_decode``, ``gqa_decode_fp8kv`` over an 8-bit e4m3 KV
cache, and their sliding-window forms ``gqa_decode_window`` /
``gqa_decode_fp8kv_window``) and absorbed MLA (``mla_decode``), plus the decode
step's cache write (``gqa_kv_append``, ``gqa_kv_append_fp8kv``,
``mla_kv_append``) and MLA's absorption GEMMs (``mla_absorb_q``,
``mla_unabsorb_out``): hand-written CUDA kernels for sm_103a behind a C ABI
(include/decattn.h).  This package is the thin Python binding; ``synth``
draws seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    DecAttnError,
    FLAG_BAD_BLOCK,
    FLAG_BAD_SEQ_LEN,
    FLAG_TIMEOUT,
    gqa_decode,
    gqa_decode_fp8kv,
    gqa_decode_fp8kv_window,
    gqa_decode_window,
    gqa_fp8_plan_splits,
    gqa_kv_append,
    gqa_kv_append_fp8kv,
    gqa_plan_splits,
    gqa_window_plan_splits,
    gqa_workspace_size,
    kv_bytes_per_token,
    lib,
    library_path,
    mla_bytes_per_token,
    mla_absorb_q,
    mla_decode,
    mla_kv_append,
    mla_plan_splits,
    mla_unabsorb_out,
    mla_workspace_size,
    status_string,
)

__version__ = "0.1.0"
