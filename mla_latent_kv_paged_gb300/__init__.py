"""Python binding of the GB300 MLA latent-KV paged decode library.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libmla_gb300.so`` (built in-tree from ``csrc/``). Tensors are
torch tensors on the current CUDA device; the calls enqueue work on
``torch.cuda.current_stream()`` (or the stream given) and return at once.
There is no CPU path: if the library is missing, importing the functions
below raises.

The names follow the C ABI in ``include/mla.h``:
  absorb_q      qt = q^C W_UK (per head), q^R copied to columns 512..575
  decode_paged  split-KV scores and softmax-weighted latent sums over pages
  combine       log-sum-exp merge of the split partials -> u, lse
  out_proj      out = u W_UV (per head)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_gb300.so")

D_NOPE, D_R, D_C, D_V, PAGE = 128, 64, 512, 128, 64
D_ROW = D_C + D_R
DEFAULT_SCALE = 1.0 / math.sqrt(D_NOPE + D_R)

STATUS = {
    0: "MLA_OK",
    1: "MLA_ERR_INVALID_ARG",
    2: "MLA_ERR_UNSUPPORTED_SHAPE",
    3: "MLA_ERR_WORKSPACE_TOO_SMALL",
    4: "MLA_ERR_CUDA",
    5: "MLA_ERR_TIMEOUT",
    6: "MLA_ERR_BOUNDS",
    7: "MLA_ERR_RANGE",
}

EXPORTS = [
    "mla_status_string", "mla_abi_version", "mla_cache_bytes_per_token", "mla_page_bytes",
    "mla_absorb_q", "mla_decode_default_splits", "mla_decode_workspace_bytes",
    "mla_decode_paged", "mla_decode_plan", "mla_decode_paged_planned", "mla_combine", "mla_out_proj",
    "mla_decode_noalloc_max_bytes", "mla_decode_noalloc",
    "mla_append_workspace_bytes", "mla_append_kv",
    "mla_merge_w_kq", "mla_absorb_q_latent",
    "mla_merge_w_comb", "mla_out_comb_workspace_bytes", "mla_out_comb",
    "mla_quantize_fp8", "mla_decode_paged_fp8", "mla_decode_paged_planned_fp8",
    "mla_copy16",
]


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


DEBUG_LIB_PATH = os.path.join(_HERE, "libmla_gb300_debug.so")
DEBUG_EXPORTS = ["mla_debug_read_counters", "mla_debug_reset", "mla_debug_set_wait_limit",
                 "mla_debug_set_skip_producer"]

_lock = threading.Lock()
_lib = None
_debug_lib = None


def build(force: bool = False, debug: bool = False) -> str:
    from . import _build
    return _build.build(force=force, debug=debug)


def lib():
    """The loaded C library (ctypes). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(LIB_PATH)
    return _lib


def debug_lib():
    """The test build of the library (include/mla_debug.h), built on first use: the same
    entry points plus the decode kernel's instrumentation. For tests only."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            build(debug=True)
            L = _load(DEBUG_LIB_PATH)
            L.mla_debug_read_counters.restype = ctypes.c_int
            L.mla_debug_read_counters.argtypes = [ctypes.c_void_p, ctypes.c_int]
            L.mla_debug_reset.restype = ctypes.c_int
            L.mla_debug_set_wait_limit.restype = ctypes.c_int
            L.mla_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
            L.mla_debug_set_skip_producer.restype = ctypes.c_int
            L.mla_debug_set_skip_producer.argtypes = [ctypes.c_int]
            _debug_lib = L
    return _debug_lib


def _load(path: str):
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; run __graft_entry__.build() first")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_status_string.argtypes = [i]
    L.mla_abi_version.restype = i
    L.mla_cache_bytes_per_token.restype = sz
    L.mla_cache_bytes_per_token.argtypes = [i, i]
    L.mla_page_bytes.restype = sz
    L.mla_page_bytes.argtypes = [i, i, i]
    L.mla_absorb_q.restype = i
    L.mla_absorb_q.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    L.mla_decode_default_splits.restype = i
    L.mla_decode_default_splits.argtypes = [i]
    L.mla_decode_workspace_bytes.restype = sz
    L.mla_decode_workspace_bytes.argtypes = [i, i, i, i]
    L.mla_decode_paged.restype = i
    L.mla_decode_paged.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp, vp]
    L.mla_decode_plan.restype = i
    L.mla_decode_plan.argtypes = [vp, i, i, i, i, i, i, i, vp, sz, vp, vp]
    L.mla_decode_paged_planned.restype = i
    L.mla_decode_paged_planned.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp, vp]
    L.mla_combine.restype = i
    L.mla_combine.argtypes = [vp, i, i, i, i, vp, vp, vp]
    L.mla_out_proj.restype = i
    L.mla_out_proj.argtypes = [vp, vp, vp, i, i, i, i, vp]
    L.mla_decode_noalloc_max_bytes.restype = sz
    L.mla_decode_noalloc.restype = i
    L.mla_decode_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, vp, vp]
    L.mla_append_workspace_bytes.restype = sz
    L.mla_append_workspace_bytes.argtypes = [i, i]
    L.mla_append_kv.restype = i
    L.mla_append_kv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp, vp]
    L.mla_merge_w_kq.restype = i
    L.mla_merge_w_kq.argtypes = [vp, vp, vp, i, i, i, i, vp]
    L.mla_absorb_q_latent.restype = i
    L.mla_absorb_q_latent.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    L.mla_merge_w_comb.restype = i
    L.mla_merge_w_comb.argtypes = [vp, vp, vp, i, i, i, i, vp]
    L.mla_out_comb_workspace_bytes.restype = sz
    L.mla_out_comb_workspace_bytes.argtypes = [i, i, i]
    L.mla_out_comb.restype = i
    L.mla_out_comb.argtypes = [vp, vp, vp, i, i, i, i, vp, sz, vp]
    L.mla_quantize_fp8.restype = i
    L.mla_quantize_fp8.argtypes = [vp, vp, vp, ctypes.c_int64, vp]
    L.mla_copy16.restype = i
    L.mla_copy16.argtypes = [vp, vp, sz, vp]
    L.mla_decode_paged_fp8.restype = i
    L.mla_decode_paged_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp, vp]
    L.mla_decode_paged_planned_fp8.restype = i
    L.mla_decode_paged_planned_fp8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp, vp]
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise MlaError(status, where)


def _bits(t):
    """bf16 tensors are passed as their raw 16-bit patterns."""
    import torch
    assert t.dtype in (torch.bfloat16, torch.int16, torch.uint16), t.dtype
    assert t.is_contiguous(), "tensors must be contiguous"
    return t


# ---------------------------------------------------------------- small helpers
def cache_bytes_per_token(d_c: int = D_C, d_r: int = D_R) -> int:
    return int(lib().mla_cache_bytes_per_token(d_c, d_r))


def page_bytes(page_size: int = PAGE, d_c: int = D_C, d_r: int = D_R) -> int:
    return int(lib().mla_page_bytes(page_size, d_c, d_r))


def default_splits(n_q: int) -> int:
    g = int(lib().mla_decode_default_splits(n_q))
    if g < 1:
        raise MlaError(4, "mla_decode_default_splits")
    return g


def workspace_bytes(B: int, n_q: int, H: int, num_splits: int) -> int:
    n = int(lib().mla_decode_workspace_bytes(B, n_q, H, num_splits))
    if n == 0:
        raise MlaError(1, "mla_decode_workspace_bytes")
    return n


# ---------------------------------------------------------------- the four calls
def absorb_q(q_nope, q_rope, w_uk, q_abs=None, stream=None):
    """q_nope [T,H,128], q_rope [T,H,64], w_uk [H,128,512] (bf16) -> q_abs [T,H,576]."""
    import torch
    T, H = q_nope.shape[0], q_nope.shape[1]
    if q_abs is None:
        q_abs = torch.empty((T, H, D_ROW), dtype=torch.bfloat16, device=q_nope.device)
    st = lib().mla_absorb_q(_ptr(_bits(q_nope)), _ptr(_bits(q_rope)), _ptr(_bits(w_uk)),
                            _ptr(_bits(q_abs)), T, H, q_nope.shape[-1], q_rope.shape[-1],
                            w_uk.shape[-1], _stream(stream))
    _check(st, "mla_absorb_q")
    return q_abs


def merge_w_kq(w_uq, w_uk, w_kq=None, stream=None):
    """Merged query-side weight: w_uq [d_q,H,128], w_uk [H,128,512] (bf16) -> w_kq [d_q,H,512]."""
    import torch
    d_q, H = w_uq.shape[0], w_uq.shape[1]
    if w_kq is None:
        w_kq = torch.empty((d_q, H, D_C), dtype=torch.bfloat16, device=w_uq.device)
    st = lib().mla_merge_w_kq(_ptr(_bits(w_uq)), _ptr(_bits(w_uk)), _ptr(_bits(w_kq)), d_q, H, w_uq.shape[-1],
                              w_uk.shape[-1], _stream(stream))
    _check(st, "mla_merge_w_kq")
    return w_kq


def absorb_q_latent(c_q, q_rope, w_kq, q_abs=None, stream=None):
    """c_q [T,d_q], q_rope [T,H,64], w_kq [d_q,H,512] (bf16) -> q_abs [T,H,576]."""
    import torch
    T, d_q = c_q.shape
    H = w_kq.shape[1]
    if q_abs is None:
        q_abs = torch.empty((T, H, D_ROW), dtype=torch.bfloat16, device=c_q.device)
    st = lib().mla_absorb_q_latent(_ptr(_bits(c_q)), _ptr(_bits(q_rope)), _ptr(_bits(w_kq)), _ptr(_bits(q_abs)),
                                   T, H, d_q, q_rope.shape[-1], w_kq.shape[-1], _stream(stream))
    _check(st, "mla_absorb_q_latent")
    return q_abs


def merge_w_comb(w_uv, w_o, w_comb=None, stream=None):
    """Merged value/output weight: w_uv [H,128,512], w_o [d_model,H,128] (bf16) -> w_comb [d_model,H,512]."""
    import torch
    H = w_uv.shape[0]
    d_model = w_o.shape[0]
    if w_comb is None:
        w_comb = torch.empty((d_model, H, D_C), dtype=torch.bfloat16, device=w_uv.device)
    st = lib().mla_merge_w_comb(_ptr(_bits(w_uv)), _ptr(_bits(w_o)), _ptr(_bits(w_comb)), H, w_uv.shape[1],
                                w_uv.shape[2], d_model, _stream(stream))
    _check(st, "mla_merge_w_comb")
    return w_comb


def out_comb_workspace_bytes(T: int, H: int, d_model: int) -> int:
    n = int(lib().mla_out_comb_workspace_bytes(T, H, d_model))
    if n == 0:
        raise MlaError(1, "mla_out_comb_workspace_bytes")
    return n


def out_comb(u, w_comb, out=None, *, workspace=None, stream=None):
    """u [T,H,512], w_comb [d_model,H,512] (bf16) -> out [T,d_model], the layer output."""
    import torch
    T, H = u.shape[0], u.shape[1]
    d_model = w_comb.shape[0]
    if out is None:
        out = torch.empty((T, d_model), dtype=torch.bfloat16, device=u.device)
    if workspace is None:
        workspace = torch.empty(out_comb_workspace_bytes(T, H, d_model), dtype=torch.uint8, device=u.device)
    st = lib().mla_out_comb(_ptr(_bits(u)), _ptr(_bits(w_comb)), _ptr(_bits(out)), T, H, u.shape[-1], d_model,
                            _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "mla_out_comb")
    return out


def decode_plan(seq_lens, *, n_q: int, H: int, max_pages: int, num_pages: int, num_splits: int | None = None,
                workspace=None, err_word=None, stream=None, page_size: int = PAGE):
    """The split plan alone, into ``workspace`` (allocated if None). Returns (workspace,
    num_splits); pass both to ``decode_paged(..., planned=True)``. ``page_size`` (64 or
    128 tokens) must be the cache's."""
    import torch
    B = seq_lens.shape[0]
    if num_splits is None:
        num_splits = default_splits(n_q)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(B, n_q, H, num_splits), dtype=torch.uint8, device=seq_lens.device)
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    st = lib().mla_decode_plan(_ptr(seq_lens), B, n_q, H, num_pages, page_size, max_pages, num_splits, _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(err_word), _stream(stream))
    _check(st, "mla_decode_plan")
    return workspace, num_splits


def decode_paged(q_abs, cache, block_table, seq_lens, *, n_q: int, num_splits: int | None = None,
                 softmax_scale: float = DEFAULT_SCALE, workspace=None, err_word=None, stream=None,
                 planned: bool = False):
    """Split-KV decode over the paged cache. Returns (workspace, num_splits).

    q_abs [B*n_q, H, 576] (or [B, n_q, H, 576]), cache [num_pages, page_size, 576] with
    page_size 64 or 128,
    block_table [B, max_pages] int32, seq_lens [B] int32 (contexts include the
    n_q new tokens). The workspace holds the plan and the partials for
    ``combine``.
    """
    import torch
    B, max_pages = block_table.shape
    H = q_abs.shape[-2]
    num_pages, page_size = cache.shape[0], cache.shape[1]
    if num_splits is None:
        num_splits = default_splits(n_q)
    need = workspace_bytes(B, n_q, H, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_abs.device)
    assert block_table.dtype == torch.int32 and block_table.is_contiguous()
    if planned:  # the workspace holds the plan written by decode_plan
        st = lib().mla_decode_paged_planned(_ptr(_bits(q_abs)), _ptr(_bits(cache)), _ptr(block_table), B, n_q, H,
                                            num_pages, page_size, max_pages, float(softmax_scale), num_splits,
                                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _ptr(err_word), _stream(stream))
        _check(st, "mla_decode_paged_planned")
        return workspace, num_splits
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    st = lib().mla_decode_paged(_ptr(_bits(q_abs)), _ptr(_bits(cache)), _ptr(block_table),
                                _ptr(seq_lens), B, n_q, H, num_pages, page_size, max_pages,
                                float(softmax_scale), num_splits, _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(err_word),
                                _stream(stream))
    _check(st, "mla_decode_paged")
    return workspace, num_splits


def combine(workspace, *, B: int, n_q: int, H: int, num_splits: int, u=None, lse=None, stream=None):
    """Merge the partials in ``workspace`` -> u [B*n_q, H, 512] bf16, lse [B*n_q, H] float."""
    import torch
    dev = workspace.device
    if u is None:
        u = torch.empty((B * n_q, H, D_C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B * n_q, H), dtype=torch.float32, device=dev)
    st = lib().mla_combine(_ptr(workspace), B, n_q, H, num_splits, _ptr(_bits(u)), _ptr(lse),
                           _stream(stream))
    _check(st, "mla_combine")
    return u, lse


def copy16(src, dst, stream=None):
    """Copy the bytes of tensor ``src`` into ``dst`` (same byte size, a multiple of 16,
    contiguous) with a kernel: device tensors or pinned host tensors, in any combination."""
    assert src.is_contiguous() and dst.is_contiguous(), "tensors must be contiguous"
    nbytes = src.numel() * src.element_size()
    assert nbytes == dst.numel() * dst.element_size(), "byte sizes differ"
    _check(lib().mla_copy16(_ptr(src), _ptr(dst), nbytes, _stream(stream)), "mla_copy16")
    return dst


def quantize_fp8(rows, scales, codes=None, stream=None):
    """e4m3 codes of bf16 rows [..., 576] with per-column scales [576] float32 (FP8 latent cache)."""
    import torch
    if codes is None:
        codes = torch.empty(rows.shape, dtype=torch.uint8, device=rows.device)
    assert scales.dtype == torch.float32 and scales.is_contiguous() and scales.numel() == D_ROW
    n_rows = rows.numel() // D_ROW
    st = lib().mla_quantize_fp8(_ptr(_bits(rows)), _ptr(scales), _ptr(codes), n_rows, _stream(stream))
    _check(st, "mla_quantize_fp8")
    return codes


def decode_paged_fp8(q_abs, cache8, scales, block_table, seq_lens, *, n_q: int, num_splits: int | None = None,
                     softmax_scale: float = DEFAULT_SCALE, workspace=None, err_word=None, stream=None,
                     planned: bool = False):
    """decode_paged on an FP8 cache: cache8 [num_pages, 64, 576] uint8 e4m3 codes, scales [576]
    float32 per column. Returns (workspace, num_splits) for ``combine``."""
    import torch
    B, max_pages = block_table.shape
    H = q_abs.shape[-2]
    num_pages, page_size = cache8.shape[0], cache8.shape[1]
    if num_splits is None:
        num_splits = default_splits(n_q)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(B, n_q, H, num_splits), dtype=torch.uint8, device=q_abs.device)
    assert cache8.dtype == torch.uint8 and cache8.is_contiguous()
    assert scales.dtype == torch.float32 and scales.is_contiguous()
    assert block_table.dtype == torch.int32 and block_table.is_contiguous()
    nb = workspace.numel() * workspace.element_size()
    if planned:
        st = lib().mla_decode_paged_planned_fp8(_ptr(_bits(q_abs)), _ptr(cache8), _ptr(scales), _ptr(block_table),
                                                B, n_q, H, num_pages, page_size, max_pages, float(softmax_scale),
                                                num_splits, _ptr(workspace), nb, _ptr(err_word), _stream(stream))
        _check(st, "mla_decode_paged_planned_fp8")
    else:
        assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
        st = lib().mla_decode_paged_fp8(_ptr(_bits(q_abs)), _ptr(cache8), _ptr(scales), _ptr(block_table),
                                        _ptr(seq_lens), B, n_q, H, num_pages, page_size, max_pages,
                                        float(softmax_scale), num_splits, _ptr(workspace), nb, _ptr(err_word),
                                        _stream(stream))
        _check(st, "mla_decode_paged_fp8")
    return workspace, num_splits


def decode_noalloc(q_abs, cache, block_table, seq_lens, *, n_q: int, u, lse=None, num_splits: int | None = None,
                   softmax_scale: float = DEFAULT_SCALE, err_word=None, stream=None):
    """decode_paged + combine with the scratch kept inside the library (no workspace).

    For callers that must not allocate device memory during a step: neither this
    wrapper nor the C call allocates, so the outputs come from the caller, u
    [B*n_q, H, 512] bf16 and (optional, None skips it) lse [B*n_q, H] float32. See
    ``mla_decode_noalloc`` in include/mla.h for the size limit and for the rule
    that calls overlapping on the GPU race on the shared scratch.
    """
    B, max_pages = block_table.shape
    H = q_abs.shape[-2]
    if num_splits is None:
        num_splits = default_splits(n_q)
    if u is None:
        raise ValueError("decode_noalloc: pass the output tensor u (this call allocates nothing)")
    st = lib().mla_decode_noalloc(_ptr(_bits(q_abs)), _ptr(_bits(cache)), _ptr(block_table), _ptr(seq_lens),
                                  B, n_q, H, cache.shape[0], cache.shape[1], max_pages, float(softmax_scale),
                                  num_splits, _ptr(_bits(u)), _ptr(lse), _ptr(err_word), _stream(stream))
    _check(st, "mla_decode_noalloc")
    return u, lse


def append_workspace_bytes(T: int, d_model: int) -> int:
    n = int(lib().mla_append_workspace_bytes(T, d_model))
    if n == 0:
        raise MlaError(1, "mla_append_workspace_bytes")
    return n


def append_kv(h, w_dkr, cache, block_table, seq_lens, *, n_q: int, rope_theta: float = 10000.0,
              workspace=None, err_word=None, stream=None):
    """Write the new tokens' cache rows: [h W^DKV ; RoPE(h W^KR)] into their pages.

    h [B*n_q, d_model] (or [B, n_q, d_model]) bf16, w_dkr [576, d_model] bf16
    (W^DKV and W^KR transposed, stacked), cache / block_table / seq_lens as for
    decode_paged (seq_lens already counting the new tokens). The workspace (fp32
    partial sums of the split d_model reduction; allocated when none is given)
    is returned for reuse.
    """
    import torch
    B, max_pages = block_table.shape
    d_model = h.shape[-1]
    need = append_workspace_bytes(B * n_q, d_model)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=h.device)
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
    st = lib().mla_append_kv(_ptr(_bits(h)), _ptr(_bits(w_dkr)), _ptr(_bits(cache)), _ptr(block_table),
                             _ptr(seq_lens), B, n_q, d_model, cache.shape[0], cache.shape[1], max_pages,
                             float(rope_theta), _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _ptr(err_word), _stream(stream))
    _check(st, "mla_append_kv")
    return workspace


def out_proj(u, w_uv, out=None, stream=None):
    """u [T,H,512], w_uv [H,128,512] (bf16) -> out [T,H,128]."""
    import torch
    T, H = u.shape[0], u.shape[1]
    if out is None:
        out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=u.device)
    st = lib().mla_out_proj(_ptr(_bits(u)), _ptr(_bits(w_uv)), _ptr(_bits(out)), T, H,
                            u.shape[-1], w_uv.shape[1], _stream(stream))
    _check(st, "mla_out_proj")
    return out


def decode_step(q_nope, q_rope, w_uk, w_uv, cache, block_table, seq_lens, *, n_q: int,
                num_splits: int | None = None, softmax_scale: float = DEFAULT_SCALE,
                bufs: dict | None = None, err_word=None, stream=None, fp8_scales=None):
    """One full decode step: decode_plan -> absorb_q -> decode_paged (planned) ->
    combine -> out_proj (the plan is computed beside the kernel before it).

    ``cache`` is the bf16 cache, or the FP8 cache (uint8 e4m3 codes of the same
    shape, from ``quantize_fp8``) together with its column scales ``fp8_scales``
    [576] float32, which the decode then reads through decode_paged_fp8.
    ``bufs`` may hold preallocated q_abs, workspace, u, lse, out tensors; steps
    enqueued back to back may share one workspace (the step's up-projection lets
    the next step's plan start only once the step has finished).
    Returns dict(q_abs, u, lse, out).
    """
    bufs = bufs or {}
    B, max_pages = block_table.shape
    T, H = q_nope.shape[0], q_nope.shape[1]
    ws, g = decode_plan(seq_lens, n_q=n_q, H=H, max_pages=max_pages, num_pages=cache.shape[0],
                        num_splits=num_splits, workspace=bufs.get("workspace"), err_word=err_word, stream=stream,
                        page_size=cache.shape[1])
    q_abs = absorb_q(q_nope, q_rope, w_uk, bufs.get("q_abs"), stream)
    import torch
    if cache.dtype == torch.uint8:
        if fp8_scales is None:
            raise ValueError("an FP8 cache (uint8 codes) needs its column scales fp8_scales")
        decode_paged_fp8(q_abs, cache, fp8_scales, block_table, seq_lens, n_q=n_q, num_splits=g,
                         softmax_scale=softmax_scale, workspace=ws, err_word=err_word, stream=stream, planned=True)
    else:
        decode_paged(q_abs, cache, block_table, seq_lens, n_q=n_q, num_splits=g, softmax_scale=softmax_scale,
                     workspace=ws, err_word=err_word, stream=stream, planned=True)
    u, lse = combine(ws, B=B, n_q=n_q, H=H, num_splits=g, u=bufs.get("u"), lse=bufs.get("lse"),
                     stream=stream)
    out = out_proj(u, w_uv, bufs.get("out"), stream)
    return dict(q_abs=q_abs, u=u, lse=lse, out=out, workspace=ws, num_splits=g)


class CapturedStep:
    """A whole decode step (decode_plan -> absorb_q -> decode_paged -> combine ->
    out_proj) captured once in a CUDA graph, for serving loops with fixed shapes.

    The step owns its query, workspace and output buffers; it keeps pointers to
    the caller's weights, cache, block_table and seq_lens, so changing their
    contents in place between calls (appending tokens, new pages) is seen by
    the next replay: the split plan is derived on the device from seq_lens
    every time. Shapes (batch, max pages per sequence, heads, n_q) and
    num_splits are fixed at construction. An FP8 cache (uint8 codes) is given with
    its column scales ``fp8_scales``, as for ``decode_step``. Calling the object copies the new
    queries in (from host or device tensors, asynchronously) and replays the
    graph on the current stream; the returned tensors are the step's own
    buffers, overwritten by the next call.

    With ``host_io=True`` the step also owns pinned host buffers (``.host``:
    q_nope, q_rope, block_table, seq_lens in, packed into one input area; out,
    lse out), and a second graph that copies the inputs to the device in one
    copy (a kernel that reads the pinned memory, ``copy16``) and runs the step
    on them, with out_proj and combine writing out and lse straight into the
    pinned buffers. One serving step is then: write the new inputs into
    ``.host``, call ``replay_host()``, synchronise the stream, read
    ``.host["out"]``. (That graph uses the block table and lengths of
    ``.host``, not the block_table / seq_lens tensors given here.)
    """

    def __init__(self, w_uk, w_uv, cache, block_table, seq_lens, *, n_q: int, num_splits: int | None = None,
                 softmax_scale: float = DEFAULT_SCALE, err_word=None, host_io: bool = False, fp8_scales=None):
        import torch
        B = block_table.shape[0]
        H = w_uk.shape[0]
        T = B * n_q
        dev = cache.device
        g = default_splits(n_q) if num_splits is None else num_splits
        bf = torch.bfloat16
        self.q_nope = torch.empty((T, H, D_NOPE), dtype=bf, device=dev)
        self.q_rope = torch.empty((T, H, D_R), dtype=bf, device=dev)
        self.bufs = dict(q_abs=torch.empty((T, H, D_ROW), dtype=bf, device=dev),
                         workspace=torch.empty(workspace_bytes(B, n_q, H, g), dtype=torch.uint8, device=dev),
                         u=torch.empty((T, H, D_C), dtype=bf, device=dev),
                         lse=torch.empty((T, H), dtype=torch.float32, device=dev),
                         out=torch.empty((T, H, D_V), dtype=bf, device=dev))
        self.q_nope.zero_()
        self.q_rope.zero_()
        args = (self.q_nope, self.q_rope, w_uk, w_uv, cache, block_table, seq_lens)
        kw = dict(n_q=n_q, num_splits=g, softmax_scale=softmax_scale, bufs=self.bufs, err_word=err_word,
                  fp8_scales=fp8_scales)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):  # one eager run: kernel attributes, module loading
            decode_step(*args, **kw)
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            decode_step(*args, **kw)
        self.num_splits = g
        self.host = None
        if host_io:
            # one packed input area, on the device and pinned on the host, so a
            # replay moves the inputs in a single copy; the outputs are written to
            # the pinned host area by the kernels that produce them
            def layout(parts):
                off, views = 0, {}
                for name, shape, dtype in parts:
                    n = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
                    views[name] = (off, n, shape, dtype)
                    off = (off + n + 255) // 256 * 256
                return off, views

            def carve(buf, views):
                return {k: buf[o:o + n].view(dt).view(shape) for k, (o, n, shape, dt) in views.items()}

            in_bytes, in_views = layout([("q_nope", self.q_nope.shape, bf), ("q_rope", self.q_rope.shape, bf),
                                         ("block_table", block_table.shape, torch.int32),
                                         ("seq_lens", seq_lens.shape, torch.int32)])
            out_bytes, out_views = layout([("out", (T, H, D_V), bf), ("lse", (T, H), torch.float32)])
            self._dev_in = torch.zeros(in_bytes, dtype=torch.uint8, device=dev)
            self._host_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
            self._host_out = torch.zeros(out_bytes, dtype=torch.uint8).pin_memory()
            d_in = carve(self._dev_in, in_views)
            self.host = {**carve(self._host_in, in_views), **carve(self._host_out, out_views)}
            self.host["block_table"].copy_(block_table.cpu())
            self.host["seq_lens"].copy_(seq_lens.cpu())
            io_bufs = dict(self.bufs, out=self.host["out"], lse=self.host["lse"])
            io_args = (d_in["q_nope"], d_in["q_rope"], w_uk, w_uv, cache, d_in["block_table"], d_in["seq_lens"])
            io_kw = dict(kw, bufs=io_bufs)

            # the input copy runs as a kernel of the library (mla_copy16): the GPU
            # reads the pinned buffer itself, as out_proj and combine write theirs
            def io_step():
                copy16(self._host_in, self._dev_in)
                decode_step(*io_args, **io_kw)

            self.graph_io = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph_io):
                io_step()

    def __call__(self, q_nope=None, q_rope=None):
        """q_nope [T,H,128], q_rope [T,H,64] (bf16, host or device); None keeps the previous ones."""
        if q_nope is not None:
            self.q_nope.copy_(q_nope, non_blocking=True)
        if q_rope is not None:
            self.q_rope.copy_(q_rope, non_blocking=True)
        self.graph.replay()
        return dict(q_abs=self.bufs["q_abs"], u=self.bufs["u"], lse=self.bufs["lse"], out=self.bufs["out"])

    def replay_host(self):
        """One step from and to the pinned host buffers ``.host`` (``host_io=True``):
        inputs copied in, the step writing out and lse into ``.host``, all inside
        one graph replay on the current stream. Synchronise before reading ``.host``."""
        if self.host is None:
            raise RuntimeError("CapturedStep was built without host_io=True")
        self.graph_io.replay()
