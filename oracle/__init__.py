"""CPU oracle for MLA latent-KV decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package. It wraps ``mla_oracle.c`` (plain C, fp64 and fp32
loops, OpenMP over query rows) through ctypes. It shares no code with the CUDA
library in ``mla_latent_kv_paged_gb300``.

Every function takes the logical arrays produced by ``mla_inputs`` (bf16 bit
patterns in uint16 arrays) and returns float64 (or float32) numpy arrays.
Parity status of each function is listed in ``PINS`` below; all are pinned by
tests in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None
_mutants = {}

PINS = {
    "absorbed_f64": "pinned: equals the explicit path (1e-10), torch SDPA on explicit K/V, closed forms",
    "explicit_f64": "pinned: torch SDPA on the same explicit K/V; softmax rows sum to 1",
    "absorbed_probs_f64": "pinned: content+positional split equals the concatenated dot",
    "explicit_keys_f64": "pinned: rank <= d_c; equals numpy matmul",
    "split_partials_f64": "pinned: one piece equals the unsplit result; merge identity",
    "combine_f64": "pinned: merge of the pieces equals the unsplit absorbed result",
    "absorbed_f32": "baseline only (timed); agrees with the fp64 path to fp32 rounding",
    "absorb_q_f64": "pinned: numpy matmul; equals the q_abs of absorbed_f64",
    "out_proj_f64": "pinned: numpy matmul; W_UV applied to absorbed_f64's u gives its out",
    "append_f64": "pinned: numpy matmul; the generator's rotation; identity weights; position 0; "
                  "norm and relative-position properties of the rotation",
    "merge_w_kq_f64": "pinned: numpy per-head matmul; identity W_UQ gives W_UK; scores through the "
                      "merged weight equal the explicit keys' scores",
    "absorb_latent_f64": "pinned: equals absorb_q_f64 on the unmerged two-step query (associativity); "
                         "zero and one-hot compressed queries",
    "merge_w_comb_f64": "pinned: numpy per-head product; an identity output projection gives W_UV",
    "out_comb_f64": "pinned: equals out_proj_f64 followed by the output projection (associativity); "
                    "identity output projection gives out_proj_f64's heads side by side",
    "e4m3_decode": "pinned: torch's float8_e4m3fn values for all 256 codes; 1.0, 448, 2^-9, NaN codes",
    "dequant_fp8_f64": "pinned: the generator's quantiser round trip within e4m3's half-quantum bound",
    "absorbed_fp8_f64": "pinned: equals absorbed_f64 bit for bit when the dequantised latents are the bf16 "
                        "inputs (scale 1, e4m3-exact values)",
}


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile the oracle shared library with gcc (OpenMP if available).

    ``mutant`` > 0 builds a separate copy with one planted mistake (see the
    MLA_ORACLE_MUTANT comment in the C source); only the pin-sensitivity
    tests use it.
    """
    os.makedirs(_BUILD, exist_ok=True)
    path = _LIB_PATH if not mutant else os.path.join(_BUILD, f"libmla_oracle_mutant{mutant}.so")
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", f"-DMLA_ORACLE_MUTANT={int(mutant)}",
            _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, path)
    return path


def mutant_absorbed_f64(mutant: int, inp, rows=None, scale=None):
    """absorbed_f64 computed by a copy of the oracle with planted mistake ``mutant``."""
    with _lock:
        if mutant not in _mutants:
            lib = ctypes.CDLL(build(mutant=mutant))
            _mutants[mutant] = lib
    return absorbed_f64(inp, rows, scale, _lib_override=_mutants[mutant])


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB_PATH)
            _lib.mla_oracle_num_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def num_threads() -> int:
    return int(_load().mla_oracle_num_threads())


def default_scale(d_nope: int = 128, d_r: int = 64) -> float:
    """1/sqrt(d_k) with d_k = d_nope + d_r, the query/key width after concatenation."""
    return 1.0 / math.sqrt(d_nope + d_r)


def _common(inp):
    arrs = dict(
        q_nope=np.ascontiguousarray(inp.q_nope, dtype=np.uint16),
        q_rope=np.ascontiguousarray(inp.q_rope, dtype=np.uint16),
        c=np.ascontiguousarray(inp.c, dtype=np.uint16),
        kr=np.ascontiguousarray(inp.kr, dtype=np.uint16),
        seq_off=np.ascontiguousarray(inp.seq_off, dtype=np.int64),
        seq_lens=np.ascontiguousarray(inp.seq_lens, dtype=np.int32),
        w_uk=np.ascontiguousarray(inp.w_uk, dtype=np.uint16),
        w_uv=np.ascontiguousarray(inp.w_uv, dtype=np.uint16),
    )
    d_nope = arrs["q_nope"].shape[-1]
    d_r = arrs["q_rope"].shape[-1]
    d_c = arrs["c"].shape[-1]
    d_v = arrs["w_uv"].shape[1]
    return arrs, (inp.B, inp.n_q, inp.H, d_nope, d_r, d_c, d_v)


def all_rows(inp) -> np.ndarray:
    return np.arange(inp.B * inp.n_q * inp.H, dtype=np.int64)


def absorbed_f64(inp, rows=None, scale=None, _lib_override=None):
    """Absorbed MLA decode in fp64. Returns dict q_abs [n,d_c+d_r], u [n,d_c], lse [n], out [n,d_v]."""
    lib = _lib_override if _lib_override is not None else _load()
    a, dims = _common(inp)
    B, n_q, H, d_nope, d_r, d_c, d_v = dims
    rows = all_rows(inp) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = default_scale(d_nope, d_r) if scale is None else scale
    n = len(rows)
    q_abs = np.empty((n, d_c + d_r)); u = np.empty((n, d_c)); lse = np.empty(n); out = np.empty((n, d_v))
    rc = lib.mla_oracle_absorbed_f64(
        _p(a["q_nope"]), _p(a["q_rope"]), _p(a["c"]), _p(a["kr"]), _p(a["seq_off"]), _p(a["seq_lens"]),
        _p(a["w_uk"]), _p(a["w_uv"]), *[ctypes.c_int(x) for x in dims], ctypes.c_double(scale),
        _p(rows), ctypes.c_int64(n), _p(q_abs), _p(u), _p(lse), _p(out))
    if rc != 0:
        raise ValueError("oracle: bad row or context shorter than n_q")
    return dict(q_abs=q_abs, u=u, lse=lse, out=out)


def explicit_f64(inp, rows=None, scale=None, max_tokens=0):
    """Explicit (non-absorbed) attention in fp64: K = W_UK c, V = W_UV c per token."""
    lib = _load()
    a, dims = _common(inp)
    B, n_q, H, d_nope, d_r, d_c, d_v = dims
    rows = all_rows(inp) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = default_scale(d_nope, d_r) if scale is None else scale
    n = len(rows)
    lse = np.empty(n); out = np.empty((n, d_v))
    logits = np.empty((n, max_tokens)) if max_tokens else None
    probs = np.empty((n, max_tokens)) if max_tokens else None
    rc = lib.mla_oracle_explicit_f64(
        _p(a["q_nope"]), _p(a["q_rope"]), _p(a["c"]), _p(a["kr"]), _p(a["seq_off"]), _p(a["seq_lens"]),
        _p(a["w_uk"]), _p(a["w_uv"]), *[ctypes.c_int(x) for x in dims], ctypes.c_double(scale),
        _p(rows), ctypes.c_int64(n), _p(lse), _p(out), _p(logits), _p(probs), ctypes.c_int64(max_tokens))
    if rc != 0:
        raise ValueError("oracle: bad row or context shorter than n_q")
    res = dict(lse=lse, out=out)
    if max_tokens:
        res.update(logits=logits, probs=probs)
    return res


def absorbed_probs_f64(inp, row, scale=None):
    """Per-token content term, positional term, logits and probabilities of one row."""
    lib = _load()
    a, dims = _common(inp)
    B, n_q, H, d_nope, d_r, d_c, d_v = dims
    scale = default_scale(d_nope, d_r) if scale is None else scale
    b = row // (H * n_q)
    n_max = int(inp.seq_lens[b])
    content = np.zeros(n_max); pos = np.zeros(n_max); logits = np.zeros(n_max); probs = np.zeros(n_max)
    n = lib.mla_oracle_absorbed_probs_f64(
        _p(a["q_nope"]), _p(a["q_rope"]), _p(a["c"]), _p(a["kr"]), _p(a["seq_off"]), _p(a["seq_lens"]),
        _p(a["w_uk"]), *[ctypes.c_int(x) for x in dims[:6]], ctypes.c_double(scale), ctypes.c_int64(row),
        _p(content), _p(pos), _p(logits), _p(probs))
    if n < 0:
        raise ValueError("oracle: bad row")
    return dict(content=content[:n], pos=pos[:n], logits=logits[:n], probs=probs[:n])


def explicit_keys_f64(c_bits: np.ndarray, w_uk_bits: np.ndarray, h: int) -> np.ndarray:
    """K[s][i] = sum_c W_UK[h][i][c] c_s[c] for all rows of ``c_bits``."""
    lib = _load()
    c_bits = np.ascontiguousarray(c_bits, dtype=np.uint16)
    w_uk_bits = np.ascontiguousarray(w_uk_bits, dtype=np.uint16)
    L, d_c = c_bits.shape
    d_nope = w_uk_bits.shape[1]
    k = np.empty((L, d_nope))
    lib.mla_oracle_explicit_keys_f64(_p(c_bits), _p(w_uk_bits), ctypes.c_int64(L), ctypes.c_int(h),
                                     ctypes.c_int(d_nope), ctypes.c_int(d_c), _p(k))
    return k


def split_partials_f64(inp, pieces, rows=None, scale=None):
    """Normalised partials (u_k, lse_k) over token ranges ``pieces`` [[t0, t1), ...]."""
    lib = _load()
    a, dims = _common(inp)
    B, n_q, H, d_nope, d_r, d_c, d_v = dims
    rows = all_rows(inp) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = default_scale(d_nope, d_r) if scale is None else scale
    pieces = np.ascontiguousarray(np.asarray(pieces, dtype=np.int64).reshape(-1, 2))
    n, k = len(rows), len(pieces)
    u = np.empty((n, k, d_c)); lse = np.empty((n, k))
    rc = lib.mla_oracle_split_partials_f64(
        _p(a["q_nope"]), _p(a["q_rope"]), _p(a["c"]), _p(a["kr"]), _p(a["seq_off"]), _p(a["seq_lens"]),
        _p(a["w_uk"]), *[ctypes.c_int(x) for x in dims[:6]], ctypes.c_double(scale),
        _p(rows), ctypes.c_int64(n), _p(pieces), ctypes.c_int(k), _p(u), _p(lse))
    if rc != 0:
        raise ValueError("oracle: bad row")
    return dict(u=u, lse=lse)


def combine_f64(u_part: np.ndarray, lse_part: np.ndarray):
    """Log-sum-exp merge of normalised partials: u_part [n,k,d_c], lse_part [n,k]."""
    lib = _load()
    u_part = np.ascontiguousarray(u_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    n, k, d_c = u_part.shape
    u = np.empty((n, d_c)); lse = np.empty(n)
    lib.mla_oracle_combine_f64(_p(u_part), _p(lse_part), ctypes.c_int64(n), ctypes.c_int(k),
                               ctypes.c_int(d_c), _p(u), _p(lse))
    return dict(u=u, lse=lse)


def absorbed_f32(inp, rows=None, scale=None):
    """fp32 absorbed loops (the timed CPU baseline). Returns u, lse, out as float32."""
    lib = _load()
    a, dims = _common(inp)
    B, n_q, H, d_nope, d_r, d_c, d_v = dims
    rows = all_rows(inp) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = default_scale(d_nope, d_r) if scale is None else scale
    n = len(rows)
    u = np.empty((n, d_c), np.float32); lse = np.empty(n, np.float32); out = np.empty((n, d_v), np.float32)
    rc = lib.mla_oracle_absorbed_f32(
        _p(a["q_nope"]), _p(a["q_rope"]), _p(a["c"]), _p(a["kr"]), _p(a["seq_off"]), _p(a["seq_lens"]),
        _p(a["w_uk"]), _p(a["w_uv"]), *[ctypes.c_int(x) for x in dims], ctypes.c_float(scale),
        _p(rows), ctypes.c_int64(n), _p(u), _p(lse), _p(out))
    if rc != 0:
        raise ValueError("oracle: bad row")
    return dict(u=u, lse=lse, out=out)


def absorb_q_f64(q_nope_bits, q_rope_bits, w_uk_bits):
    """The absorption step alone: [T,H,d_nope] x [H,d_nope,d_c] -> [T,H,d_c+d_r] (fp64)."""
    lib = _load()
    qn = np.ascontiguousarray(q_nope_bits, dtype=np.uint16)
    qr = np.ascontiguousarray(q_rope_bits, dtype=np.uint16)
    wk = np.ascontiguousarray(w_uk_bits, dtype=np.uint16)
    T, H, d_nope = qn.shape
    d_r, d_c = qr.shape[-1], wk.shape[-1]
    out = np.empty((T, H, d_c + d_r))
    lib.mla_oracle_absorb_q_f64(_p(qn), _p(qr), _p(wk), ctypes.c_int64(T), ctypes.c_int(H),
                                ctypes.c_int(d_nope), ctypes.c_int(d_r), ctypes.c_int(d_c), _p(out))
    return out


def out_proj_f64(u_bits, w_uv_bits):
    """The up-projection step alone: [T,H,d_c] x [H,d_v,d_c] -> [T,H,d_v] (fp64)."""
    lib = _load()
    u = np.ascontiguousarray(u_bits, dtype=np.uint16)
    wv = np.ascontiguousarray(w_uv_bits, dtype=np.uint16)
    T, H, d_c = u.shape
    d_v = wv.shape[1]
    out = np.empty((T, H, d_v))
    lib.mla_oracle_out_proj_f64(_p(u), _p(wv), ctypes.c_int64(T), ctypes.c_int(H), ctypes.c_int(d_c),
                                ctypes.c_int(d_v), _p(out))
    return out


def append_f64(h_bits: np.ndarray, w_dkr_bits: np.ndarray, pos, theta: float = 10000.0, d_c: int = 512):
    """Cache rows of new tokens: [c (d_c) ; rotated k^R (d_r)] for h [T][d_model] and the
    transposed weights w_dkr [d_c + d_r][d_model] (bf16 bits), positions pos [T]."""
    L = _load()
    h = np.ascontiguousarray(h_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_dkr_bits, dtype=np.uint16)
    T, d_model = h.shape
    D = w.shape[0]
    assert w.shape[1] == d_model and D > d_c and (D - d_c) % 2 == 0
    p = np.ascontiguousarray(pos, dtype=np.int64)
    assert p.shape == (T,)
    out = np.zeros((T, D), dtype=np.float64)
    L.mla_oracle_append_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
    L.mla_oracle_append_f64(_p(h), _p(w), _p(p), T, d_model, d_c, D - d_c, float(theta), _p(out))
    return out



def merge_w_kq_f64(w_uq_bits, w_uk_bits):
    """Merged query weight per head: w_uq [d_q][H][d_nope] x w_uk [H][d_nope][d_c] ->
    w_kq [d_q][H][d_c] (fp64), w_kq[k][h] = sum_i w_uq[k][h][i] w_uk[h][i]."""
    L = _load()
    wq = np.ascontiguousarray(w_uq_bits, dtype=np.uint16)
    wk = np.ascontiguousarray(w_uk_bits, dtype=np.uint16)
    d_q, H, d_nope = wq.shape
    assert wk.shape[:2] == (H, d_nope)
    d_c = wk.shape[2]
    out = np.empty((d_q, H, d_c))
    L.mla_oracle_merge_w_kq_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.mla_oracle_merge_w_kq_f64(_p(wq), _p(wk), d_q, H, d_nope, d_c, _p(out))
    return out


def absorb_latent_f64(c_q_bits, w_kq, q_rope_bits):
    """Absorbed query from the compressed query latent: c_q [T][d_q] (bf16 bits) x
    w_kq [d_q][H][d_c] (float64 values, or bf16 bits as uint16) -> [T][H][d_c + d_r],
    the positional query q_rope [T][H][d_r] copied behind (fp64)."""
    L = _load()
    cq = np.ascontiguousarray(c_q_bits, dtype=np.uint16)
    w = np.asarray(w_kq)
    if w.dtype == np.uint16:
        w = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    qr = np.ascontiguousarray(q_rope_bits, dtype=np.uint16)
    T, d_q = cq.shape
    assert w.shape[0] == d_q
    H, d_c = w.shape[1], w.shape[2]
    d_r = qr.shape[-1]
    assert qr.shape == (T, H, d_r)
    out = np.empty((T, H, d_c + d_r))
    L.mla_oracle_absorb_latent_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_void_p]
    L.mla_oracle_absorb_latent_f64(_p(cq), _p(w), _p(qr), T, H, d_q, d_r, d_c, _p(out))
    return out


def merge_w_comb_f64(w_uv_bits, w_o_bits):
    """Merged value/output weight per head: w_uv [H][d_v][d_c] x w_o [d_model][H][d_v] ->
    w_comb [d_model][H][d_c] (fp64), w_comb[n][h] = sum_v w_o[n][h][v] w_uv[h][v]."""
    L = _load()
    wv = np.ascontiguousarray(w_uv_bits, dtype=np.uint16)
    wo = np.ascontiguousarray(w_o_bits, dtype=np.uint16)
    H, d_v, d_c = wv.shape
    d_model = wo.shape[0]
    assert wo.shape == (d_model, H, d_v)
    out = np.empty((d_model, H, d_c))
    L.mla_oracle_merge_w_comb_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.mla_oracle_merge_w_comb_f64(_p(wv), _p(wo), H, d_v, d_c, d_model, _p(out))
    return out


def out_comb_f64(u_bits, w_comb):
    """Layer output through the merged weight: u [T][H][d_c] (bf16 bits) and w_comb
    [d_model][H][d_c] (float64 values, or bf16 bits as uint16) -> out [T][d_model] (fp64)."""
    L = _load()
    u = np.ascontiguousarray(u_bits, dtype=np.uint16)
    w = np.asarray(w_comb)
    if w.dtype == np.uint16:
        w = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T, H, d_c = u.shape
    d_model = w.shape[0]
    assert w.shape == (d_model, H, d_c)
    out = np.empty((T, d_model))
    L.mla_oracle_out_comb_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.mla_oracle_out_comb_f64(_p(u), _p(w), T, H, d_c, d_model, _p(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    """Values of e4m3 codes (uint8), from the format's definition (NaN codes -> NaN)."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib.mla_oracle_e4m3_decode.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    lib.mla_oracle_e4m3_decode(_p(c), c.size, _p(out))
    return out


def dequant_fp8_f64(codes, scales) -> np.ndarray:
    """Dequantised FP8 rows: codes [..., D] (uint8) times per-column scales [D] (float32), fp64."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    D = c.shape[-1]
    assert sc.shape == (D,)
    out = np.empty(c.shape, dtype=np.float64)
    lib.mla_oracle_dequant_fp8_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_void_p]
    lib.mla_oracle_dequant_fp8_f64(_p(c), _p(sc), c.size // D, D, _p(out))
    return out


def absorbed_lat_f64(inp, c, kr, rows=None, scale=None):
    """absorbed_f64 with the latents given as float64 arrays c [total][d_c], kr [total][d_r]."""
    lib = _load()
    a, dims = _common(inp)
    B, n_q, H, d_nope, d_r, d_c, d_v = dims
    c = np.ascontiguousarray(c, dtype=np.float64)
    kr = np.ascontiguousarray(kr, dtype=np.float64)
    assert c.shape == (inp.total_tokens, d_c) and kr.shape == (inp.total_tokens, d_r)
    rows = all_rows(inp) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = default_scale(d_nope, d_r) if scale is None else scale
    n = len(rows)
    q_abs = np.empty((n, d_c + d_r)); u = np.empty((n, d_c)); lse = np.empty(n); out = np.empty((n, d_v))
    rc = lib.mla_oracle_absorbed_lat_f64(
        _p(a["q_nope"]), _p(a["q_rope"]), _p(c), _p(kr), _p(a["seq_off"]), _p(a["seq_lens"]),
        _p(a["w_uk"]), _p(a["w_uv"]), *[ctypes.c_int(x) for x in dims], ctypes.c_double(scale),
        _p(rows), ctypes.c_int64(n), _p(q_abs), _p(u), _p(lse), _p(out))
    if rc != 0:
        raise ValueError("oracle: bad row or context shorter than n_q")
    return dict(q_abs=q_abs, u=u, lse=lse, out=out)


def absorbed_fp8_f64(inp, codes, scales, rows=None, scale=None):
    """The absorbed path on an FP8 latent cache: the logical rows' e4m3 codes [total][576]
    dequantised with the per-column scales, then the exact fp64 absorbed loops."""
    d_c = inp.c.shape[-1]
    deq = dequant_fp8_f64(codes, scales)
    return absorbed_lat_f64(inp, deq[:, :d_c], deq[:, d_c:], rows, scale)
