"""Seeded synthetic inputs for MLA latent-KV paged decode.

This module is shared by the CPU oracle tests, the CUDA parity tests and the
benchmark. It draws random numbers, rounds them to bf16, applies the rotary
position rotation that the cached positional key carries, and scatters the
logical cache rows into a shuffled page pool. It contains none of the decode
arithmetic (no absorption, scoring, softmax, aggregation or projection).

Workloads (all at DeepSeek-V3 head shape d_nope=128, d_r=64, d_c=512, d_v=128,
page size 64), following the worked numbers of the Huny's Dev Blog page "MLA
아키텍처 해부", section 5 (DeepSeek-V3 parameters n_h=128, d_h=128, d_c=512,
d_R=64):

  1 tiny     : B=2,   H=16,  context 256 each, n_q=1
  2 v3       : B=32,  H=128, context 4096 each, n_q=1
  3 ragged   : B=128, H=128, context ~ U{512..16384} per sequence, n_q=1
  4 long     : B=4,   H=128, context 131072 each, n_q=1
  5 multitok : B=64,  H=128, context 8192 each, n_q=2 (causal within the pair)

Recipe (seed = workload index - 1, numpy PCG64 ``default_rng(seed)``), in
draw order:

  1. seq_lens: constant, or ``rng.integers(512, 16385, B)`` for the ragged one.
  2. per sequence b in order: c_b ~ N(0,1) [L_b, 512], then k_raw_b ~ N(0,1)
     [L_b, 64] (float32 draws).
  3. q_nope ~ N(0,1) [B, n_q, H, 128], then q_raw ~ N(0,1) [B, n_q, H, 64].
  4. W_UK, W_UV ~ N(0,1) * (1/sqrt(512)) [H, 128, 512] each (standard
     deviation 1/sqrt(512), float32).
  5. Rotary rotation (interleaved pairs, theta = 10000) in float64: k_rope of
     token s at position s, q_rope of query j at position L_b - n_q + j.
  6. Every tensor is rounded float32 -> bf16 with round-to-nearest-even.
  7. Paging: physical page ids are a random permutation (``perm_seed``) of a
     pool with ``spare_pages`` extra pages; slack rows of each sequence's last
     page and all spare pages are filled with bf16 NaN; unused block-table
     entries are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D_NOPE = 128
D_R = 64
D_C = 512
D_V = 128
D_ROW = D_C + D_R  # 576 values per cached token
PAGE = 64
ROPE_THETA = 10000.0
BF16_NAN = np.uint16(0x7FC0)


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    H: int
    n_q: int
    context: int | None  # None => ragged draw
    spare_pages: int = 64

    @property
    def seed(self) -> int:
        return self.index - 1


WORKLOADS = {
    1: Workload(1, "tiny B=2 H=16 L=256", 2, 16, 1, 256, spare_pages=4),
    2: Workload(2, "v3 B=32 H=128 L=4096", 32, 128, 1, 4096),
    3: Workload(3, "ragged B=128 H=128 L~U[512,16384]", 128, 128, 1, None),
    4: Workload(4, "long B=4 H=128 L=131072", 4, 128, 1, 131072),
    5: Workload(5, "multitoken B=64 H=128 L=8192 n_q=2", 64, 128, 2, 8192),
}


# ----------------------------------------------------------------------------
# bf16 helpers (bit patterns held in uint16 arrays)
# ----------------------------------------------------------------------------
def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); NaN -> 0x7FC0.

    In 32-bit arithmetic: for every finite or infinite input the sum below stays
    under 2^32 (the largest bit pattern, -inf, is 0xFF800000); only NaN patterns
    can wrap, and those are replaced afterwards."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    t = u >> np.uint32(16)
    t &= np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    out = t.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# rotary rotation of the decoupled positional stream
# ----------------------------------------------------------------------------
def rope_rotate(x: np.ndarray, pos: np.ndarray, theta: float = ROPE_THETA) -> np.ndarray:
    """Rotate the last axis (even length d) pairwise: (x[2i], x[2i+1]) by pos*theta^(-2i/d).

    ``pos`` broadcasts against ``x[..., 0]``. Computed in float64.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    inv = theta ** (-np.arange(0, d, 2, dtype=np.float64) / d)  # [d/2]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv     # [..., d/2]
    cs, sn = np.cos(ang), np.sin(ang)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * cs - xo * sn
    out[..., 1::2] = xe * sn + xo * cs
    return out


# ----------------------------------------------------------------------------
# logical (unpaged) inputs
# ----------------------------------------------------------------------------
@dataclass
class Inputs:
    B: int
    H: int
    n_q: int
    seq_lens: np.ndarray  # int32 [B] (includes the n_q new tokens)
    seq_off: np.ndarray   # int64 [B+1] row offsets into c / kr
    c: np.ndarray         # bf16 bits [sum L, 512]
    kr: np.ndarray        # bf16 bits [sum L, 64] (rotated)
    q_nope: np.ndarray    # bf16 bits [B, n_q, H, 128]
    q_rope: np.ndarray    # bf16 bits [B, n_q, H, 64] (rotated)
    w_uk: np.ndarray      # bf16 bits [H, 128, 512]
    w_uv: np.ndarray      # bf16 bits [H, 128, 512]
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.B * self.n_q

    @property
    def total_tokens(self) -> int:
        return int(self.seq_off[-1])


def make_inputs(B: int, H: int, n_q: int, seq_lens, seed: int, *,
                w_std: float = 1.0 / math.sqrt(512.0)) -> Inputs:
    """Draw one batch following the recipe in the module docstring."""
    rng = np.random.default_rng(seed)
    if callable(seq_lens):
        lens = np.asarray(seq_lens(rng), dtype=np.int64)
    else:
        lens = np.asarray(seq_lens, dtype=np.int64)
        if lens.ndim == 0:
            lens = np.full(B, int(lens), dtype=np.int64)
    assert lens.shape == (B,), lens.shape
    assert (lens >= n_q).all(), "every context must hold its n_q new tokens"
    off = np.zeros(B + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens)
    total = int(off[-1])
    c = np.empty((total, D_C), dtype=np.uint16)
    kr = np.empty((total, D_R), dtype=np.uint16)
    for b in range(B):
        L = int(lens[b])
        cb = rng.standard_normal((L, D_C), dtype=np.float32)
        kb = rng.standard_normal((L, D_R), dtype=np.float32)
        c[off[b]:off[b + 1]] = f32_to_bf16(cb)
        kb = rope_rotate(kb, np.arange(L))
        kr[off[b]:off[b + 1]] = f32_to_bf16(kb.astype(np.float32))
    q_nope = rng.standard_normal((B, n_q, H, D_NOPE), dtype=np.float32)
    q_raw = rng.standard_normal((B, n_q, H, D_R), dtype=np.float32)
    w_uk = rng.standard_normal((H, D_NOPE, D_C), dtype=np.float32) * np.float32(w_std)
    w_uv = rng.standard_normal((H, D_V, D_C), dtype=np.float32) * np.float32(w_std)
    qpos = (lens[:, None] - n_q + np.arange(n_q)[None, :]).astype(np.float64)  # [B, n_q]
    q_rope = rope_rotate(q_raw, qpos[:, :, None])
    return Inputs(
        B=B, H=H, n_q=n_q, seq_lens=lens.astype(np.int32), seq_off=off,
        c=c, kr=kr, q_nope=f32_to_bf16(q_nope), q_rope=f32_to_bf16(q_rope.astype(np.float32)),
        w_uk=f32_to_bf16(w_uk), w_uv=f32_to_bf16(w_uv),
        meta={"seed": seed},
    )


def with_rising_scores(inp: Inputs, *, gamma: float = 8.0, top: float = 64.0, col: int = 0,
                       kind: str = "ramp") -> Inputs:
    """A copy of ``inp`` whose later tokens score higher for every head, by a shift that
    bf16 holds exactly: column ``col`` of every (rotated) positional query is set to
    ``gamma`` and column ``col`` of token s's positional key to beta(s / L), with
    beta(x) = top * x ("ramp") or top * [x >= 1/2] ("step"), rounded to bf16. Every
    head's score of token s then grows by gamma * beta(s / L) / sqrt(192) (37 in
    natural-log units for the defaults), so the running softmax maximum keeps rising
    along a sequence. The rest of the inputs are those of ``inp``."""
    import dataclasses
    qr = bf16_to_f32(inp.q_rope).copy()
    qr[..., col] = gamma
    kr = bf16_to_f32(inp.kr).copy()
    for b in range(inp.B):
        L = int(inp.seq_lens[b])
        o = int(inp.seq_off[b])
        x = np.arange(L, dtype=np.float64) / L
        beta = top * x if kind == "ramp" else top * (x >= 0.5)
        kr[o:o + L, col] = beta.astype(np.float32)
    return dataclasses.replace(inp, q_rope=f32_to_bf16(qr), kr=f32_to_bf16(kr),
                               meta=dict(inp.meta, rising=(gamma, top, col, kind)))


def workload_inputs(index: int) -> Inputs:
    w = WORKLOADS[index]
    if w.context is None:
        lens = lambda rng: rng.integers(512, 16385, size=w.B)  # noqa: E731
    else:
        lens = w.context
    inp = make_inputs(w.B, w.H, w.n_q, lens, w.seed)
    inp.meta.update(workload=index, name=w.name)
    return inp


# ----------------------------------------------------------------------------
# paging
# ----------------------------------------------------------------------------
@dataclass
class Paged:
    cache: np.ndarray        # bf16 bits [num_pages, PAGE, 576]
    block_table: np.ndarray  # int32 [B, max_pages]
    num_pages: int
    max_pages: int
    page_size: int = PAGE


def pages_for(lens: np.ndarray, page: int = PAGE) -> np.ndarray:
    return (np.asarray(lens, dtype=np.int64) + page - 1) // page


def make_paged(inp: Inputs, *, perm_seed: int = 12345, spare_pages: int = 4,
               max_pages: int | None = None, page: int = PAGE,
               poison: bool = True) -> Paged:
    """Scatter the logical rows [c || kr] into a randomly permuted page pool."""
    npg = pages_for(inp.seq_lens, page)
    used = int(npg.sum())
    num_pages = used + spare_pages
    if max_pages is None:
        max_pages = int(npg.max())
    assert max_pages >= int(npg.max())
    perm = np.random.default_rng(perm_seed).permutation(num_pages).astype(np.int32)
    cache = np.empty((num_pages, page, D_ROW), dtype=np.uint16)
    cache[...] = BF16_NAN if poison else np.uint16(0)
    bt = np.full((inp.B, max_pages), -1, dtype=np.int32)
    nxt = 0
    for b in range(inp.B):
        L = int(inp.seq_lens[b])
        base = int(inp.seq_off[b])
        for p in range(int(npg[b])):
            phys = int(perm[nxt])
            nxt += 1
            bt[b, p] = phys
            t0 = p * page
            t1 = min(L, t0 + page)
            cache[phys, : t1 - t0, :D_C] = inp.c[base + t0: base + t1]
            cache[phys, : t1 - t0, D_C:] = inp.kr[base + t0: base + t1]
    return Paged(cache=cache, block_table=bt, num_pages=num_pages, max_pages=max_pages, page_size=page)


# ----------------------------------------------------------------------------
# FP8 (e4m3) latent cache with per-channel scales
# ----------------------------------------------------------------------------
E4M3_MAX = 448.0  # largest finite e4m3 value: 2^8 * 1.75


def fp8_channel_scales(inp: Inputs) -> np.ndarray:
    """Per-channel scales of the FP8 cache, one per column of the 576-wide row (the
    fine-grained per-channel scaling the Huny's Dev Blog page asks for in section 6,
    item 4): s[d] = max over every cached token |row[d]| / 448, float32 (1 where the
    column is all zero), so each column's largest value maps to the largest e4m3."""
    amax = np.concatenate([np.abs(bf16_to_f32(inp.c)).max(axis=0), np.abs(bf16_to_f32(inp.kr)).max(axis=0)])
    s = (amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    s[s == 0] = np.float32(1.0)
    return s


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round float32 values to e4m3 codes (uint8): nearest, ties to even, magnitudes
    beyond 448 saturated to 448, NaN -> 0x7F. e4m3: sign, 4 exponent bits (bias 7),
    3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; 0x7F / 0xFF are
    NaN and there is no infinity. Rounding is done in float64, where dividing by the
    quantum (a power of two) is exact."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, e2 = np.frexp(a)                       # a = f * 2^e2, f in [0.5, 1)
    e = np.clip(e2 - 1, -6, 8)                # binade exponent (subnormals share -6)
    quantum = np.ldexp(1.0, e - 3)            # 3 mantissa bits
    v = np.round(a / quantum) * quantum       # numpy rounds halves to even
    v = np.minimum(v, E4M3_MAX)
    # encode the rounded magnitude
    _, ev = np.frexp(v)
    eb = np.clip(ev - 1, -6, 8)
    normal = v >= 2.0 ** -6
    mant = np.where(normal, v / np.ldexp(1.0, eb) - 1.0, v / 2.0 ** -9)
    mant = np.nan_to_num(mant)  # NaN inputs get their code below
    mbits = np.where(normal, np.round(mant * 8.0), np.round(mant)).astype(np.int64)
    ebits = np.where(normal, eb + 7, 0).astype(np.int64)
    code = (ebits << 3) | mbits
    code = code | (sign.astype(np.int64) << 7)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_fp8(rows_bf16: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """e4m3 codes of bf16 rows [..., 576] with per-column scales: the float32 quotient
    row / s (one correctly rounded division), then f32_to_e4m3."""
    x = bf16_to_f32(rows_bf16).astype(np.float32) / np.asarray(scales, dtype=np.float32)
    return f32_to_e4m3(x.astype(np.float32))


E4M3_NAN = np.uint8(0x7F)


@dataclass
class PagedFP8:
    cache: np.ndarray        # e4m3 codes [num_pages, PAGE, 576] (uint8)
    scales: np.ndarray       # float32 [576]
    block_table: np.ndarray  # int32 [B, max_pages]
    num_pages: int
    max_pages: int
    page_size: int = PAGE


def make_paged_fp8(inp: Inputs, pg: Paged, scales: np.ndarray | None = None) -> PagedFP8:
    """The FP8 cache holding the same tokens in the same pages as ``pg``: every row
    quantised with per-channel scales (fp8_channel_scales unless given); slack rows
    and spare pages hold the e4m3 NaN code."""
    s = fp8_channel_scales(inp) if scales is None else np.asarray(scales, dtype=np.float32)
    rows = pg.cache.reshape(-1, D_ROW)
    codes = quantize_fp8(rows, s)
    codes[(rows[:, 0] == BF16_NAN)] = E4M3_NAN  # poisoned rows stay poisoned
    return PagedFP8(cache=codes.reshape(pg.cache.shape), scales=s, block_table=pg.block_table,
                    num_pages=pg.num_pages, max_pages=pg.max_pages, page_size=pg.page_size)


def latent_query_inputs(T: int, H: int, d_q: int, seed: int, d_nope: int = D_NOPE):
    """Compressed query latents and the query up-projection for the query-side
    absorption (seeded, numpy PCG64 ``default_rng(seed)``), in draw order:
    c_q ~ N(0,1) [T, d_q], then w_uq ~ N(0,1) * (1/sqrt(d_q)) [d_q, H, d_nope]
    (input-major: w_uq[k][h][i] maps compressed column k to head h's no-RoPE
    query column i), float32 draws rounded to bf16. Returns (c_q, w_uq) bits."""
    rng = np.random.default_rng(seed)
    c_q = f32_to_bf16(rng.standard_normal((T, d_q), dtype=np.float32))
    w_uq = f32_to_bf16((rng.standard_normal((d_q, H, d_nope), dtype=np.float32)
                        * np.float32(1.0 / math.sqrt(d_q))).astype(np.float32))
    return c_q, w_uq


def output_projection(d_model: int, H: int, seed: int, d_v: int = D_V):
    """The attention output projection W^O, one row per output column, w_o[n][h][v]
    ~ N(0,1) * (1/sqrt(H * d_v)) [d_model, H, d_v] (float32 draws rounded to bf16,
    numpy PCG64 ``default_rng(seed)``). Returns bf16 bits."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((d_model, H, d_v), dtype=np.float32) * np.float32(1.0 / math.sqrt(H * d_v))
    return f32_to_bf16(w.astype(np.float32))


def workload_bytes(inp: Inputs) -> dict:
    """Algorithmic byte and flop counts of one decode step (cache read once)."""
    T, H = inp.T, inp.H
    att = 0
    for b in range(inp.B):
        for j in range(inp.n_q):
            att += int(inp.seq_lens[b]) - inp.n_q + j + 1
    cache_bytes = int(inp.seq_lens.sum()) * D_ROW * 2
    decode_bytes = (cache_bytes + T * H * D_ROW * 2 + T * H * D_C * 2 + T * H * 4
                    + inp.B * 4 + int(pages_for(inp.seq_lens).sum()) * 4)
    decode_flops = att * H * (2 * D_ROW + 2 * D_C)
    absorb_bytes = H * D_NOPE * D_C * 2 + T * H * (D_NOPE + D_R + D_ROW) * 2
    absorb_flops = 2 * T * H * D_NOPE * D_C
    outproj_bytes = H * D_V * D_C * 2 + T * H * (D_C + D_V) * 2
    outproj_flops = 2 * T * H * D_C * D_V
    return dict(cache_bytes=cache_bytes, decode_bytes=decode_bytes, decode_flops=decode_flops,
                absorb_bytes=absorb_bytes, absorb_flops=absorb_flops,
                outproj_bytes=outproj_bytes, outproj_flops=outproj_flops,
                attended=att)
