"""Shared helpers for the tests: device transfer of generator outputs and error metrics."""
import numpy as np

import mla_inputs as mi

# Tolerances for floating-point parity (bf16 inputs, fp32 accumulation), applied
# to out, u and lse: max |gpu - oracle| and sum|gpu - oracle| / sum|oracle|.
MAX_ABS = 2e-2
MEAN_REL = 5e-3


def to_dev_bf16(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.cuda().view(torch.bfloat16)


def to_dev_i32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_to_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_bf16_to_f64(t) -> np.ndarray:
    return mi.bf16_to_f32(dev_to_bits(t)).astype(np.float64)


def errors(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(gpu - ref)
    return float(d.max()), float(d.sum() / max(np.abs(ref).sum(), 1e-300))


def assert_close(gpu, ref, what: str, max_abs=MAX_ABS, mean_rel=MEAN_REL):
    assert np.isfinite(gpu).all(), f"{what}: non-finite values"
    ma, mr = errors(gpu, ref)
    assert ma <= max_abs and mr <= mean_rel, f"{what}: max_abs {ma:.3e} mean_rel {mr:.3e}"
    return ma, mr


def device_inputs(inp, pg):
    """Move one batch to the device: returns dict of torch tensors."""
    T = inp.B * inp.n_q
    return dict(
        q_nope=to_dev_bf16(inp.q_nope.reshape(T, inp.H, -1)),
        q_rope=to_dev_bf16(inp.q_rope.reshape(T, inp.H, -1)),
        w_uk=to_dev_bf16(inp.w_uk),
        w_uv=to_dev_bf16(inp.w_uv),
        cache=to_dev_bf16(pg.cache),
        block_table=to_dev_i32(pg.block_table),
        seq_lens=to_dev_i32(inp.seq_lens),
    )


def plan_mirror(seq_lens, n_q, max_pages, G, page=64, switch_pages=3, tile=64):
    """Python statement of the split plan documented in include/mla.h (integer work):
    contexts clipped to the block table's max_pages * page tokens, cut into tiles of
    64 tokens; the tiles of all sequences in order, each sequence start after the
    first costing `switch_pages` extra tiles (dropped when a step is not longer than
    that); cut p at floor(p * V / G') on that line, G' = min(G, P). The items'
    bounds are tile indices."""
    lens = np.clip(np.asarray(seq_lens, dtype=np.int64), n_q, max_pages * page)
    pages = (lens + tile - 1) // tile
    starts = np.concatenate([[0], np.cumsum(pages)])
    P = int(starts[-1])
    B = len(lens)
    Ge = min(G, P)
    a = switch_pages if (P + switch_pages * (B - 1)) // Ge >= switch_pages + 1 else 0
    V = P + a * (B - 1)

    def to_page(x):  # a point of the cost line -> global page where the cut lands
        line0 = [0] + [int(starts[b]) + a * (b - 1) for b in range(1, B)]
        b = max(i for i in range(B) if line0[i] <= x)
        return int(starts[b]) + max(0, x - (int(starts[b]) + a * b))

    cut_at = [to_page((p * V) // Ge) for p in range(Ge + 1)]
    assert all(x < y for x, y in zip(cut_at[:-1], cut_at[1:])), "an empty range"
    cuts = sorted(set(cut_at))
    items = []  # (seq, page0, page1)
    seq_item = []
    for b in range(B):
        seq_item.append(len(items))
        lo, hi = int(starts[b]), int(starts[b + 1])
        bounds = [lo] + [x for x in cuts if lo < x < hi] + [hi]
        for x0, x1 in zip(bounds[:-1], bounds[1:]):
            items.append((b, x0 - lo, x1 - lo))
    seq_item.append(len(items))
    range_item = []
    glob_start = [int(starts[b]) + p0 for (b, p0, _) in items]
    for p in range(G + 1):
        if p >= Ge:
            range_item.append(len(items))
        else:
            range_item.append(glob_start.index(cut_at[p]))
    return dict(items=np.array(items, dtype=np.int64), seq_item=np.array(seq_item),
                range_item=np.array(range_item), total=P, Ge=Ge, lens=lens, switch=a)


def abi_step(L, d, inp, pg, num_splits=None, err=None, scale=None):
    """One decode step through the C ABI of the ctypes library ``L`` (the release or the
    test build): mla_absorb_q -> mla_decode_paged -> mla_combine -> mla_out_proj on the
    device tensors ``d`` (from device_inputs). Returns dict(q_abs, u, lse, out, workspace)."""
    import ctypes
    import math

    import torch
    T, H = inp.B * inp.n_q, inp.H
    dev = d["cache"].device
    G = int(L.mla_decode_default_splits(inp.n_q)) if num_splits is None else num_splits
    scale = 1.0 / math.sqrt(192.0) if scale is None else scale
    q_abs = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(int(L.mla_decode_workspace_bytes(inp.B, inp.n_q, H, G)), dtype=torch.uint8, device=dev)
    u = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.mla_absorb_q(p(d["q_nope"]), p(d["q_rope"]), p(d["w_uk"]), p(q_abs), T, H, 128, 64, 512, s)
    assert st == 0, ("mla_absorb_q", st)
    st = L.mla_decode_paged(p(q_abs), p(d["cache"]), p(d["block_table"]), p(d["seq_lens"]), inp.B, inp.n_q, H,
                            pg.num_pages, 64, pg.max_pages, ctypes.c_float(scale), G, p(ws), ws.numel(), p(err), s)
    assert st == 0, ("mla_decode_paged", st)
    st = L.mla_combine(p(ws), inp.B, inp.n_q, H, G, p(u), p(lse), s)
    assert st == 0, ("mla_combine", st)
    st = L.mla_out_proj(p(u), p(d["w_uv"]), p(out), T, H, 512, 128, s)
    assert st == 0, ("mla_out_proj", st)
    return dict(q_abs=q_abs, u=u, lse=lse, out=out, workspace=ws)
