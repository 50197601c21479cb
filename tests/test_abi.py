"""The C-ABI library: it loads without a GPU, exports every declared symbol,
rejects bad arguments on the host before any launch, and its closed-form
size functions give the numbers printed on the pages. No compute call runs."""
import os
import re

import numpy as np
import pytest

import mla_latent_kv_paged_gb300 as mla
from tests.helpers import plan_mirror

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mla.build()
    return mla.lib()


DEBUG_HEADER = "mla_debug.h"  # the test build's extra entry points


def declared_functions(headers=None):
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h") and (headers is None or h in headers):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    release = [h for h in os.listdir(os.path.join(ROOT, "include")) if h.endswith(".h") and h != DEBUG_HEADER]
    decl = declared_functions(release)
    assert "mla_decode_paged" in decl and "mla_combine" in decl
    for name in decl:
        assert hasattr(lib, name), name
    assert set(mla.EXPORTS) <= set(decl)
    assert lib.mla_abi_version() == 3
    # the release library carries none of the test build's instrumentation
    for name in declared_functions([DEBUG_HEADER]):
        assert not hasattr(lib, name), name


def test_test_build_exports_everything():
    """libmla_gb300_debug.so: every declared entry point, the test-only ones included."""
    dbg = mla.debug_lib()
    decl = declared_functions()
    assert set(mla.DEBUG_EXPORTS) == set(declared_functions([DEBUG_HEADER]))
    for name in decl:
        assert hasattr(dbg, name), name
    assert dbg.mla_abi_version() == 3


def test_status_strings(lib):
    for code, name in mla.STATUS.items():
        assert lib.mla_status_string(code).decode() == name
    assert lib.mla_status_string(99).decode() == "MLA_ERR_UNKNOWN"


def golden():
    rows = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "cache_sizes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, val, unit, src = [x.strip() for x in line.split("|")]
        rows[key] = float(val)
    return rows


def test_cache_size_numbers_from_the_pages(lib):
    g = golden()
    mla_b = lib.mla_cache_bytes_per_token(512, 64)
    assert mla_b == g["mla_bytes_per_token_layer"] == 1152
    assert mla_b // 2 == g["mla_values_per_token"]
    mha_b = 2 * 128 * 128 * 2  # MHA cache formula 2 n_h d_h b at the V3 shape
    assert mha_b == g["mha_bytes_per_token_layer"]
    assert mha_b // 2 == g["mha_values_per_token"]
    assert round(100 * (1 - mla_b / mha_b), 2) == g["mla_vs_mha_saving_pct"]
    assert round(100 * (1 - mla_b / g["gqa8_bytes_per_token_layer"]), 2) == g["mla_vs_gqa8_saving_pct"]
    assert round(100 * (mla_b / 2) / g["mha_values_per_token"], 2) == g["mla_fraction_pct"]
    assert (mla_b / 2) / (2 * 128) == g["mla_equivalent_gqa_groups"]
    assert 2 * 8 * 128 == g["gqa8_values_per_token"]
    MiB = 1 << 20
    assert mla_b * 8192 / MiB == g["mla_8k_per_layer"]
    assert mha_b * 8192 / MiB == g["mha_8k_per_layer"]
    assert g["gqa8_bytes_per_token_layer"] * 8192 / MiB == g["gqa8_8k_per_layer"]
    assert g["mqa_bytes_per_token_layer"] * 8192 / MiB == g["mqa_8k_per_layer"]
    assert 512 / (128 * 128) == g["latent_fraction_of_kv_dims"]
    assert 2 * 40 * 128 == g["mha_dims_40_heads"]
    assert lib.mla_page_bytes(16, 512, 64) * 80 == g["mla_block_bytes_v2_80_layers_block16"]
    assert lib.mla_page_bytes(64, 512, 64) == 73728


def test_workspace_size_query(lib):
    n = lib.mla_decode_workspace_bytes(32, 1, 128, 76)
    assert n >= (76 + 32) * 128 * 512 * 2  # fp16 partials
    assert lib.mla_decode_workspace_bytes(0, 1, 128, 76) == 0
    assert lib.mla_decode_workspace_bytes(32, 3, 128, 76) == 0
    assert lib.mla_decode_workspace_bytes(32, 1, 129, 76) == 0
    assert lib.mla_decode_workspace_bytes(32, 1, 128, 0) == 0


FAKE = 1 << 20  # a 16-byte aligned, never dereferenced address


def test_host_validation_absorb_and_out_proj(lib):
    p = FAKE
    assert lib.mla_absorb_q(None, p, p, p, 4, 128, 128, 64, 512, None) == 1
    assert lib.mla_absorb_q(p, p, p, p + 2, 4, 128, 128, 64, 512, None) == 1
    assert lib.mla_absorb_q(p, p, p, p, 0, 128, 128, 64, 512, None) == 1
    assert lib.mla_absorb_q(p, p, p, p, 4, 128, 64, 64, 512, None) == 2
    assert lib.mla_absorb_q(p, p, p, p, 4, 256, 128, 64, 512, None) == 2
    assert lib.mla_out_proj(p, None, p, 4, 128, 512, 128, None) == 1
    assert lib.mla_out_proj(p, p, p, 4, 128, 256, 128, None) == 2
    assert lib.mla_out_proj(p, p, p, 4, 128, 512, 64, None) == 2


def test_host_validation_decode_and_combine(lib):
    p = FAKE
    ws = lib.mla_decode_workspace_bytes(2, 1, 16, 4)

    def dec(**kw):
        a = dict(q=p, cache=p, bt=p, sl=p, B=2, n_q=1, H=16, num_pages=8, page=64, maxp=4,
                 scale=0.07, G=4, ws=p, wsb=ws, err=None)
        a.update(kw)
        return lib.mla_decode_paged(a["q"], a["cache"], a["bt"], a["sl"], a["B"], a["n_q"], a["H"],
                                    a["num_pages"], a["page"], a["maxp"], a["scale"], a["G"],
                                    a["ws"], a["wsb"], a["err"], None)

    assert dec(q=None) == 1
    assert dec(cache=p + 8) == 1
    assert dec(B=0) == 1
    assert dec(G=0) == 1
    assert dec(scale=0.0) == 1
    assert dec(scale=float("nan")) == 1
    assert dec(num_pages=0) == 1
    assert dec(n_q=3) == 2
    assert dec(H=200) == 2
    assert dec(page=16) == 2
    assert dec(B=5000) == 2
    assert dec(wsb=ws - 1) == 3
    assert lib.mla_combine(None, 2, 1, 16, 4, p, p, None) == 1
    assert lib.mla_combine(p, 2, 3, 16, 4, p, p, None) == 2
    assert lib.mla_combine(p, 2, 1, 16, 4, p + 4, p, None) == 1


def test_host_validation_plan_and_planned_decode(lib):
    p = FAKE
    ws = lib.mla_decode_workspace_bytes(2, 1, 16, 4)

    def plan(**kw):
        a = dict(sl=p, B=2, n_q=1, H=16, num_pages=8, page=64, maxp=4, G=4, ws=p, wsb=ws, err=None)
        a.update(kw)
        return lib.mla_decode_plan(a["sl"], a["B"], a["n_q"], a["H"], a["num_pages"], a["page"], a["maxp"], a["G"],
                                   a["ws"], a["wsb"], a["err"], None)

    def dec(**kw):
        a = dict(q=p, cache=p, bt=p, B=2, n_q=1, H=16, num_pages=8, page=64, maxp=4, scale=0.07, G=4, ws=p,
                 wsb=ws, err=None)
        a.update(kw)
        return lib.mla_decode_paged_planned(a["q"], a["cache"], a["bt"], a["B"], a["n_q"], a["H"], a["num_pages"],
                                            a["page"], a["maxp"], a["scale"], a["G"], a["ws"], a["wsb"], a["err"],
                                            None)

    assert plan(sl=None) == 1 and plan(sl=p + 4) == 1 and plan(ws=None) == 1 and plan(B=0) == 1
    assert plan(G=0) == 1 and plan(n_q=3) == 2 and plan(H=129) == 2
    # pages of 64 or 128 tokens; positions up to max_pages * page_size must stay below 2^30
    assert plan(page=256) == 2 and plan(page=96) == 2 and plan(page=0) == 2
    assert plan(page=128, maxp=(1 << 23) + 1) == 2 and plan(page=64, maxp=(1 << 24) + 1) == 2
    assert plan(wsb=ws - 1) == 3
    assert dec(q=None) == 1 and dec(bt=p + 4) == 1 and dec(scale=0.0) == 1 and dec(ws=p + 8) == 1
    assert dec(n_q=0) == 2
    assert dec(page=32) == 2 and dec(wsb=ws - 1) == 3


def test_host_validation_append(lib):
    p = FAKE
    ws = lib.mla_append_workspace_bytes(2, 512)
    assert ws > 0
    assert lib.mla_append_workspace_bytes(0, 512) == 0
    assert lib.mla_append_workspace_bytes(2, 100) == 0
    assert lib.mla_append_workspace_bytes(2, 0) == 0

    def app(**kw):
        a = dict(h=p, w=p, cache=p, bt=p, sl=p, B=2, n_q=1, d=512, num_pages=8, page=64, maxp=4, theta=1e4,
                 ws=p, wsb=ws, err=None)
        a.update(kw)
        return lib.mla_append_kv(a["h"], a["w"], a["cache"], a["bt"], a["sl"], a["B"], a["n_q"], a["d"],
                                 a["num_pages"], a["page"], a["maxp"], a["theta"], a["ws"], a["wsb"], a["err"], None)

    assert app(h=None) == 1
    assert app(cache=p + 2) == 1
    assert app(B=0) == 1
    assert app(theta=0.5) == 1
    assert app(theta=float("nan")) == 1
    assert app(n_q=3) == 2
    assert app(d=96) == 2
    assert app(page=256) == 2 and app(page=32) == 2
    assert app(page=128, maxp=(1 << 23) + 1) == 2
    assert app(wsb=ws - 1) == 3


def test_host_validation_query_side_absorption(lib):
    p = FAKE

    def merge(**kw):
        a = dict(wq=p, wk=p, out=p, d_q=1536, H=128, dn=128, dc=512)
        a.update(kw)
        return lib.mla_merge_w_kq(a["wq"], a["wk"], a["out"], a["d_q"], a["H"], a["dn"], a["dc"], None)

    def latent(**kw):
        a = dict(cq=p, qr=p, w=p, out=p, T=32, H=128, d_q=1536, dr=64, dc=512)
        a.update(kw)
        return lib.mla_absorb_q_latent(a["cq"], a["qr"], a["w"], a["out"], a["T"], a["H"], a["d_q"], a["dr"],
                                       a["dc"], None)

    assert merge(wq=None) == 1 and merge(out=p + 8) == 1 and merge(d_q=0) == 1
    assert merge(d_q=100) == 2 and merge(d_q=16384 + 64) == 2 and merge(H=129) == 2
    assert merge(dn=64) == 2 and merge(dc=256) == 2
    assert latent(qr=None) == 1 and latent(cq=p + 2) == 1 and latent(T=0) == 1
    assert latent(d_q=96) == 2 and latent(dr=32) == 2 and latent(dc=576) == 2 and latent(H=0) == 2


def test_host_validation_merged_output_projection(lib):
    p = FAKE
    ws = lib.mla_out_comb_workspace_bytes(32, 128, 7168)
    assert ws == 32 * 7168 * 4 * (304 // 56)  # one row tile, five splits of fp32 partials
    assert lib.mla_out_comb_workspace_bytes(0, 128, 7168) == 0
    assert lib.mla_out_comb_workspace_bytes(32, 128, 7100) == 0
    assert lib.mla_out_comb_workspace_bytes(32, 129, 7168) == 0

    def merge(**kw):
        a = dict(wv=p, wo=p, out=p, H=128, dv=128, dc=512, d=7168)
        a.update(kw)
        return lib.mla_merge_w_comb(a["wv"], a["wo"], a["out"], a["H"], a["dv"], a["dc"], a["d"], None)

    def comb(**kw):
        a = dict(u=p, w=p, out=p, T=32, H=128, dc=512, d=7168, ws=p, wsb=ws)
        a.update(kw)
        return lib.mla_out_comb(a["u"], a["w"], a["out"], a["T"], a["H"], a["dc"], a["d"], a["ws"], a["wsb"], None)

    assert merge(wo=None) == 1 and merge(out=p + 4) == 1 and merge(d=0) == 1
    assert merge(d=7100) == 2 and merge(dv=64) == 2 and merge(dc=576) == 2 and merge(H=0) == 2
    assert comb(ws=None) == 1 and comb(u=p + 2) == 1 and comb(T=0) == 1
    assert comb(T=2 * 4096 + 1) == 2 and comb(d=64) == 2 and comb(dc=256) == 2
    assert comb(wsb=ws - 1) == 3


@pytest.mark.parametrize("lens,G", [([256, 256], 76), ([4096] * 32, 76), ([64] * 3, 2),
                                    ([1, 65, 130, 64, 5000], 7), ([100], 1), ([7, 9], 5),
                                    ([4096] * 32, 38), ([64] * 500, 76), ([1] * 4096, 76),
                                    ([640, 64, 64, 64, 640], 4), ([64 * 9] * 3, 6)])
def test_plan_statement_covers_every_page_once(lens, G):
    """The documented split plan: each range holds consecutive pages whose cost
    (pages plus the switch cost for every further sequence it moves on to) is
    near-equal; each sequence's pieces tile its pages in order."""
    pl = plan_mirror(lens, 1, 200, G)
    P, Ge = pl["total"], pl["Ge"]
    pages = (np.asarray(lens) + 63) // 64
    assert P == pages.sum() and Ge == min(G, P)
    for b in range(len(lens)):
        its = pl["items"][pl["seq_item"][b]:pl["seq_item"][b + 1]]
        assert (its[:, 0] == b).all()
        assert its[0, 1] == 0 and its[-1, 2] == pages[b]
        assert (its[1:, 1] == its[:-1, 2]).all() and (its[:, 2] > its[:, 1]).all()
    sizes, costs = [], []
    a = pl["switch"]
    for p in range(G):
        its = pl["items"][pl["range_item"][p]:pl["range_item"][p + 1]]
        assert (len(its) > 0) == (p < Ge)
        sizes.append(int((its[:, 2] - its[:, 1]).sum()) if len(its) else 0)
        if len(its):
            costs.append(sizes[-1] + a * (len(its) - 1))
    assert sum(sizes) == P
    # a step of the cost line is floor or ceil of V / G'; a range that starts on a
    # sequence start may have been handed up to `a` points of the switch before it
    assert max(costs) - min(costs) <= 1 + a
    assert len(pl["items"]) <= G + len(lens) - 1


def test_plan_switch_cost_moves_pages_off_ranges_that_switch():
    """32 sequences of 64 pages over 76 ranges: the ranges that hold a sequence
    start inside them get about `switch` fewer pages than those that do not."""
    pl = plan_mirror([4096] * 32, 1, 64, 76)
    assert pl["switch"] == 3
    one, two = [], []
    for p in range(76):
        its = pl["items"][pl["range_item"][p]:pl["range_item"][p + 1]]
        n = int((its[:, 2] - its[:, 1]).sum())
        (one if len(its) == 1 else two).append(n)
    assert 24 <= len(two) <= 28 and max(two) <= 26 and min(one) >= 25
    assert np.mean(one) - np.mean(two) >= 2
    flat = plan_mirror([4096] * 32, 1, 64, 76, switch_pages=0)
    assert flat["switch"] == 0 and len(flat["items"]) == 76 + 28


def test_plan_switch_cost_dropped_when_steps_are_short():
    """4096 one-page sequences over 76 ranges: a step of the line (~215 points)
    exceeds the cost, so it applies; 3 one-page sequences over 3 ranges do not."""
    assert plan_mirror([1] * 4096, 1, 4, 76)["switch"] == 3
    pl = plan_mirror([1] * 3, 1, 4, 3)
    assert pl["switch"] == 0 and len(pl["items"]) == 3


def test_host_validation_fp8(lib):
    p = FAKE
    assert lib.mla_quantize_fp8(None, p, p, 4, None) == 1
    assert lib.mla_quantize_fp8(p, p + 4, p, 4, None) == 1
    assert lib.mla_quantize_fp8(p, p, p, 0, None) == 1
    ws = lib.mla_decode_workspace_bytes(2, 1, 16, 4)

    def dec(**kw):
        a = dict(q=p, cache=p, s=p, bt=p, sl=p, B=2, n_q=1, H=16, num_pages=8, page=64, maxp=4,
                 scale=0.07, G=4, ws=p, wsb=ws, err=None)
        a.update(kw)
        return lib.mla_decode_paged_fp8(a["q"], a["cache"], a["s"], a["bt"], a["sl"], a["B"], a["n_q"], a["H"],
                                        a["num_pages"], a["page"], a["maxp"], a["scale"], a["G"], a["ws"], a["wsb"],
                                        a["err"], None)

    def planned(**kw):
        a = dict(q=p, cache=p, s=p, bt=p, B=2, n_q=1, H=16, num_pages=8, page=64, maxp=4, scale=0.07, G=4, ws=p,
                 wsb=ws, err=None)
        a.update(kw)
        return lib.mla_decode_paged_planned_fp8(a["q"], a["cache"], a["s"], a["bt"], a["B"], a["n_q"], a["H"],
                                                a["num_pages"], a["page"], a["maxp"], a["scale"], a["G"], a["ws"],
                                                a["wsb"], a["err"], None)

    for call in (dec, planned):
        assert call(s=None) == 1
        assert call(s=p + 4) == 1
        assert call(cache=p + 1) == 1
        assert call(scale=-1.0) == 1
        assert call(n_q=3) == 2
        assert call(page=256) == 2 and call(page=128, maxp=(1 << 23) + 1) == 2
        assert call(wsb=ws - 1) == 3
    assert dec(sl=None) == 1


def test_host_validation_copy16(lib):
    p = FAKE
    assert lib.mla_copy16(None, p, 16, None) == 1
    assert lib.mla_copy16(p, None, 16, None) == 1
    assert lib.mla_copy16(p, p + 16, 0, None) == 1
    assert lib.mla_copy16(p, p + 64, 24, None) == 1       # not a multiple of 16
    assert lib.mla_copy16(p + 8, p + 64, 16, None) == 1   # misaligned
    assert lib.mla_copy16(p, p + 64, 16, None) == 1       # an address the runtime does not know
