"""The seeded input generator: rounding, rotary rotation and paging (no GPU)."""
import numpy as np
import pytest
import torch

import mla_inputs as mi


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000, dtype=np.float32) * 10.0,
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-30, np.inf, -np.inf], np.float32)])
    ours = mi.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert mi.f32_to_bf16(np.array([np.nan], np.float32))[0] == 0x7FC0
    back = mi.bf16_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_rope_preserves_norm_and_depends_on_relative_position():
    """Huny's Dev Blog "MLA 아키텍처 해부", section 2.2: R_t is an orthogonal
    rotation and (R_t q).(R_s k) depends only on t - s."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    for t, s in [(5, 3), (1000, 7), (131071, 131000), (42, 42)]:
        rq, rk = mi.rope_rotate(q, t), mi.rope_rotate(k, s)
        assert abs(np.linalg.norm(rq) - np.linalg.norm(q)) <= 1e-12
        lhs = rq @ rk
        rhs = mi.rope_rotate(q, t - s) @ k
        assert abs(lhs - rhs) <= 1e-9
    # position 0 is the identity; pair (0, 1) at position 1 turns by exactly 1 radian
    assert np.array_equal(mi.rope_rotate(q, 0), q)
    e = np.zeros(64); e[0] = 1.0
    r = mi.rope_rotate(e, 1)
    assert abs(r[0] - np.cos(1.0)) <= 1e-15 and abs(r[1] - np.sin(1.0)) <= 1e-15


def test_generator_is_deterministic_and_shaped():
    a = mi.workload_inputs(1)
    b = mi.workload_inputs(1)
    for name in ["c", "kr", "q_nope", "q_rope", "w_uk", "w_uv", "seq_lens"]:
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    assert a.c.shape == (512, 512) and a.kr.shape == (512, 64)
    assert a.q_nope.shape == (2, 1, 16, 128) and a.w_uk.shape == (16, 128, 512)
    w = mi.bf16_to_f32(a.w_uk).astype(np.float64)
    assert abs(w.std() - 1.0 / np.sqrt(512.0)) < 2e-3


def test_paging_round_trip_and_poison():
    inp = mi.make_inputs(B=3, H=2, n_q=1, seq_lens=[1, 64, 130], seed=9)
    pg = mi.make_paged(inp, perm_seed=3, spare_pages=5)
    assert pg.num_pages == 1 + 1 + 3 + 5
    assert pg.cache.nbytes == pg.num_pages * 64 * 576 * 2
    used = set()
    for b in range(3):
        L = int(inp.seq_lens[b])
        rows = []
        for s in range(L):
            phys = pg.block_table[b, s // 64]
            rows.append(pg.cache[phys, s % 64])
            used.add(int(phys))
        rows = np.stack(rows)
        assert np.array_equal(rows[:, :512], inp.c[inp.seq_off[b]:inp.seq_off[b + 1]])
        assert np.array_equal(rows[:, 512:], inp.kr[inp.seq_off[b]:inp.seq_off[b + 1]])
        last = pg.block_table[b, (L - 1) // 64]
        assert (pg.cache[last, (L - 1) % 64 + 1:] == 0x7FC0).all()
        npg = (L + 63) // 64
        assert (pg.block_table[b, npg:] == -1).all()
    spare = set(range(pg.num_pages)) - used
    assert len(spare) == 5
    for p in spare:
        assert (pg.cache[p] == 0x7FC0).all()


def test_two_permutations_hold_the_same_logical_rows():
    inp = mi.make_inputs(B=2, H=2, n_q=1, seq_lens=[100, 200], seed=4)
    p1 = mi.make_paged(inp, perm_seed=1)
    p2 = mi.make_paged(inp, perm_seed=2)
    assert not np.array_equal(p1.block_table, p2.block_table)
    for b in range(2):
        for pg in range((int(inp.seq_lens[b]) + 63) // 64):
            assert np.array_equal(p1.cache[p1.block_table[b, pg]], p2.cache[p2.block_table[b, pg]])


@pytest.mark.parametrize("index,pages,cache_bytes", [(1, 8, 589_824), (2, 2048, 150_994_944)])
def test_workload_sizes(index, pages, cache_bytes):
    w = mi.WORKLOADS[index]
    lens = np.full(w.B, w.context)
    assert int(mi.pages_for(lens).sum()) == pages
    assert int(lens.sum()) * 576 * 2 == cache_bytes


def test_ragged_lengths_follow_the_recipe():
    rng = np.random.default_rng(2)  # workload 3 uses seed 2
    lens = rng.integers(512, 16385, size=128)
    assert lens.min() >= 512 and lens.max() <= 16384
