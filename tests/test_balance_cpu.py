"""Balanced static task orders, host view: no GPU needed.

The persistent CTAs take tasks round-robin (task t on CTA t mod G).

* Without the causal mask, P equal tasks end with a partial wave of
  r = P mod G tasks.  When 2r <= G the kernel runs each tile of those r tasks
  as one task whose two stages take the two halves of the key blocks ("Infra:
  Flash Attention", "Prefill and decode": key segments computed apart merge
  exactly).
* With the causal mask, m_blocks m and M-1-m of a unit have a constant total of
  key blocks; the paired order puts both on one CTA in consecutive waves
  ("Flash Attention 4 on Blackwell", "Scheduling": longest-processing-time
  balancing of causal tiles).

These tests check, through the library's host copy of the schedule, that the
tasks still cover every (tile, key block) once, where the balanced tasks land,
when each order applies, and the per-CTA work they give.
"""
import pytest

import exact_attention_forward_08_gb300 as fa


def plan_tasks(plan):
    return [fa.fa_plan_task(plan, t) for t in range(plan.num_tasks)]


def coverage(plan, tasks):
    """(b, g, tile position, key block) -> visits, from a task list."""
    seen = {}
    for t in tasks:
        if t.key_split:
            ranges = [(t.pos0[0], 0, t.n_blocks[0]), (t.pos0[0], t.key_split, t.n_blocks[1])]
        else:
            ranges = [(t.pos0[s], 0, t.n_blocks[s]) for s in range(2)]
        for pos0, first, n in ranges:
            for j in range(first, first + n):
                key = (t.b, t.g, pos0, j)
                seen[key] = seen.get(key, 0) + 1
    return seen


def expected_cells(plan):
    cells = set()
    for b in range(plan.batch):
        for g in range(plan.groups):
            for tile in range(plan.tiles):
                for j in range(plan.kv_blocks):
                    cells.add((b, g, tile * plan.pos_per_tile, j))
    return cells


CASES = [
    # (B, Hq, Hkv, Sq, Sk, grid)
    (4, 16, 16, 8192, 8192, 152),   # the MHA workload: 2048 tasks, 72 in the last wave
    (1, 2, 2, 1024, 1024, 152),     # fewer tasks than CTAs: every task splits
    (1, 4, 4, 1000, 1000, 7),       # ragged keys; CTAs 0-3 run two pairs, then a split task
    (1, 3, 3, 384, 640, 5),         # odd tiles (an empty split task) and odd key blocks (3 + 2)
    (1, 8, 2, 512, 512, 3),         # GQA rows packed 4 heads per tile
    (2, 5, 5, 700, 1500, 13),       # 30 tasks on 13 CTAs: 4 left over
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}/{c[2]}S{c[3]}x{c[4]}g{c[5]}" for c in CASES])
def test_split_tasks_cover_every_tile_and_block_once(case):
    B, Hq, Hkv, Sq, Sk, grid = case
    plan = fa.fa_make_plan(B, Hq, Hkv, Sq, Sk, 128, 128, 0)
    pairs = plan.num_tasks
    assert plan.tail_first == pairs
    fa.fa_plan_set_grid(plan, grid)
    r = pairs % grid if pairs >= grid else pairs
    assert plan.tail_first == pairs - r and plan.num_tasks == pairs + r, "split expected for these cases"
    tasks = plan_tasks(plan)
    seen = coverage(plan, tasks)
    assert set(seen) == expected_cells(plan)
    assert all(v == 1 for v in seen.values())
    for t, task in enumerate(tasks):
        if t < plan.tail_first:
            assert task.key_split == 0
            continue
        # a split task: one tile, halves of (nearly) equal length, stage 0 the longer
        pair = fa.fa_plan_task(fa.fa_make_plan(B, Hq, Hkv, Sq, Sk, 128, 128, 0),
                               plan.tail_first + (t - plan.tail_first) // 2)
        tile = (t - plan.tail_first) % 2
        assert (task.b, task.g, task.mblock) == (pair.b, pair.g, pair.mblock)
        assert task.pos0[0] == task.pos0[1] == pair.pos0[tile]
        if pair.n_blocks[tile] == 0:  # a tile past the end of the sequence
            assert task.n_blocks[0] == task.n_blocks[1] == task.key_split == 0
            continue
        nb = plan.kv_blocks
        assert task.n_blocks[0] == (nb + 1) // 2 and task.n_blocks[1] == nb // 2
        assert task.key_split == task.n_blocks[0]


def test_split_tasks_run_in_the_last_wave():
    """With round-robin assignment the split tasks are the last task of
    distinct CTAs, after every CTA has run the same number of whole tasks, and
    the busiest CTA's key blocks drop from 14 tasks' worth to 13.5."""
    plan = fa.fa_make_plan(4, 16, 16, 8192, 8192, 128, 128, 0)
    grid = 152

    def busiest(pl):
        load = [0] * grid
        for t in range(pl.num_tasks):
            task = fa.fa_plan_task(pl, t)
            # stage-steps: the two stages run side by side, a task takes its longer stage's blocks
            load[t % grid] += max(task.n_blocks)
        return max(load)

    before = busiest(plan)
    fa.fa_plan_set_grid(plan, grid)
    first = plan.tail_first
    assert first % grid == 0
    ctas = [t % grid for t in range(first, plan.num_tasks)]
    assert len(set(ctas)) == len(ctas)
    assert before == 14 * 64 and busiest(plan) == 13 * 64 + 32


@pytest.mark.parametrize("case", [
    (1, 4, 4, 1024, 384, 0, 152),      # 3 key blocks: too few to split
    (1, 16, 16, 4096, 4096, 0, 152),   # 256 tasks: 104 left over, 2 x 104 > 152
    (2, 16, 16, 4864, 4096, 0, 152),   # 608 tasks = 4 x 152: no partial wave
])
def test_no_split(case):
    B, Hq, Hkv, Sq, Sk, causal, grid = case
    plan = fa.fa_make_plan(B, Hq, Hkv, Sq, Sk, 128, 128, causal)
    pairs = plan.num_tasks
    fa.fa_plan_set_grid(plan, grid)
    assert plan.num_tasks == pairs and plan.tail_first == pairs
    assert all(fa.fa_plan_task(plan, t).key_split == 0 for t in range(0, plan.num_tasks, 37))


# ---------------------------------------------------------------------------
# the paired causal order
# ---------------------------------------------------------------------------

def blocks(task):
    return task.n_blocks[0] + task.n_blocks[1]


PAIRED = [
    # (B, Hq, Hkv, S, grid)
    (32, 16, 16, 1024, 152),    # 1024 pairs: 6 whole blocks, 112 left over on one CTA each
    (4, 16, 16, 8192, 152),
    (1, 16, 16, 32768, 152),
    (4, 32, 8, 8192, 152),      # GQA: 2048 pairs, 72 left over split over two CTAs each
    (4, 32, 1, 8192, 152),      # MQA
    (2, 16, 16, 16384, 152),
    (1, 3, 3, 1024, 5),         # 6 pairs on 5 CTAs: one left over
    (1, 2, 2, 2048, 16),        # 8 pairs on 16 CTAs: no whole block
]


@pytest.mark.parametrize("case", PAIRED, ids=[f"B{c[0]}H{c[1]}/{c[2]}S{c[3]}g{c[4]}" for c in PAIRED])
def test_paired_order(case):
    B, Hq, Hkv, S, grid = case
    base = fa.fa_make_plan(B, Hq, Hkv, S, S, 128, 128, 1)
    plan = fa.fa_make_plan(B, Hq, Hkv, S, S, 128, 128, 1)
    fa.fa_plan_set_grid(plan, grid)
    M = plan.mblocks
    units = plan.batch * plan.groups
    pairs = units * M // 2
    full, r = divmod(pairs, grid)
    body = 2 * full * grid
    packed = r and 2 * r > grid and plan.num_tasks != body + grid + r
    if packed:  # left-over heavy tasks on CTAs 0 .. r-1, light ones dealt over the others
        want = body + -(-r // (grid - r)) * grid
    else:
        want = body + (0 if r == 0 else (2 * r if 2 * r <= grid else grid + r))
    assert M % 2 == 0 and plan.num_tasks == want
    tasks = plan_tasks(plan)
    # every (b, g, m_block) exactly once, with the blocks the plain order gives it
    plain = {(t.b, t.g, t.mblock): (tuple(t.pos0), tuple(t.n_blocks)) for t in plan_tasks(base)}
    seen = {}
    for t in tasks:
        if t.n_blocks[0] == 0 and t.n_blocks[1] == 0:  # an empty entry
            assert t.pos0[0] == t.pos0[1] == S
            continue
        key = (t.b, t.g, t.mblock)
        assert key not in seen
        seen[key] = (tuple(t.pos0), tuple(t.n_blocks))
    assert seen == plain
    # inside the whole blocks CTA c runs a light task and then its heavy complement
    for i in range(0, body, 2 * grid):
        for c in range(grid):
            l, h = tasks[i + c], tasks[i + grid + c]
            assert (h.b, h.g) == (l.b, l.g) and h.mblock + l.mblock == M - 1 and h.mblock >= M // 2
            if plan.pack == 1:  # (4m + 3) + (4(M - 1 - m) + 3) key blocks
                assert blocks(h) + blocks(l) == 4 * M + 2
            else:  # packed rows: 128 / pack positions per tile, the same total within a block
                assert abs(blocks(h) + blocks(l) - 2 * plan.kv_blocks - 1) <= 1
    # the pairs left over: their two tasks on two CTAs (2r <= G), on one, or packed
    tail = tasks[body:]
    if packed:
        heavy = [(t.b, t.g, t.mblock) for t in tail[:r]]
        assert all(m >= M // 2 for _, _, m in heavy)
        lights = [(i, t) for i, t in enumerate(tail) if blocks(t) and i % grid >= r]
        assert len(lights) == r and all(blocks(t) == 0 for i, t in enumerate(tail[grid:]) if i % grid < r)
        assert sorted((b, g, M - 1 - m) for b, g, m in heavy) == sorted((t.b, t.g, t.mblock) for _, t in lights)
    elif r and 2 * r <= grid:
        for c in range(r):
            assert tail[c].mblock + tail[r + c].mblock == M - 1 and tail[r + c].mblock >= M // 2
    elif r:
        for c in range(r):
            assert tail[c].mblock + tail[grid + c].mblock == M - 1 and tail[grid + c].mblock >= M // 2
        assert all(blocks(t) == 0 for t in tail[r:grid])


def cta_load(plan, grid, ovh=2.5):
    """Per-CTA work: blocks of both stages / 2 per task plus a fixed start-up."""
    load = [0.0] * grid
    for t in range(plan.num_tasks):
        task = fa.fa_plan_task(plan, t)
        if blocks(task):
            load[t % grid] += blocks(task) / 2 + ovh
    return load


@pytest.mark.parametrize("S", [1024, 2048, 4096, 8192, 16384, 32768])
def test_paired_order_balances_the_causal_sweep(S):
    """The causal benchmark sweep (32k tokens, 16 heads): the busiest CTA's
    modelled work drops from 6-13 % above the average to at most 2 % (whole
    pairs alone would leave the quantisation ceil(P / G) / (P / G): 3.9 % for
    1024 pairs on 152 CTAs; packing the last wave's light tasks removes most
    of it)."""
    B, grid = 32768 // S, 152
    plain = fa.fa_make_plan(B, 16, 16, S, S, 128, 128, 1, 64 << 20)
    paired = fa.fa_make_plan(B, 16, 16, S, S, 128, 128, 1, 64 << 20)
    fa.fa_plan_set_grid(paired, grid)
    a, b = cta_load(plain, grid), cta_load(paired, grid)
    avg = sum(a) / grid
    assert abs(sum(b) / grid - avg) < 1e-9
    assert max(a) / avg > 1.05
    # the last wave packs the light complements of its heavy tasks (model: 0.5-1.8 % over the average)
    assert max(b) / avg <= 1.02


def test_paired_order_needs_even_mblocks():
    plan = fa.fa_make_plan(1, 4, 4, 768, 768, 128, 128, 1)  # 3 m_blocks
    n = plan.num_tasks
    fa.fa_plan_set_grid(plan, 152)
    assert plan.num_tasks == n
    assert [fa.fa_plan_task(plan, t).mblock for t in range(n)] == \
        [fa.fa_plan_task(fa.fa_make_plan(1, 4, 4, 768, 768, 128, 128, 1), t).mblock for t in range(n)]


def test_set_grid_rejects_bad_calls():
    plan = fa.fa_make_plan(1, 2, 2, 1024, 1024, 128, 128, 0)
    with pytest.raises(fa.FaError):
        fa.fa_plan_set_grid(plan, 0)
    fa.fa_plan_set_grid(plan, 152)
    with pytest.raises(fa.FaError):  # already applied
        fa.fa_plan_set_grid(plan, 152)


def test_packing_only_when_the_light_tasks_fit():
    """With r close to G the light complements of the left-over heavy tasks
    would pile up on the few free CTAs beyond a whole pair's cost: the cost
    model then keeps each pair on one CTA."""
    # 1 x 16 heads, 64 m_blocks: 512 pairs; grid 257 leaves r = 255 (G - r = 2)
    plan = fa.fa_make_plan(1, 16, 16, 16384, 16384, 128, 128, 1)
    fa.fa_plan_set_grid(plan, 257)
    pairs, grid = 512, 257
    full, r = divmod(pairs, grid)
    assert r == 255
    assert plan.num_tasks == 2 * full * grid + grid + r  # whole pairs on one CTA each
    # a grid that leaves few enough light tasks per free CTA packs them
    plan = fa.fa_make_plan(4, 16, 16, 8192, 8192, 128, 128, 1)
    fa.fa_plan_set_grid(plan, 152)
    assert plan.num_tasks == 2 * 6 * 152 + 3 * 152  # 112 left over: 3 waves of light tasks
