"""Balanced last wave (key-split tail tasks), host view: no GPU needed.

A non-causal problem of P tasks on G persistent CTAs (task t on CTA t mod G)
ends with a partial wave of r = P mod G tasks.  When 2r <= G the kernel runs
each tile of those r tasks as one task whose two stages take the two halves of
the key blocks ("Infra: Flash Attention", "Prefill and decode": key segments
computed apart merge exactly).  These tests check, through the library's host
copy of the schedule, that the tasks still cover every (tile, key block) once,
that the split tasks land in the last wave, and when the split applies.
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
    (4, 16, 16, 8192, 8192, 1, 152),   # causal: the longest-first order already balances
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


def test_set_grid_rejects_bad_calls():
    plan = fa.fa_make_plan(1, 2, 2, 1024, 1024, 128, 128, 0)
    with pytest.raises(fa.FaError):
        fa.fa_plan_set_grid(plan, 0)
    fa.fa_plan_set_grid(plan, 152)
    with pytest.raises(fa.FaError):  # already applied
        fa.fa_plan_set_grid(plan, 152)
