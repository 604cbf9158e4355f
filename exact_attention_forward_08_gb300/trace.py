"""Reader of the forward kernel's event log (``fa_options.trace``).

The trace build of the kernel stamps the SM clock at each step of the
hand-off protocol between its roles: lane 0 of each role's first warp writes
one 64-bit record {event code (bits 56-63), argument (bits 32-55), clock low
32 bits} to its track.  Buffer layout, for CTA c < trace_ctas and track k:
word (c * 5 + k) * (cap + 1) holds the record count, the records follow.

``decode`` turns the words into per-CTA, per-track event lists with clock
values unwrapped relative to the CTA (all tracks of a CTA read the same SM
clock).  ``summarize`` measures the intervals the kernel's performance
argument rests on: per Q stage and K/V block, the softmax's wait for S and
its work from S to P (TMEM load, row maximum, exponentials, P stored); the
MMA warp's latency to see P and its issue times; the
latency from a Q K^T issue to the softmax seeing S; the period of a stage's
blocks; and, per task boundary, the gap between one task's last P V and the
next task's first.  Times are in SM clock cycles.

``summarize_bwd`` does the same for the backward kernels' log (one kernel's
half of the buffer): per 64-row stage and streamed block, the row warps'
wait for S and dP and their work to P (and dS) stored, the MMA warp's issue
of the accumulating GEMMs and of the next S and dP, its waits, and the
hand-offs between them.
"""
from __future__ import annotations

import statistics

TRACKS = ("softmax0", "softmax1", "correction", "mma", "tma")
EVENTS = {
    1: "sm_task", 2: "sm_wait", 3: "sm_s", 4: "sm_ld", 5: "sm_max", 6: "sm_exp0", 7: "sm_exp1", 8: "sm_p",
    16: "co_task", 17: "co_corr", 18: "co_rescaled", 19: "co_arrive", 20: "co_odone", 21: "co_epi",
    32: "mm_task", 33: "mm_kv", 34: "mm_q", 35: "mm_p", 36: "mm_pv", 37: "mm_qk",
    48: "ld_task", 49: "ld_q", 50: "ld_kvwait", 51: "ld_kv",
    # backward (tracks softmax0 / softmax1 = row warps of stage 0 / 1, mma, tma)
    64: "br_task", 65: "br_wait", 66: "br_s", 67: "br_p", 68: "br_acc", 69: "br_epi",
    80: "bm_task", 81: "bm_p", 82: "bm_acc", 83: "bm_t", 84: "bm_sdp",
    96: "bl_task", 97: "bl_t",
}
CODES = {v: k for k, v in EVENTS.items()}


def trace_words(ctas: int, cap: int) -> int:
    """64-bit words of a trace buffer for `ctas` recording CTAs and `cap` records per track."""
    return ctas * len(TRACKS) * (cap + 1)


def decode(words, ctas: int, cap: int):
    """Per CTA, a dict track name -> list of (cycle, event name, argument).

    words: a sequence of unsigned 64-bit integers (e.g. a numpy uint64 array).
    Cycles are relative to the CTA's first recorded event, unwrapped from the
    32-bit clock field (events of one launch lie within 2^31 cycles of it).
    Records past `cap` were counted by the kernel but not kept.
    """
    out = []
    stride = cap + 1
    for c in range(ctas):
        raw = {}
        for k, name in enumerate(TRACKS):
            base = (c * len(TRACKS) + k) * stride
            n = int(words[base])
            recs = []
            for i in range(min(n, cap)):
                w = int(words[base + 1 + i])
                recs.append((w & 0xFFFFFFFF, EVENTS.get(w >> 56, str(w >> 56)), (w >> 32) & 0xFFFFFF))
            raw[name] = (n, recs)
        firsts = [recs[0][0] for _, recs in raw.values() if recs]
        ref = firsts[0] if firsts else 0
        # the earliest event, taken modulo 2^32 around any one of them
        rel = [((f - ref + (1 << 31)) % (1 << 32)) - (1 << 31) for f in firsts]
        ref = (ref + min(rel)) % (1 << 32) if rel else 0
        cta = {}
        for name, (n, recs) in raw.items():
            cta[name] = [(((t - ref + (1 << 31)) % (1 << 32)) - (1 << 31), ev, arg) for t, ev, arg in recs]
        cta["_counts"] = {name: raw[name][0] for name in TRACKS}
        out.append(cta)
    return out


def _stats(xs):
    if not xs:
        return None
    xs = sorted(xs)
    q = lambda f: xs[min(len(xs) - 1, int(f * (len(xs) - 1) + 0.5))]
    return {"n": len(xs), "median": q(0.5), "mean": round(statistics.fmean(xs), 1), "p10": q(0.1), "p90": q(0.9)}


def _stage_of(arg: int) -> int:
    return arg >> 16


def _block_of(arg: int) -> int:
    return arg & 0xFFFF


def summarize(ctas) -> dict:
    """Interval statistics over every decoded CTA (cycles)."""
    acc = {}

    def add(key, v):
        acc.setdefault(key, []).append(v)

    for cta in ctas:
        # softmax phases, per stage; the n-th S / P of a stage pairs with the
        # n-th MMA commit / wait of that stage
        sm_s = {0: [], 1: []}
        sm_p = {0: [], 1: []}
        for s in (0, 1):
            evs = cta[f"softmax{s}"]
            cur = {}
            for t, ev, arg in evs:
                if ev == "sm_wait":
                    cur = {"sm_wait": t, "j": arg}
                elif ev == "sm_s":
                    cur["sm_s"] = t
                    sm_s[s].append((t, arg))
                elif ev == "sm_p":
                    sm_p[s].append((t, arg))
                    if "sm_wait" in cur and "sm_s" in cur:
                        tag = "first" if cur["j"] == 0 else "steady"
                        add(f"softmax.{tag}.wait_for_S", cur["sm_s"] - cur["sm_wait"])
                        add(f"softmax.{tag}.work_S_to_P", t - cur["sm_s"])
            # block period of a stage: consecutive S inside a task (j -> j + 1)
            for (t0, j0), (t1, j1) in zip(sm_s[s], sm_s[s][1:]):
                if j1 == j0 + 1:
                    add("stage.block_period", t1 - t0)
        # MMA warp
        mm = cta["mma"]
        mm_qk = {0: [], 1: []}
        mm_p = {0: [], 1: []}
        last_issue = None  # the last Q K^T or P V issued
        last_p = last_pv_t = None
        pv_last_of_task = []
        first_pv_of_task = []
        task_first_qk = []
        seen_pv_in_task = False
        for t, ev, arg in mm:
            if ev == "mm_task":
                if last_pv_t is not None:
                    pv_last_of_task.append(last_pv_t)
                seen_pv_in_task = False
                task_first_qk.append(None)
            elif ev == "mm_qk":
                mm_qk[_stage_of(arg)].append((t, _block_of(arg)))
                if task_first_qk and task_first_qk[-1] is None:
                    task_first_qk[-1] = t
                elif last_pv_t is not None and seen_pv_in_task:
                    add("mma.issue_QK_after_PV", t - last_pv_t)
                last_issue = t
            elif ev == "mm_p":
                mm_p[_stage_of(arg)].append((t, _block_of(arg)))
                if last_issue is not None:
                    add("mma.wait_for_P" + (".first" if _block_of(arg) == 0 else ".steady"), t - last_issue)
                last_p = t
            elif ev == "mm_pv":
                if last_p is not None:
                    add("mma.issue_PV", t - last_p)
                if not seen_pv_in_task:
                    first_pv_of_task.append(t)
                    seen_pv_in_task = True
                last_pv_t = last_issue = t
        # hand-off latencies (the n-th of each stage)
        for s in (0, 1):
            for (tq, jq), (ts, js) in zip(mm_qk[s], sm_s[s]):
                add("handoff.QK_issue_to_softmax_S" + (".first" if js == 0 else ".steady"), ts - tq)
            for (tp, jp), (tm, jm) in zip(sm_p[s], mm_p[s]):
                add("handoff.softmax_P_to_mma_P" + (".first" if jp == 0 else ".steady"), tm - tp)
        # task boundaries: last P V of task k -> first P V of task k + 1
        for a, b in zip(pv_last_of_task, first_pv_of_task[1:]):
            add("task.last_PV_to_next_first_PV", b - a)
        for a, b in zip(pv_last_of_task, [x for x in task_first_qk[1:] if x is not None]):
            add("task.last_PV_to_next_first_QK", b - a)
        # correction: O-done wait after the last P V, epilogue length
        co = cta["correction"]
        od = {}
        for t, ev, arg in co:
            if ev == "co_odone":
                od[arg] = t
            elif ev == "co_epi" and arg in od:
                add("correction.epilogue_per_stage", t - od.pop(arg))
        # TMA: tile issue to the MMA warp seeing it ready (the n-th tile)
        ld = [(t, arg) for t, ev, arg in cta["tma"] if ev == "ld_kv"]
        kv = {}
        for t, ev, arg in mm:
            if ev == "mm_kv" and arg not in kv:
                kv[arg] = t
        for t, it in ld:
            if it in kv:
                add("tma.tile_issue_to_mma_ready", kv[it] - t)
        span = [t for name in TRACKS for t, _, _ in cta[name]]
        if span:
            add("cta.span", max(span) - min(span))
    return {k: _stats(v) for k, v in sorted(acc.items())}


def summarize_bwd(ctas) -> dict:
    """Interval statistics of the backward event log over every decoded CTA
    (cycles).  Row events carry the streamed block `it` of the task, MMA
    events stage << 16 | it."""
    acc = {}

    def add(key, v):
        acc.setdefault(key, []).append(v)

    for cta in ctas:
        br_s = {0: [], 1: []}
        br_p = {0: [], 1: []}
        for s in (0, 1):
            cur = {}
            for t, ev, arg in cta[f"softmax{s}"]:
                if ev == "br_wait":
                    cur = {"wait": t, "it": arg}
                elif ev == "br_s":
                    cur["s"] = t
                    br_s[s].append((t, arg))
                elif ev == "br_p":
                    br_p[s].append((t, arg))
                    if "wait" in cur and "s" in cur:
                        tag = "first" if cur["it"] == 0 else "steady"
                        add(f"row.{tag}.wait_for_S", cur["s"] - cur["wait"])
                        add(f"row.{tag}.work_S_to_P", t - cur["s"])
                elif ev == "br_acc":
                    cur = {"acc": t}
                elif ev == "br_epi" and "acc" in cur:
                    add("row.epilogue", t - cur["acc"])
            for (t0, i0), (t1, i1) in zip(br_p[s], br_p[s][1:]):
                if i1 == i0 + 1:
                    add("stage.block_period", t1 - t0)
        bm_p = {0: [], 1: []}
        bm_sdp = {0: [], 1: []}
        last = None
        last_acc = None
        task_last_acc, task_first_acc = [], []
        first_in_task = True
        for t, ev, arg in cta["mma"]:
            s = _stage_of(arg)
            if ev == "bm_task":
                if last_acc is not None:
                    task_last_acc.append(last_acc)
                first_in_task = True
                last = t
            elif ev == "bm_p":
                bm_p[s].append((t, _block_of(arg)))
                if last is not None:
                    add("mma.wait_for_P", t - last)
                last = t
            elif ev == "bm_acc":
                if last is not None:
                    add("mma.issue_acc", t - last)
                if first_in_task:
                    task_first_acc.append(t)
                    first_in_task = False
                last = last_acc = t
            elif ev == "bm_t":
                if last is not None:
                    add("mma.wait_T", t - last)
                last = t
            elif ev == "bm_sdp":
                bm_sdp[s].append((t, _block_of(arg)))
                if last is not None:
                    add("mma.issue_S_dP", t - last)
                last = t
        for s in (0, 1):
            for (tr_, _), (tm, _) in zip(br_p[s], bm_p[s]):
                add("handoff.row_P_to_mma_P", tm - tr_)
            for (tq, _), (ts, _) in zip(bm_sdp[s], br_s[s]):
                add("handoff.S_dP_issue_to_row_S", ts - tq)
        for a, b in zip(task_last_acc, task_first_acc[1:]):
            add("task.last_acc_to_next_first_acc", b - a)
        issued = [t for t, ev, _ in cta["tma"] if ev == "bl_t"]
        ready = [t for t, ev, _ in cta["mma"] if ev == "bm_t"]
        for a, b in zip(issued, ready):
            add("tma.half_tile_issue_to_mma_ready", b - a)
        span = [t for name in TRACKS for t, _, _ in cta[name]]
        if span:
            add("cta.span", max(span) - min(span))
    return {k: _stats(v) for k, v in sorted(acc.items())}
