"""bench.py's host-side helpers (no GPU): the task-order label of the JSON
line comes from the library's host copy of the schedule."""
import bench


def test_balance_labels():
    g = 152
    assert bench.balance_of(bench.get_workload("mha8k"), g) == \
        "a partial last wave of 72 tasks runs as 144 key-split tiles"
    assert bench.balance_of(bench.get_workload("causal8k"), g) == "heavy and light m_blocks paired on one CTA"
    assert bench.balance_of(bench.get_workload("prof_mha"), g) == "plain order"  # 112 left over: 224 > 152
    assert bench.balance_of(bench.get_workload("varlen32k"), g) == ""  # dynamic assignment


def test_config_task_assignment():
    w = bench.get_workload("mha8k")
    cfg = bench.config_of(w, 1, w.flops(), False, 1, bench.balance_of(w, 152))
    assert cfg["task_assignment"].startswith("static round-robin; a partial last wave")
    assert bench.config_of(w, 1, w.flops(), True, 1, "x")["task_assignment"] == "dynamic (task counter)"
    d = bench.get_workload("decode32k")
    assert bench.config_of(d, 1, d.flops(), False, 7, "x")["task_assignment"] == "static round-robin"


def test_order_label_ablations():
    w = bench.get_workload("causal8k")
    assert bench.order_label(w, 152) == "heavy and light m_blocks paired on one CTA"
    assert bench.order_label(w, 152, no_balance=True) == "plain order (ablation)"
    assert bench.order_label(w, 152, stagger=True).endswith("; staggered exponentials (ablation)")
    assert bench.order_label(w, 152, store_mode=1).endswith("; staged TMA epilogue forced (ablation)")
    assert bench.order_label(w, 152, store_mode=2).endswith("; direct epilogue forced (ablation)")
    # the epilogue modes exist only in the fixed-length static kernels
    assert "epilogue" not in bench.order_label(w, 152, store_mode=1, dynamic=True)
    assert "epilogue" not in bench.order_label(bench.get_workload("varlen32k"), 152, store_mode=2)
