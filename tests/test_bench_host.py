"""Host logic of bench.py that needs no GPU: how the timed steps are split into graph launches."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def test_graph_replays_run_exactly_k_steps():
    for k in range(0, 130):
        for gs in (1, 4, 28):
            rest = k % gs if gs > 1 else 0
            for r in (rest, -1):
                seq = bench.graph_replays(k, gs, r)
                assert sum(n for _, n in seq) == k
                assert sum(1 for kind, _ in seq if kind == "rest") <= 1
                if gs > 1:
                    assert [kind for kind, _ in seq[:k // gs]] == ["multi"] * (k // gs)
                    assert all(n == gs for kind, n in seq if kind == "multi")
                else:
                    assert seq == [("single", 1)] * k


def test_graph_replays_default_and_short_runs():
    # 2000 steps in graphs of 28: 71 whole graphs and one graph of the last 12 steps
    assert bench.graph_replays(2000, 28, 12) == [("multi", 28)] * 71 + [("rest", 12)]
    # fewer steps than one graph holds: the whole run is the one remainder graph
    assert bench.graph_replays(20, 28, 20) == [("rest", 20)]
    # without a remainder graph the rest runs as single-step graphs
    assert bench.graph_replays(30, 28, -1) == [("multi", 28), ("single", 1), ("single", 1)]
    assert bench.graph_replays(56, 28, 0) == [("multi", 28)] * 2
