"""The benchmark's timed region holds graph replays only.

Decode steps are replayed from CUDA graphs of `group` steps; a graph is
captured the first time a length is asked for.  These host checks replay the
bench's own planning functions over many warm-up / step counts and assert
that every graph length the warm-up, the timed steps and the percentile
replays ask for is in the set captured before the first timed event, so no
capture can fall between the events (the bench also raises if one does).
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("group", [1, 3, 8, 16])
def test_every_replayed_graph_is_captured_before_timing(group):
    for warmup in range(0, 40):
        for steps in range(1, 70):
            pre = set(bench.precapture_sizes(warmup, steps, group))
            timed = bench.graph_sizes(steps, group)
            assert set(timed) <= pre, (warmup, steps, group)
            assert set(bench.graph_sizes(warmup, group)) <= pre
            assert group in pre                       # percentile replays
            # the replays add up to exactly the requested step count
            full, rest = divmod(steps, group)
            assert full * group + rest == steps
            assert sum(bench.graph_sizes(steps, group)) == (group if full else 0) + rest


def test_driver_configuration():
    # the configuration the full test run uses: 20 steps after 5 warm-ups over
    # 8 rotating tables -> graphs of 8 and 4 steps, and of 5 for the warm-up
    assert bench.graph_sizes(20, 8) == [8, 4]
    assert bench.precapture_sizes(5, 20, 8) == [4, 5, 8]


def test_every_named_workload_is_defined_and_selectable():
    # the headline, its secondary lines and the one-thread baselines name
    # workloads that workloads.NAMED builds and --workload accepts
    import workloads
    names = {bench.HEADLINE, *bench.SECONDARY, *bench.ONE_THREAD_TOO}
    assert names <= set(workloads.NAMED)
    assert names <= set(bench.WORKLOAD_TEXT)
    for n in names:
        assert bench.parse_args(["--workload", n]).workload == n
