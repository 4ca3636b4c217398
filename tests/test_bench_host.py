"""Host logic of bench.py that needs no GPU: the order in which the timed steps
replay their CUDA graphs (whole cycles of input sets, single steps for the
rest) must run exactly the requested steps, each on its own input set, in order."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _trace(first, count, nsets):
    sets = []
    bench.replay_steps(first, count, nsets, lambda: sets.extend(range(nsets)), sets.append)
    return sets


@pytest.mark.parametrize("nsets", [1, 2, 5, 7])
@pytest.mark.parametrize("first", [0, 1, 3, 5, 10])
@pytest.mark.parametrize("count", [0, 1, 4, 5, 6, 50, 53])
def test_replay_steps_runs_each_step_on_its_set(nsets, first, count):
    assert _trace(first, count, nsets) == [i % nsets for i in range(first, first + count)]


def test_replay_steps_uses_whole_cycles_when_aligned():
    calls = []
    bench.replay_steps(5, 50, 5, lambda: calls.append("cycle"), lambda k: calls.append(k))
    assert calls == ["cycle"] * 10
    calls.clear()
    bench.replay_steps(3, 9, 5, lambda: calls.append("cycle"), lambda k: calls.append(k))
    assert calls == [3, 4, "cycle", 0, 1]
