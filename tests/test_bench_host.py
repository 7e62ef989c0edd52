"""Host logic of bench.py's timing (no GPU): a timed region of K steps is
enqueued as CUDA graphs of at most m consecutive steps that cover exactly
steps start .. start + K - 1, one graph when K <= m, and graphs are shared
only between segments that use the same weight copies."""
import pytest


class _FakeGraph:
    def __init__(self, steps):
        self.replays = 0

    def replay(self):
        self.replays += 1


@pytest.fixture
def fake_capture(monkeypatch):
    import bench
    made = []

    def capture(fn, stream):
        g = _FakeGraph(None)
        made.append(g)
        return g

    monkeypatch.setattr(bench, "capture", capture)
    return made


def _steps_of(sg, start, k):
    return [s + j for s, n in sg._segments(start, k) for j in range(n)]


@pytest.mark.parametrize("K,m", [(20, 64), (64, 64), (65, 64), (100, 64), (2000, 64), (7, 3)])
def test_segments_cover_exactly_k_steps(K, m):
    import bench
    sg = bench.StepGraphs(lambda i: None, n_copies=1, m=min(m, K), stream=None)
    for start in (0, K, 3 * K):
        steps = _steps_of(sg, start, K)
        assert steps == list(range(start, start + K))
        assert all(n <= min(m, K) for _, n in sg._segments(start, K))
    if K <= m:
        assert len(list(sg._segments(0, K))) == 1       # one graph of exactly K steps


def test_graphs_shared_by_phase_only(fake_capture):
    import bench
    sg = bench.StepGraphs(lambda i: None, n_copies=10, m=16, stream=None)
    sg.prepare(0, 20)            # segments (0, 16), (16, 4): keys (0, 16), (6, 4)
    sg.prepare(20, 20)           # segments (20, 16), (36, 4): the same keys
    assert set(sg.cache) == {(0, 16), (6, 4)}
    sg.prepare(5, 16)            # another phase: a graph of its own
    assert (5, 16) in sg.cache
    n = len(fake_capture)
    sg.enqueue(0, 20)
    sg.enqueue(20, 20)
    assert len(fake_capture) == n                         # nothing captured while enqueuing
    assert sum(g.replays for g in fake_capture) == 4


def test_spread_reports_median_and_range():
    import bench
    s = bench.spread([3.0, 1.0, 2.0, 5.0, 4.0], 10.0, 1)
    assert s == {"median": 30.0, "min": 10.0, "max": 50.0, "n": 5}
