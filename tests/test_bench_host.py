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


def test_profiled_traffic_matches_kernel_source_and_token_count(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed summary only when its source
    hash is the current one of the kernel the line times: gemv.cu for one
    token, gemv_batch.cu for nt > 1 (per token count), gemv_f32.cu for f32."""
    import os
    import shutil
    import bench
    csrc = tmp_path / "quant_quantized_gemv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("gemv.cu", "gemv_batch.cu", "gemv_f32.cu", "gemv_common.cuh", "layout.h", "gemv_gateup.cu"):
        shutil.copy(os.path.join(bench.ROOT, "quant_quantized_gemv_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    one, batch, f32 = bench.gemv_source_hash(), bench.gemv_source_hash(batch=True), bench.gemv_source_hash("f32")
    assert len({one, batch, f32}) == 3
    (tmp_path / "profiles" / "gemv_w.md").write_text(f"source_sha256_16: {one}\ntraffic_bytes_per_launch: 100\n")
    (tmp_path / "profiles" / "gemv_batch_w.md").write_text(
        f"source_sha256_16: {batch}\ntraffic_bytes_per_launch_nt2: 200\ntraffic_bytes_per_launch_nt4: 400\n")
    (tmp_path / "profiles" / "gemv_f32_w.md").write_text(f"source_sha256_16: {one}\ntraffic_bytes_per_launch: 300\n")
    assert bench.profiled_traffic("w") == 100
    assert bench.profiled_traffic("w", tokens=2) == 200 and bench.profiled_traffic("w", tokens=4) == 400
    assert bench.profiled_traffic("w", tokens=8) is None                 # no capture at that count
    assert bench.profiled_traffic("w", "f32") is None                    # taken on another kernel's source
    assert bench.profiled_traffic("w", gateup=True) is None              # the source set differs
    (csrc / "gemv_batch.cu").write_text("// changed\n")
    assert bench.profiled_traffic("w", tokens=2) is None                 # kernel changed since the capture
    assert bench.profiled_traffic("w") == 100
