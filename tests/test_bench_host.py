"""Host-side logic of bench.py that decides what the timed region measures:
how many resident input copies keep the calls from being served from L2, and
the order in which the captured graphs walk through them."""
import bench

L2 = 126 << 20


def walk(R, G, K):
    """Copies used by the timed region's K calls: graphs[t % NG] for the
    first K / G - 1 replays, then the event graph on the copies next in turn."""
    plan = bench.graph_copies(R, G)
    NG = len(plan)
    seq = []
    for t in range(K // G - 1):
        seq += plan[t % NG]
    seq += plan[(K // G - 1) % NG]
    return seq


def test_large_inputs_keep_two_alternating_copies():
    # the mixed serving batch: 1.24 GB of logits and draft probs per call
    R = bench.input_copies(1_240_000_000, L2, 10)
    assert R == 2
    assert bench.graph_copies(R, 10) == [[0, 1] * 5]


def test_small_inputs_rotate_past_twice_l2():
    for call_bytes in (512_000, 17_800_000, 76_000_000, 140_000_000):
        for G in (10, 5, 4):
            R = bench.input_copies(call_bytes, L2, G)
            assert R * call_bytes >= 2 * L2
            assert R == 2 or R % G == 0
            assert R * call_bytes < 2 * L2 + G * call_bytes + 2 * call_bytes  # no more than needed


def test_walk_never_reuses_a_copy_within_r_calls():
    for call_bytes, G, K in ((17_800_000, 10, 500), (512_000, 10, 2000), (76_000_000, 10, 500),
                             (1_240_000_000, 10, 2000), (1_240_000_000, 3, 9), (17_800_000, 4, 8)):
        R = bench.input_copies(call_bytes, L2, G)
        seq = walk(R, G, K)
        assert len(seq) == K
        assert seq == [c % R for c in range(K)] or (R == 2 and seq == [c % 2 for c in range(K)])
        for a in range(0, K - R + 1, max(1, R // 2)):
            assert len(set(seq[a:a + R])) == R


class _FakeEvent:
    def __init__(self, enable_timing=False):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return 2.0


class _FakeStream:
    def __init__(self, device=None):
        pass

    def synchronize(self):
        pass


class _Ctx:
    def __init__(self, *a, **k):
        pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


class _FakeGraph:
    capturing = None

    def __init__(self):
        self.calls = []

    def replay(self):
        _FakeRun.used.extend(self.calls)


class _GraphCtx(_Ctx):
    def __init__(self, g, stream=None):
        self.g = g

    def __enter__(self):
        _FakeGraph.capturing = self.g
        return self

    def __exit__(self, *exc):
        _FakeGraph.capturing = None
        return False


class _FakeRun:
    """Stands in for runner.DeviceRun: records which logits copy each call
    (captured into a graph, or run eagerly) uses."""
    used = []

    def __init__(self, w, device=None, candidates=True, tile=0, **kw):
        import numpy as np
        import torch
        self.w = w
        n = w.n_positions
        self.d = {"logits": torch.zeros((n, w.V), dtype=torch.float32)}
        if w.is_verify:
            self.d["draft_probs"] = torch.zeros((int(w.cu_draft[-1]), w.V), dtype=torch.float32)
        self.plan = type("P", (), {"tile": 8192, "stage1_ctas": 304, "num_tiles": -(-w.V // 8192),
                                   "last_launches": lambda self: 3 if w.is_verify else 2})()
        self._np = np

    def __call__(self, stream=None, logits=None, draft_probs=None, events=None):
        key = (logits.data_ptr(), None if draft_probs is None else draft_probs.data_ptr())
        if _FakeGraph.capturing is not None:
            _FakeGraph.capturing.calls.append(key)

    def diag(self):
        return self._np.zeros(8, self._np.uint32)


def test_run_ours_walks_every_copy(monkeypatch, capsys):
    """bench.run_ours end to end on the CPU with stand-ins for the CUDA calls:
    the timed region's calls walk the resident copies in turn, and the JSON
    line reports them.  A small L2 takes the two-copy path of the large
    workloads; the real size takes the rotation."""
    import argparse
    import json
    import re
    import torch
    from spec_verification_gb300 import build, runner
    from spec_verification_gb300 import workloads as W
    monkeypatch.setattr(build, "build", lambda *a, **k: None)
    monkeypatch.setattr(runner, "DeviceRun", _FakeRun)
    monkeypatch.setattr(torch.cuda, "set_device", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "Stream", _FakeStream)
    monkeypatch.setattr(torch.cuda, "Event", _FakeEvent)
    monkeypatch.setattr(torch.cuda, "stream", _Ctx)
    monkeypatch.setattr(torch.cuda, "CUDAGraph", _FakeGraph)
    monkeypatch.setattr(torch.cuda, "graph", _GraphCtx)
    monkeypatch.setattr(bench, "event_ms", lambda a, b: 0.01)
    cases = [(W.verify_workload(3, 4, 20000, [2, 0, 1, 3], dtype="f32", q_dtype="f32"), 40),
             (W.sample_workload(5, 4, 9000, "f32"), 20),
             (W.sample_workload(5, 4, 9000, "f32"), 2000)]
    for l2 in (L2, 64 << 10):
        monkeypatch.setattr(torch.cuda, "get_device_properties",
                            lambda d, l2=l2: type("Props", (), {"L2_cache_size": l2})())
        for w, K in cases:
            _FakeRun.used = []
            args = argparse.Namespace(steps=K, warmup=3, tile=0, no_e2e=True, no_cpu=True, workload="c2", no_configs=True,
                                      cpu_seconds=1.0, e2e_steps=3)
            bench.run_ours(args, w, "test workload")
            line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
            assert line["steps"] == K and line["value"] > 0
            R = int(re.search(r"(\d+) resident copies", line["config"]["l2"]).group(1))
            call_bytes = w.n_positions * w.V * 4 + (int(w.cu_draft[-1]) * w.V * 4 if w.is_verify else 0)
            G = max(d for d in range(1, min(10, K) + 1) if K % d == 0)
            assert R == bench.input_copies(call_bytes, l2, G)
            assert R * call_bytes >= 2 * l2
            if l2 < call_bytes:
                assert R == 2
            timed = _FakeRun.used[-K:]  # the timed region is the last K calls replayed
            n = min(R, K)
            assert len(set(timed)) == n
            for a in range(0, K - n + 1):
                assert len(set(timed[a:a + n])) == n
