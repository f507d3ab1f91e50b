"""Host logic of bench.py's timed region, on CPU with a stand-in for
torch.cuda: exactly K layer calls are timed, cycling through the input
copies in order, captured into graphs of at most 64 calls."""
import os
import sys
import types

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def _fake_torch(log):
    class Event:
        def __init__(self, **kw):
            pass

        def record(self):
            log.append(("event",))

        def elapsed_time(self, other):
            return 2.5

    class Graph:
        def __init__(self):
            self.calls = []

        def replay(self):
            log.extend(("step", i) for i in self.calls)

    class Capture:
        current = None

        def __init__(self, g):
            self.g = g

        def __enter__(self):
            Capture.current = self.g
            return self

        def __exit__(self, *a):
            Capture.current = None
            return False

    cuda = types.SimpleNamespace(CUDAGraph=Graph, graph=Capture, synchronize=lambda: None,
                                 _sleep=lambda n: None, Event=Event)
    return types.SimpleNamespace(cuda=cuda), Capture


@pytest.mark.parametrize("steps", [1, 7, 8, 63, 64, 65, 130, 2000])
def test_layer_sequence_times_exactly_k_steps(steps):
    import bench
    log = []
    torch, cap = _fake_torch(log)
    fns = []
    for i in range(bench.NCOPY):
        def fn(i=i):
            assert cap.current is not None, "calls happen only inside a capture"
            cap.current.calls.append(i)
        fns.append(fn)
    barriers = []
    total, how = bench.time_layer_sequence(torch, fns, steps, barrier=lambda: barriers.append(1))
    G = min(steps, 64)
    assert total == 2.5
    assert f"graphs of {G} " in how
    # the timed part: everything between the two event records after the loaded warm-up
    ev = [i for i, e in enumerate(log) if e == ("event",)]
    assert len(ev) == 2
    timed = [e[1] for e in log[ev[0] + 1:ev[1]]]
    assert len(timed) == steps
    # copies in turn; each graph starts again at copy 0
    expect = [j % bench.NCOPY for j in range(G)] * (steps // G) + \
        [j % bench.NCOPY for j in range(steps % G)]
    assert timed == expect
    assert len(barriers) == 2


def test_one_core_pins_every_thread_and_restores_them():
    import threading
    import bench
    stop = threading.Event()
    worker = threading.Thread(target=stop.wait)
    worker.start()
    try:
        tids = [int(t) for t in os.listdir("/proc/self/task")]
        before = {t: os.sched_getaffinity(t) for t in tids}
        with bench.OneCore() as one:
            assert one.ok
            for t in tids:
                assert os.sched_getaffinity(t) == {one.core}
        for t in tids:
            assert os.sched_getaffinity(t) == before[t]
    finally:
        stop.set()
        worker.join()
