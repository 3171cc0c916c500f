"""Host-side logic of bench.py that needs no GPU."""
import bench


class _FakeWorkload:
    def __init__(self, seconds):
        self.seconds = seconds
        self.calls = 0

    def cpu_baseline(self, args):
        self.calls += 1
        # rate 2.0 on odd passes, 4.0 on even ones
        return {"value": 2.0 if self.calls % 2 else 4.0, "unit": "TFLOP/s", "cores": 1,
                "kind": "oracle", "sample": "one image", "seconds": self.seconds}


def test_cpu_baseline_repeats_to_the_minimum_time():
    wl = _FakeWorkload(3.0)
    r = bench.cpu_baseline_sampled(wl, None, min_seconds=10.0)
    assert wl.calls == 4 and r["seconds"] == 12.0
    assert r["value"] == (2 * 3 + 4 * 3 + 2 * 3 + 4 * 3) / 12.0
    assert r["sample"] == "one image, 4 passes" and r["kind"] == "oracle"


def test_cpu_baseline_single_long_pass_and_cap():
    wl = _FakeWorkload(25.0)
    r = bench.cpu_baseline_sampled(wl, None, min_seconds=10.0)
    assert wl.calls == 1 and r["sample"] == "one image, 1 pass" and r["value"] == 2.0
    wl = _FakeWorkload(0.5)
    r = bench.cpu_baseline_sampled(wl, None, min_seconds=10.0, max_passes=3)
    assert wl.calls == 3 and r["seconds"] == 1.5
