"""Host logic of bench.py on the CPU: the roofline bound and fraction, the
traffic record lookup (reported only while the kernel sources are the ones
profiled), the clock-sample summary, and the order the pipelined end-to-end
steps impose on copies and kernels (checked against a recording stand-in for
the few torch stream/event calls it makes)."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench        # noqa: E402
import workloads    # noqa: E402


def fixed_peaks(monkeypatch, tflops=2000.0, gbs=8000.0):
    monkeypatch.setattr(bench, "read_peaks", lambda window_s=0.0: (tflops, gbs, "test"))


def test_roofline_tensor_bound_square(monkeypatch):
    fixed_peaks(monkeypatch)
    w = workloads.WORKLOADS["fused8192"]
    ms = 0.55
    r = bench.roofline(w, ms, None, {"path": 2, "stages": 3, "tile_m": 256, "tile_n": 256}, 0.01)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(2 * 8192 ** 3 / (ms * 1e-3) / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["ridge_flop_per_byte"] == pytest.approx(2000e12 / 8000e9)
    assert r["intensity_flop_per_byte"] > r["ridge_flop_per_byte"]


def test_roofline_hbm_bound_skinny(monkeypatch):
    fixed_peaks(monkeypatch)
    w = workloads.WORKLOADS["skinny16x8192x8192"]
    ms = 0.03
    r = bench.roofline(w, ms, 1.0e8, {"path": 3, "stages": 12, "tile_m": 16, "tile_n": 128}, 0.01)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(w.alg_bytes() / (ms * 1e-3) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 8000.0)
    assert r["traffic"] == 1.0e8


def test_read_peaks_falls_back_without_measurements(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    tf, gb, src = bench.read_peaks()
    assert src == "fallback burst" and tf == bench.FALLBACK_TENSOR_TFLOPS and gb == bench.FALLBACK_HBM_GBS
    tf, gb, src = bench.read_peaks(bench.SUSTAINED_WINDOW_S)
    assert src == "fallback sustained" and tf == bench.FALLBACK_TENSOR_SUSTAINED_TFLOPS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                                                              "hbm_gbs": 7000.0}))
    tf, gb, src = bench.read_peaks()
    assert src == "measured bf16 burst" and tf == pytest.approx(1900.0 * bench.FP16_PER_BF16) and gb == 7000.0
    # a timed window long enough to run under the power cap: the sustained peak
    tf, gb, src = bench.read_peaks(0.7)
    assert src == "measured bf16 sustained" and tf == pytest.approx(1700.0 * bench.FP16_PER_BF16)
    tf, _, _ = bench.read_peaks(0.012)
    assert tf == pytest.approx(1900.0 * bench.FP16_PER_BF16)


def test_committed_traffic_only_for_the_profiled_sources(monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    rec = {"w": {"kernel_source_hash": "abc", "dram_bytes_per_launch": 123}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda sources=None: "abc")
    assert bench.committed_traffic("w") == 123
    assert bench.committed_traffic("other") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda sources=None: "changed")
    assert bench.committed_traffic("w") is None


def test_committed_records_are_consistent():
    # every record names the hash of the sources it was taken from (a record
    # whose sources changed since is reported as null, not as a wrong number)
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for name, r in rec.items():
        h = r["kernel_source_hash"]
        assert len(h) == 16 and int(h, 16) >= 0, name
        assert r["dram_bytes_per_launch"] == r["dram_bytes_read"] + r["dram_bytes_write"], name


def test_clock_samples_parse_and_window():
    lines = [
        "2026/12/03 01:00:00.100, 0, 1400, 2070, 1380.5, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 01:00:00.200, 0, 1380, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 01:00:05.000, 0, 2070, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = bench.ClockSampler.parse(lines)
    assert len(s) == 3
    assert s[0][1] == 1400 and s[0][3] == {"sw_power_cap"} and s[2][3] == set()
    t0, t1 = s[0][0], s[1][0]
    summ = bench.ClockSampler.summarize(s, t0, t1, pad_s=0.05)
    assert summ["window"] == "timed" and summ["samples"] == 2
    assert summ["sm_mhz"] == pytest.approx(1390) and summ["reasons"] == ["sw_power_cap"]
    # a window with no sample in it falls back to the whole run
    summ = bench.ClockSampler.summarize(s, t1 + 1.0, t1 + 1.5, pad_s=0.0)
    assert summ["samples"] == 3 and summ["window"].startswith("whole run")


# ---------------------------------------------------------------- pipelined end-to-end steps

class _Event:
    def __init__(self, enable_timing=False):
        self.after = None          # (stream, position) recorded

    def record(self, stream):
        self.after = (stream, len(stream.ops))
        stream.ops.append(("record", self))

    def elapsed_time(self, other):
        return 1.0


class _Stream:
    def __init__(self, device=None):
        self.ops = []

    def wait_event(self, ev):
        self.ops.append(("wait", ev))


class _FakeTorch:
    """The stream / event calls pipelined_e2e makes, recorded per stream."""
    def __init__(self):
        self.current = None
        fake = self

        class _Ctx:
            def __init__(self, s):
                self.s = s

            def __enter__(self):
                self.prev, fake.current = fake.current, self.s

            def __exit__(self, *a):
                fake.current = self.prev

        class _Cuda:
            Stream = _Stream
            Event = _Event

            @staticmethod
            def stream(s):
                return _Ctx(s)

            @staticmethod
            def synchronize(dev=None):
                pass

            @staticmethod
            def current_stream():
                return fake.current

        self.cuda = _Cuda


def test_pipelined_e2e_orders_copies_and_kernels():
    torch = _FakeTorch()
    comp = _Stream()
    log = []

    def op(kind):
        def f(b):
            torch.current.ops.append((kind, b))
            log.append((kind, b, torch.current))
        return f

    bench.pipelined_e2e(torch, None, 1, 6, comp, op("in"), op("compute"), op("out"))
    # the timed run is the second call to run(): its six steps follow the three warm-up steps
    streams = {id(s): s for _, _, s in log}
    s_in = log[0][2]
    s_out = [s for k, _, s in log if k == "out"][0]
    assert len(streams) == 3 and log[1][2] is comp

    def position(stream, kind, i):
        seen = [j for j, o in enumerate(stream.ops) if o[0] == kind]
        return seen[i]

    def waits_before(stream, idx):
        """events this stream waits on before its op at position idx"""
        return [o[1] for o in stream.ops[:idx] if o[0] == "wait"]

    def event_of(stream, kind, i):
        # the event recorded right after the i-th op of this kind
        idx = position(stream, kind, i)
        nxt = stream.ops[idx + 1]
        assert nxt[0] == "record"
        return nxt[1]

    total = 3 + 6      # three warm-up steps, then the six timed ones; each run() counts from 0
    for i in range(total):
        li = i if i < 3 else i - 3
        b = li & 1
        assert s_in.ops[position(s_in, "in", i)] == ("in", b)
        assert comp.ops[position(comp, "compute", i)] == ("compute", b)
        assert s_out.ops[position(s_out, "out", i)] == ("out", b)
        # compute i waits for its copy-in; copy-out i waits for compute i
        assert event_of(s_in, "in", i) in waits_before(comp, position(comp, "compute", i))
        assert event_of(comp, "compute", i) in waits_before(s_out, position(s_out, "out", i))
        if li >= 2:   # within a run(): set b is reused two steps later
            # copy-in i overwrites set b only after compute i - 2 read it, and
            # compute i writes set b's result only after copy-out i - 2 read it
            assert event_of(comp, "compute", i - 2) in waits_before(s_in, position(s_in, "in", i))
            assert event_of(s_out, "out", i - 2) in waits_before(comp, position(comp, "compute", i))


def test_launch_stats_median_min_p90():
    import bench
    xs = [float(v) for v in range(1, 21)]          # 1 .. 20 ms
    st = bench.launch_stats(list(reversed(xs)))
    assert st["min"] == 1.0 and st["median"] == 10.5 and st["p90"] == 18.0 and st["n"] == 20
    assert st["mean"] == sum(xs) / 20
    one = bench.launch_stats([0.5])
    assert one["min"] == one["median"] == one["p90"] == one["mean"] == 0.5
