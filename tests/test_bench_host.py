"""CPU checks of the bench's host arithmetic and timing guards: the FLOP
count of the oracle's row sample, the clock record summary, the rule that
voids a throttled number, and the single re-measurement it triggers."""
import contextlib

import bench
from attention_forward_online_gb300.inputs import Workload


def _line(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    """One nvidia-smi sample in ClockSampler.FIELDS order."""
    return f"0, {sm}, {mx}, 900.0, 0x0, {hw}, {hwt}, {swt}, {cap}\n"


def test_row_flops_sum_matches_the_nominal_count():
    w = Workload("t_noncausal", "bf16", 2, 3, 64, 96, 64, False, None, seed=0)
    rows = range(w.B * w.H * w.Nq)
    assert bench.row_flops(w, rows) == w.flops
    # causal: the sample counts the i + 1 visible keys of row i, the headline
    # halves the square; the two differ by the diagonal, a factor (N + 1) / N
    c = Workload("t_causal", "bf16", 1, 2, 128, 128, 64, True, None, seed=0)
    got = bench.row_flops(c, range(c.B * c.H * c.Nq))
    assert got == c.flops * (c.Nq + 1) / c.Nq


def test_summarize_clocks_median_max_and_reasons():
    lines = [_line(2070, 2070), _line(1980, 2070, cap="Active"), _line(2070, 2070),
             "garbage line\n", _line("[N/A]", 2070)]
    info = bench.summarize_clocks(lines)
    assert info == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                    "samples": 3}
    assert bench.summarize_clocks([]) is None
    assert bench.summarize_clocks(["x, y\n"]) is None


def test_clocks_rejected_rule():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    assert bench.clocks_rejected(ok) is None
    assert bench.clocks_rejected(None) is None
    capped = dict(ok, sm_mhz=1500.0, reasons=["sw_power_cap"])
    assert bench.clocks_rejected(capped) is None  # power cap: kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert r in bench.clocks_rejected(dict(ok, reasons=[r]))
    locked = dict(ok, sm_mhz=1200.0)  # well below max with no reason: a clock lock
    assert "no reason" in bench.clocks_rejected(locked)
    assert bench.clocks_rejected(dict(ok, sm_mhz=1700.0)) is None  # within 80 %


class _FakeEvent:
    t = 0.0

    def __init__(self, enable_timing=True):
        pass

    def record(self, stream=None):
        _FakeEvent.t += 1.0
        self.at = _FakeEvent.t

    def elapsed_time(self, other):
        return other.at - self.at


class _FakeCuda:
    Event = _FakeEvent

    @staticmethod
    def synchronize(dev=None):
        pass

    @staticmethod
    def stream(s):
        return contextlib.nullcontext()


class _FakeTorch:
    cuda = _FakeCuda


class _Flush:
    def fill_(self, v):
        pass


def _run_timed(monkeypatch, records):
    """timed_steps with scripted clock records, one per timed loop."""
    script = list(records)
    loops = []

    class FakeSampler:
        def __init__(self, gpu_index):
            pass

        def start(self):
            loops.append(0)

        def stop(self):
            return script.pop(0)

    calls = []
    monkeypatch.setattr(bench, "ClockSampler", FakeSampler)
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    ms, info = bench.timed_steps(_FakeTorch, "cpu", None, lambda: calls.append(1), _Flush(),
                                 steps=4, world=1, gpu_index=0)
    return ms, info, len(loops), len(calls)


def test_timed_steps_keeps_a_clean_run(monkeypatch):
    good = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    ms, info, loops, calls = _run_timed(monkeypatch, [dict(good)])
    assert loops == 1 and calls == 4 and len(ms) == 4 and all(m == 1.0 for m in ms)
    assert "remeasured_after" not in info


def test_timed_steps_remeasures_once_after_a_throttled_run(monkeypatch):
    good = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    bad = dict(good, reasons=["hw_thermal_slowdown"])
    ms, info, loops, calls = _run_timed(monkeypatch, [bad, dict(good)])
    assert loops == 2 and calls == 8 and len(ms) == 4
    assert info["remeasured_after"] == "hw_thermal_slowdown"
    # a second bad record is reported as it is, not retried again
    ms, info, loops, calls = _run_timed(monkeypatch, [bad, dict(bad)])
    assert loops == 2 and info["reasons"] == ["hw_thermal_slowdown"]
    assert info["remeasured_after"] == "hw_thermal_slowdown"


def test_other_configs_are_the_other_large_forward_workloads():
    # The bench line's other_configs: the two large forward workloads besides
    # the default one, each with a committed DRAM traffic record for the
    # kernel source as it is now.
    from attention_forward_online_gb300.inputs import BENCH_WORKLOAD, WORKLOADS

    assert len(bench.OTHER_CONFIGS) == 2 and BENCH_WORKLOAD not in bench.OTHER_CONFIGS
    big = sorted((w.flops, n) for n, w in WORKLOADS.items() if w.dtype == "bf16")[-3:]
    assert {n for _, n in big} == set(bench.OTHER_CONFIGS) | {BENCH_WORKLOAD}
    for name in (BENCH_WORKLOAD,) + tuple(bench.OTHER_CONFIGS):
        assert bench.committed_traffic(name) is not None, name


def test_other_configs_default_only_with_the_default_workload(monkeypatch):
    seen = {}
    monkeypatch.setattr(bench, "run_ours", lambda args, w: seen.setdefault("args", args) and 0)
    bench.main(["--steps", "3"])
    assert seen["args"].other_configs is True
    seen.clear()
    bench.main(["--steps", "3", "--workload", "bf16_b8_h40_n2048_d128"])
    assert seen["args"].other_configs is False
    seen.clear()
    bench.main(["--steps", "3", "--no-other-configs"])
    assert seen["args"].other_configs is False


def test_forward_profiles_name_the_current_kernel_source():
    # Every committed summary of the forward kernel (the three workloads, the
    # bench's launch list and the split-KV workload) names the kernel source
    # hash bench.py reports, so a kernel change cannot leave them silently
    # describing another build.
    import glob
    import os

    sha = bench.kernel_source_hash()
    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "fwd_bf16_kernel__*.md")))
    paths += [os.path.join(bench.ROOT, "profiles", "launches__bench_default.md"),
              os.path.join(bench.ROOT, "profiles", "splitkv__bf16_b1_h8_q512_kv65536_d128.md")]
    assert len(paths) == 5
    for p in paths:
        with open(p) as f:
            assert f"`{sha}`" in f.read(), os.path.basename(p)
