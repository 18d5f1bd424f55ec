"""Host-side pieces of bench.py that need no GPU: the oracle timed on every
host core (threads over row blocks), the CPU-baseline fields, the clock
sampler's time windows and the page-placement probe of the end-to-end leg."""
import numpy as np
import pytest

import bench
from memory_bound_normalization_rmsnorm_gb300 import workloads as wl


def _small():
    return wl.like(wl.WORKLOADS["rms_256x1024"], 96, 512)


def test_oracle_threads_covers_every_row():
    w = _small()
    dt, nbytes, passes = bench.oracle_threads(w, 96, 4, 0.0)
    f, b = bench.algo_bytes(96, 512, w.mode, 1)
    assert dt > 0 and passes == 1 and nbytes == f + b
    # more threads than rows: one row per block, still one pass
    dt, nbytes, passes = bench.oracle_threads(w, 3, 8, 0.0)
    assert passes == 1 and nbytes == sum(bench.algo_bytes(3, 512, w.mode, 1))


def test_cpu_baseline_reports_all_cores_and_one():
    cb = bench.cpu_baseline(_small(), seconds=0.2, threaded_seconds=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == bench.host_cores()
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0


def test_clock_window_selects_by_time():
    s = bench.ClockSampler(0)
    row = ["0", "{}", "2070", "{}", "0x0", "Not Active", "Not Active", "Not Active",
           "{}", "2026/12/03 05:00:{:02d}.000"]

    def r(mhz, watts, sec, cap="Not Active"):
        out = list(row)
        out[1], out[3], out[8], out[9] = str(mhz), str(watts), cap, row[9].format(sec)
        return out

    s.rows = [r(1500, 100, 1), r(2070, 900, 5), r(1900, 950, 6, "Active"), r(1400, 90, 20)]
    t = bench.ClockSampler._epoch("2026/12/03 05:00:04.500")
    win = s.window(t, t + 2.0)
    assert win["samples"] == 2 and win["reasons"] == ["sw_power_cap"]
    assert win["sm_mhz"] in (1900.0, 2070.0, 1985.0)
    assert s.window(t + 100, t + 200) is None


def test_pages_by_node_is_safe():
    a = np.ones(1 << 20, dtype=np.uint8)
    got = bench.pages_by_node(a.ctypes.data)
    assert got is None or all(isinstance(k, int) and v >= 0 for k, v in got.items())
    assert bench.pages_by_node(8) is None


def test_plan_str():
    p = {"cluster": 1, "threads_per_row": 128, "chunks_per_thread": 4, "groups": 4,
         "rows_per_group": 1, "stages": 7, "grid": 152, "long_rows": 0, "param_smem_bytes": 0}
    assert bench.plan_str(p) == "C1 tpr128 K4 G4 rpg1 S7 grid152"
    assert bench.plan_str(None) is None


@pytest.mark.parametrize("flag", ["--no-sweep", "--no-cold", "--ablate"])
def test_new_flags_parse(flag, monkeypatch):
    seen = {}
    monkeypatch.setattr(bench, "run_ours", lambda a: seen.setdefault("ours", a))
    monkeypatch.setattr(bench, "run_ablate", lambda a: seen.setdefault("ablate", a))
    monkeypatch.setattr("sys.argv", ["bench.py", flag])
    bench.main()
    assert seen
