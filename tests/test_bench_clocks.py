"""The bench's clock sampler (host logic, no GPU): it waits for its first
sample before the timed region starts, stamps every sample on arrival, and
summarises only the samples taken inside the region.  A stand-in for
nvidia-smi prints one line every 10 ms, its SM clock counting up, so the
window's samples are recognisable."""
import sys
import time

import bench

FAKE = [sys.executable, "-c",
        "import sys, time\n"
        "for i in range(2000):\n"
        "    r = 'Active' if i % 7 == 3 else 'Not Active'\n"
        "    print(f'0, {1000 + i}, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, {r}', flush=True)\n"
        "    time.sleep(0.01)\n"]


def test_sampler_keeps_only_the_timed_window():
    with bench.ClockSampler("0", True, command=FAKE) as c:
        assert c.samples, "the first sample arrives before the region starts"
        time.sleep(0.1)  # samples before the region
        before = max(int(ln.split(",")[1]) for _, ln in c.samples)
        c.mark_start()
        time.sleep(0.15)
        c.mark_end()
    s = c.summary()
    assert s is not None and s["samples"] >= 5
    kept = [int(ln.split(",")[1]) for ln in c.window()]
    assert min(kept) > before, "no sample from before the region"
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] > before
    assert s["reasons"] == ["sw_power_cap"]


def test_sampler_without_a_tool_reports_nothing():
    with bench.ClockSampler("0", True, command=["/nonexistent/nvidia-smi"]) as c:
        c.mark_start()
        c.mark_end()
    assert c.summary() is None
    with bench.ClockSampler("0", False) as c:
        c.mark_start()
        c.mark_end()
    assert c.summary() is None
