"""bench.py's clock record: nvidia-smi samples carry their own timestamps and only
those stamped inside the timed region count. A fake nvidia-smi on the CPU prints a
sample every 50 ms; the first ones report a hardware slowdown and must fall outside
the region marked after them."""
import os
import stat
import sys
import time

import bench

FAKE = r'''#!{python}
import sys, time
from datetime import datetime
i = 0
while True:
    now = datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    slow = "Active" if i < 3 else "Not Active"
    print(f"{{now}}, 0, {{1900 + i}}, 2070, 500.0, 0x0, {{slow}}, Not Active, Not Active, Not Active", flush=True)
    i += 1
    time.sleep(0.05)
'''


def _fake(tmp_path):
    p = tmp_path / "nvidia-smi"
    p.write_text(FAKE.format(python=sys.executable))
    p.chmod(p.stat().st_mode | stat.S_IXUSR)
    return str(p)


def test_only_samples_inside_the_region_count(tmp_path):
    with bench.ClockSampler(0, exe=_fake(tmp_path)) as clk:
        assert clk.lines, "sampling is live before the region starts"
        time.sleep(0.4)
        clk.begin()
        time.sleep(0.4)
        clk.end()
    s = clk.summary()
    assert s["samples_total"] > s["samples"] >= 4, s
    assert s["reasons"] == [], s           # the slowdown samples came before the region
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] > 1900 + 3, s       # median of in-region samples only
    assert s["period_ms"] == 50


def test_missing_tool_gives_an_empty_record(tmp_path):
    with bench.ClockSampler(0, exe=str(tmp_path / "absent")) as clk:
        clk.begin()
        clk.end()
    s = clk.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == []
