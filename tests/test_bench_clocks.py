"""The benchmark's clock record, on CPU: the samples nvidia-smi prints are
parsed by field name, only those whose timestamps fall inside the timed
region count (the sampler starts before it), throttle reasons are read from
the same samples, and a run with no sample inside the region says so.  The
nvidia-smi process is replaced by a fake that prints fixed lines."""

import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _stamp(t: float) -> str:
    return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]


class _FakeSmi:
    def __init__(self, lines):
        self.out = "\n".join(lines)

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, None


def _line(t, sm, power, cap=False, thermal=False):
    # the order of ClockSampler.FIELDS
    return ", ".join([_stamp(t), str(sm), "2070", str(power), "3996", "0x0", "Not Active",
                      "Active" if thermal else "Not Active", "Not Active", "Active" if cap else "Not Active"])


def _sampler(lines):
    c = bench.ClockSampler(0)
    c.proc = _FakeSmi(lines)
    return c


def test_only_samples_inside_the_timed_region_count():
    t0 = 1_800_000_000.0
    # idle samples (low clock, low power, a thermal flag) before the region, loaded ones inside it
    lines = [_line(t0 + 0.1 * i, 1200, 90, thermal=True) for i in range(3)]
    lines += [_line(t0 + 0.3 + 0.1 * i, 2070, 950, cap=(i == 2)) for i in range(5)]
    rec = _sampler(lines).stop(t0 + 0.25, t0 + 0.75)
    assert rec["window"] == "timed region"
    assert rec["samples"] == 5
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["power_w"] == 950.0 and rec["mem_mhz"] == 3996.0
    assert rec["reasons"] == ["sw_power_cap"], "a reason seen only outside the region does not count"


def test_no_sample_inside_the_region_falls_back_and_says_so():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.1 * i, 2070, 900) for i in range(4)]
    rec = _sampler(lines).stop(t0 + 10.0, t0 + 11.0)
    assert rec["samples"] == 4
    assert rec["window"].startswith("whole sampler run")


def test_malformed_lines_are_skipped():
    t0 = 1_800_000_000.0
    lines = ["garbage", _line(t0 + 0.5, "[N/A]", 900), _line(t0 + 0.6, 2000, "[N/A]")]
    rec = _sampler(lines).stop(t0, t0 + 1.0)
    assert rec["samples"] == 1
    assert rec["sm_mhz"] == 2000.0 and rec["power_w"] is None
