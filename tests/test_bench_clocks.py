"""The bench's clock record: nvidia-smi rows sampled during the timed region
are reduced to median clocks, power and the set of active throttle reasons
(CPU only; the sampler process is replaced by a file of rows)."""
import tempfile
import time

import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        pass


def _sampler_with(rows):
    cs = bench.ClockSampler(0)
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    f.write("".join(rows))
    f.flush()
    cs.proc, cs.file = _Done(), f
    return cs


def _row(t, sm, power, reasons, mem):
    ts = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".250"
    flags = ", ".join("Active" if r else "Not Active" for r in reasons)
    return f"{ts}, {sm}, 2070, {power}, {flags}, {mem}, 3996\n"


def test_medians_and_reasons_inside_the_window():
    t0 = float(int(time.time()))
    rows = [_row(t0 - 5, 900, 200.0, (0, 0, 0, 0), 3996)]  # before the window: ignored
    for i, sm in enumerate((1500, 1470, 1530, 1455, 1515)):
        rows.append(_row(t0 + i, sm, 1380.0 + i, (0, 0, 0, 1), 3996 - 10 * i))
    rec = _sampler_with(rows).stop(t0 - 0.5, t0 + 5)
    assert rec["samples"] == 5
    assert rec["sm_mhz"] == 1500.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]
    assert rec["mem_mhz"] == 3976.0
    assert rec["mem_max_mhz"] == 3996.0
    assert rec["power_w"] == 1382.0


def test_thermal_reasons_are_reported():
    t0 = float(int(time.time()))
    rows = [_row(t0 + i, 1400, 1300.0, (1, 0, 1, 0), 3996) for i in range(4)]
    rec = _sampler_with(rows).stop(t0 - 0.5, t0 + 4)
    assert rec["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_no_samples_gives_no_record():
    assert _sampler_with([]).stop(0.0, 1.0) is None
