"""Host-side logic of bench.py that needs no GPU: the clock record taken during
the timed region, and the rule that a committed DRAM-traffic figure only
counts while the captured kernel's sources are unchanged."""

import os
import shutil
import tempfile

import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_median_max_and_reasons():
    fh = tempfile.NamedTemporaryFile("w", suffix=".csv", delete=False)
    fh.write("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "0, 2070, 2070, 950.3, 0x4, Not Active, Not Active, Not Active, Active\n"
             "0, 2010, 2070, 940.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "garbage line\n")
    fh.close()
    s = bench.ClockSampler(0)
    s.proc, s.file = _Done(), fh
    r = s.result()
    assert r == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                 "samples_total": 3}
    assert not os.path.exists(fh.name)


def test_clock_record_keeps_only_rows_inside_the_timed_region():
    import datetime
    base = datetime.datetime(2026, 12, 3, 5, 0, 0)

    def row(sec, mhz, cap="Not Active"):
        ts = (base + datetime.timedelta(seconds=sec)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}, {ts}\n"

    fh = tempfile.NamedTemporaryFile("w", suffix=".csv", delete=False)
    # a slow row before the region, three inside (one power-capped), one slow row after
    fh.write(row(0.0, 1200) + row(1.0, 2070) + row(1.2, 2040, "Active") + row(1.4, 2070) + row(3.0, 900))
    fh.close()
    s = bench.ClockSampler(0)
    s.proc, s.file = _Done(), fh
    s.t0 = (base + datetime.timedelta(seconds=0.9)).timestamp()
    s.t1 = (base + datetime.timedelta(seconds=1.5)).timestamp()
    r = s.result()
    assert r["samples"] == 3 and r["samples_total"] == 5
    assert r["sm_mhz"] == 2070.0 and r["reasons"] == ["sw_power_cap"]
    assert abs(r["region_s"] - 0.6) < 1e-3 and abs(r["sm_mhz_x_s"] - 2070.0 * 0.6) < 0.01


def test_clock_record_without_samples_is_none():
    s = bench.ClockSampler(0)
    assert s.result() is None      # nvidia-smi never started


def test_traffic_line_is_void_once_a_kernel_source_changes(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    csrc = root / "bit_routed_expert_router_gb300" / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "bit_routed_expert_router_gb300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("_build"))
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(root))
    base = bench.load_traffic()
    # a change outside the captured kernel's sources keeps the figure
    with open(csrc / "moe_api.cu", "a") as fh:
        fh.write("\n// unrelated\n")
    assert bench.load_traffic() == base
    # a change to one of its sources voids it
    with open(csrc / "decode_cluster.cu", "a") as fh:
        fh.write("\n// changed\n")
    assert "decode_persistent" not in bench.load_traffic()
