"""bench.py's ncu bookkeeping on CPU: the summary it writes from an
`ncu --page raw --csv` export, and the rule that a summary taken on other
kernel sources is never reported."""
import csv
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _raw_csv(path):
    """A two-kernel export in ncu's raw layout: header row, unit row, one
    row per launch (a second launch of the same kernel must be ignored)."""
    names = ["ID", "Kernel Name", "dram__bytes_read.sum", "dram__bytes_write.sum",
             "gpu__time_duration.sum",
             "gpu__compute_memory_throughput.avg.pct_of_peak_sustained_elapsed",
             "launch__registers_per_thread"]
    units = ["", "", "Mbyte", "Kbyte", "usecond", "%", "register/thread"]
    rows = [["0", "void tp::k_brick_project<1, 1>(tp::Params, int)", "100", "2,000", "500", "55.5",
             "126"],
            ["1", "tp::k_brick_scatter_cubic<0>(tp::Params, int)", "160", "17", "900", "82", "109"],
            ["2", "void tp::k_brick_project<1, 1>(tp::Params, int)", "999", "999", "999", "1", "1"],
            ["3", "void at::vectorized_elementwise_kernel<4>()", "1", "1", "1", "1", "32"]]
    with open(path, "w", newline="") as f:
        w = csv.writer(f)
        w.writerow(names)
        w.writerow(units)
        w.writerows(rows)


def test_summary_merges_one_capture_per_kernel(tmp_path):
    """Exports of separate single-kernel captures merge into one summary."""
    a, b = tmp_path / "a.csv", tmp_path / "b.csv"
    for path, row in ((a, ["0", "void tp::k_brick_project<1, 2>(tp::Params, int)", "90", "500",
                          "560", "55", "128"]),
                      (b, ["0", "tp::k_brick_scatter_cubic<0>(tp::Params, int)", "160", "17", "900",
                          "82", "109"])):
        rows = list(csv.reader(open(_raw_csv(tmp_path / "full.csv") or tmp_path / "full.csv")))
        with open(path, "w", newline="") as f:
            w = csv.writer(f)
            w.writerows(rows[:2])
            w.writerow(row)
    d = bench.ncu_summary([str(a), str(b)], str(tmp_path / "out.json"))
    assert set(d["kernels"]) == {"project_3d_2d", "volume_grad_scatter"}
    assert d["kernels"]["project_3d_2d"]["dram_read_bytes"] == 90e6
    assert d["kernels"]["volume_grad_scatter"]["duration_ns"] == 900e3
    assert d["from"] == ["a.csv", "b.csv"]


def test_summary_scales_units_and_keeps_the_first_launch(tmp_path):
    src = tmp_path / "raw.csv"
    out = tmp_path / "ncu_traffic.json"
    _raw_csv(src)
    d = bench.ncu_summary(str(src), str(out))
    assert json.load(open(out)) == d
    assert d["source_sha"] == bench.kernel_source_sha()
    fwd = d["kernels"]["project_3d_2d"]
    assert fwd["dram_read_bytes"] == 100e6
    assert fwd["dram_write_bytes"] == 2e6                 # "2,000" Kbyte
    assert fwd["dram_bytes_per_launch"] == 102e6
    assert fwd["duration_ns"] == 500e3
    assert fwd["mem_sol_pct"] == 55.5 and fwd["registers"] == 126
    sc = d["kernels"]["volume_grad_scatter"]
    assert sc["dram_bytes_per_launch"] == 160e6 + 17e3        # writes in Kbyte


def test_stale_summary_is_not_reported(tmp_path, monkeypatch):
    """ncu_profile() returns the committed figures only while the kernel
    sources hash to the value recorded with them."""
    csrc = tmp_path / "backprojection_tp_project_gather_b300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(ROOT, "backprojection_tp_project_gather_b300", "csrc", name),
                    csrc / name)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "raw.csv"
    _raw_csv(src)
    bench.ncu_summary(str(src), str(tmp_path / "profiles" / "ncu_traffic.json"))
    assert bench.ncu_profile()["volume_grad_scatter"]["duration_ns"] == 900e3
    with open(csrc / bench.KERNEL_SOURCES[0], "a") as f:
        f.write("\n// changed\n")
    assert bench.ncu_profile() is None


def test_committed_summary_matches_the_sources():
    """The summary under profiles/ was taken on the kernels as committed."""
    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    assert d["source_sha"] == bench.kernel_source_sha()
    assert set(d["kernels"]) == set(bench.NCU_KERNELS)
