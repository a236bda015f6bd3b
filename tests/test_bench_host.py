"""Host-side logic of bench.py (no GPU): the guard that drops a stored DRAM-traffic
figure once the kernel sources change, and the JSON line of the reference arm."""
import argparse
import os

import bench


def _fake_root(tmp_path, kernel_src: str, stored_hash: str):
    csrc = tmp_path / "tensor_train_compressed_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(kernel_src)
    (csrc / "host.cpp").write_text("host code is not part of the hash\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# kernel workload bytes_per_launch sources_hash\n"
        f"k_bwd_mma train 65063680 {stored_hash}\n")
    return str(tmp_path)


def test_stored_traffic_is_dropped_when_kernels_change(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, "__global__ void k() {}\n", "0" * 16))
    current = bench.kernel_sources_hash()
    # a figure taken on other sources is not reported
    assert bench.stored_traffic("k_bwd_mma", "train") is None
    # the same figure stamped with the current sources' hash is
    p = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    with open(p, "a") as f:
        f.write(f"k_bwd_mma train 12345 {current}\n")
    assert bench.stored_traffic("k_bwd_mma", "train") == 12345
    assert bench.stored_traffic("k_fwd_mma", "train") is None
    # a change to a kernel source changes the hash; a host-only C++ file does not count
    with open(os.path.join(bench.ROOT, "tensor_train_compressed_gb300", "csrc", "host.cpp"),
              "a") as f:
        f.write("// edited\n")
    assert bench.kernel_sources_hash() == current
    with open(os.path.join(bench.ROOT, "tensor_train_compressed_gb300", "csrc", "k.cu"), "a") as f:
        f.write("// edited\n")
    assert bench.kernel_sources_hash() != current
    assert bench.stored_traffic("k_bwd_mma", "train") is None


def test_committed_traffic_figures_name_a_sources_hash():
    p = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                     "dram_traffic.txt")
    rows = [l.split() for l in open(p) if l.strip() and not l.startswith("#")]
    assert rows and all(len(r) == 4 and len(r[3]) == 16 and int(r[2]) > 0 for r in rows)


def test_reference_arm_json_line():
    args = argparse.Namespace(gpus=1, steps=1, warmup=0)
    line = bench.run_reference(args)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "lookups/s" and line["higher_is_better"]
    assert line["dtype"] == "f64" and line["steps"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "lookups/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
