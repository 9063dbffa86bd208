"""bench.py's host-side bookkeeping (no GPU): the source hashes that key the
DRAM traffic records, the record lookup, and the fallback peaks."""
import os
import shutil
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def fake_root(tmp_path):
    """A copy of the CUDA sources and the traffic records under tmp_path."""
    src = os.path.join(bench.ROOT, "dense_tensor_decomposition_gb300", "csrc")
    dst = tmp_path / "dense_tensor_decomposition_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o", "*.so"))
    (tmp_path / "profiles").mkdir()
    return tmp_path, dst


def test_main_kernel_hash_ignores_the_other_kernels(tmp_path, monkeypatch):
    root, csrc = fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    main = bench.MAIN_KERNEL_SOURCES["tc"]
    h_main, h_all = bench.kernel_source_hash(main), bench.kernel_source_hash()
    assert h_main != h_all
    with open(csrc / "rotations.cu", "a") as f:          # another kernel changes
        f.write("\n// edit\n")
    assert bench.kernel_source_hash(main) == h_main
    assert bench.kernel_source_hash() != h_all
    with open(csrc / "tc.cu", "a") as f:                 # the main kernel changes
        f.write("\n// edit\n")
    assert bench.kernel_source_hash(main) != h_main


def test_recorded_traffic_lookup(tmp_path, monkeypatch):
    root, _ = fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    (root / "profiles" / "dram_traffic.txt").write_text(
        "# comment line\n"
        "workload=w1 path=tc src=aaaa bytes_per_launch=100 capture=x.md (note)\n"
        "workload=w1 path=simt src=aaaa bytes_per_launch=200 capture=y.md\n"
        "workload=w2 path=tc src=bbbb bytes_per_launch=300 capture=z.md\n")
    assert bench.recorded_traffic("w1", "tc", "aaaa") == 100.0
    assert bench.recorded_traffic("w1", "simt", "aaaa") == 200.0
    assert bench.recorded_traffic("w1", "tc", "bbbb") is None      # other sources: no figure
    assert bench.recorded_traffic("w3", "tc", "aaaa") is None


def test_peaks_fall_back_when_unmeasured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.measured_peaks()
    assert src == "fallback" and peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0


def test_ttm_roofline_picks_the_slower_limit():
    import bench
    peaks = {"fp16x2": 659.3, "f32": 71.0}
    # 512^3 square products: flops dominate (tensor-bound line in TFLOP/s)
    n = 512 ** 3
    flops = [2.0 * 512 * n] * 3
    nbytes = [4.0 * (2 * n + 512 * 512)] * 3
    r = bench.ttm_roofline(flops, nbytes, ["fp16x2"] * 3, peaks, 6780.7, 1.4)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - sum(flops) / 1.4e-3 / 1e12) < 1e-2
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    t_f = flops[0] / 659.3e12
    assert abs(r["t_roof_ms"] - 3 * t_f * 1e3) < 1e-3
    # 128^4 with J = 128: bytes dominate (HBM-bound line in GB/s)
    n = 128 ** 4
    flops = [2.0 * 128 * n] * 4
    nbytes = [4.0 * (2 * n + 128 * 128)] * 4
    r = bench.ttm_roofline(flops, nbytes, ["fp16x2"] * 4, peaks, 6780.7, 2.2)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6780.7
    assert abs(r["achieved"] - sum(nbytes) / 2.2e-3 / 1e9) < 0.1
    assert abs(r["t_roof_ms"] - sum(nbytes) / 6780.7e9 * 1e3) < 1e-3
    assert abs(r["frac_of_t_roof"] - r["t_roof_ms"] / 2.2) < 1e-3
    # the CUDA-core kernel on every mode
    r = bench.ttm_roofline([1e9], [1e3], ["f32"], peaks, 6780.7, 1.0)
    assert r["bound"] == "alu"
