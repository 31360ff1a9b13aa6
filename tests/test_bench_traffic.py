"""Host-side checks of the bench's traffic records (no GPU): a record applies only to
its own kernel family and only while that family's device-code sources are the ones it
was captured with."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_record_names_its_kernel_and_bytes():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert d, "no traffic records"
    for name, rec in d.items():
        assert rec["kernel"] in ("w4a16_tc_kernel", "w4a16_gemv_kernel", "w4a8_gemm_kernel"), name
        assert rec["dram_bytes_per_launch"] > 0 and rec["algorithmic_bytes_per_launch"] > 0
        ratio = rec["dram_bytes_per_launch"] / rec["algorithmic_bytes_per_launch"]
        if "decode" in name:
            # weight streaming: DRAM traffic within a few percent of the algorithmic bytes
            assert 0.9 < ratio < 1.1, name
        else:
            # compute-bound tiles re-read A from L2 misses; never more than twice the bytes
            assert 0.9 < ratio < 2.0, name
        assert "ncu" in rec["how"] and "--clock-control none" in rec["how"], name


def test_source_hash_is_per_kernel_family():
    b = _bench()
    h16 = b.kernel_source_hash("w4a16_tc_kernel")
    assert h16 == b.kernel_source_hash("w4a16_gemv_kernel")
    assert h16 != b.kernel_source_hash("w4a8_gemm_kernel")


def test_record_applies_only_to_its_kernel():
    b = _bench()
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for name, rec in d.items():
        other = "w4a8_gemm_kernel" if rec["kernel"] != "w4a8_gemm_kernel" else "w4a16_tc_kernel"
        assert b.profiled_traffic(name, other) is None
        got = b.profiled_traffic(name, rec["kernel"])
        matches = rec["kernel_source_hash"] == b.kernel_source_hash(rec["kernel"])
        assert (got == rec["dram_bytes_per_launch"]) if matches else (got is None)
