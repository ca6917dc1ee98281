"""The benchmark's committed ncu records (profiles/ncu_traffic.json): each entry
names the capture summary it came from, and a record is used only for the
workload it was captured on and only while its kernel's sources are
unchanged (else the line reports traffic as null)."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORDS = os.path.join(ROOT, "profiles", "ncu_traffic.json")
SOURCES = {
    "fa_prefill_kernel<128>": bench.PREFILL_SOURCES,
    "fa_verify_split_kernel": bench.VERIFY_SOURCES,
    "fa_prefill_fp8_kernel": bench.FP8_SOURCES,
    "fa_bwd_dkdv_kernel<128>": bench.BWD_SOURCES,
    "fa_bwd_dq_kernel<128>": bench.BWD_SOURCES,
}


def _records():
    with open(RECORDS) as f:
        return json.load(f)


def test_every_record_names_its_summary_and_a_known_workload():
    from exact_tiled_attention_03_gb300.inputs import WORKLOADS

    for kernel, d in _records().items():
        assert kernel in SOURCES, kernel
        assert os.path.exists(os.path.join(ROOT, d["capture"])), d["capture"]
        assert d["workload"].split()[0] in WORKLOADS, d["workload"]
        assert d["units"] == 1 and d["dram_bytes"] > 0
        assert len(d["source_sha"]) == 16


def test_a_record_is_used_only_for_its_own_workload():
    for kernel, d in _records().items():
        other = "tiny_b1h1s256d64_causal"
        assert bench.ncu_traffic(kernel, SOURCES[kernel], other) is None
        got = bench.ncu_traffic(kernel, SOURCES[kernel], d["workload"].split()[0])
        if d["source_sha"] == bench.source_hash(SOURCES[kernel]):
            assert got == d["dram_bytes"]
        else:
            assert got is None


def test_unknown_kernel_has_no_record():
    assert bench.ncu_traffic("no_such_kernel", bench.PREFILL_SOURCES,
                             "prefill_b4h32s8192d128_causal") is None


def test_main_roofline_follows_the_kernel_fa_forward_dispatches_to():
    """Decode shapes (Sq <= 16) run on the split-KV verify kernel and are read
    against HBM; the rest run on the prefill kernel and are read against the
    bf16 tensor peak."""
    from exact_tiled_attention_03_gb300.inputs import WORKLOADS

    peaks = {"bf16_tflops": 1000.0, "bf16_tflops_sustained": 900.0, "hbm_gbs": 5000.0,
             "source": "test"}
    wv = WORKLOADS["verify_b16h32q5k4096d128"]
    r, launches = bench.main_roofline(wv, 200e-6, peaks, 4)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and launches == 2
    assert abs(r["achieved"] - wv.io_bytes() / 200e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 5000.0) < 1e-12
    assert bench.main_roofline(wv, 200e-6, peaks, 1)[1] == 1
    wp = WORKLOADS["prefill_b4h32s2048d128_causal"]
    r, launches = bench.main_roofline(wp, 1e-3, peaks, 0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and launches == 1
    assert abs(r["achieved"] - wp.exact_flops() / 1e-3 / 1e12) < 1e-9
    assert r["traffic"] is None  # the committed capture is of another workload
    wl = WORKLOADS["prefill_b1h32s32768d64_causal"]
    r, launches = bench.main_roofline(wl, 1e-3, peaks, 0)
    assert r["bound"] == "tensor" and r["kernel"] == "fa_prefill_kernel<64>" and launches == 1
    assert r["traffic"] is None  # no record for the d = 64 kernel
