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
