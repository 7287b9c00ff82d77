"""Host logic of the benchmark and the binding, on the CPU: the clock summary
that decides whether a timed run is kept, the lookup of recorded ncu traffic
(valid only for the source it was taken on), and the binding's refusal of CPU
memory the GPU cannot address."""
import json
import os
import shutil
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _bench():
    import bench
    return bench


def test_clock_summary_reports_throttle_reasons(tmp_path):
    bench = _bench()
    p = tmp_path / "clocks.csv"
    rows = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1201.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1390.0, 0x8, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    p.write_text("\n".join(rows) + "\n")
    cs = bench.ClockSampler(out_path=str(p))
    cs.proc = object()  # samples were taken
    s = cs.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples(tmp_path):
    bench = _bench()
    cs = bench.ClockSampler(out_path=str(tmp_path / "none.csv"))
    assert cs.summary()["reasons"] == ["nvidia-smi unavailable"]
    p = tmp_path / "empty.csv"
    p.write_text("")
    cs = bench.ClockSampler(out_path=str(p))
    cs.proc = object()
    assert cs.summary()["reasons"] == ["no samples"]


def test_traffic_record_only_for_its_source(tmp_path, monkeypatch):
    """The recorded DRAM traffic is reported only while the kernel's source is
    the one it was measured on."""
    bench = _bench()
    src_rel = os.path.join("semantic_paged_kv_head_gb300", "csrc", "ice_select.cu")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "semantic_paged_kv_head_gb300" / "csrc").mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, src_rel), tmp_path / src_rel)
    import hashlib
    sha = hashlib.sha256((tmp_path / src_rel).read_bytes()).hexdigest()[:16]
    rec = {"select_kernel<fused>": {"source_sha": sha, "dram_bytes_per_launch_full": 12345,
                                    "workload": "llama8b_36k", "units": 256}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic_for("select_kernel<fused>", "ice_select.cu", "llama8b_36k", 256) == 12345
    assert bench._traffic_for("attn_kernel", "ice_select.cu", "llama8b_36k", 256) is None
    # another workload or another launch size: the record does not describe it
    assert bench._traffic_for("select_kernel<fused>", "ice_select.cu", "qwen3_4b_250k", 256) is None
    assert bench._traffic_for("select_kernel<fused>", "ice_select.cu", "llama8b_36k", 16) is None
    with open(tmp_path / src_rel, "a") as f:
        f.write("\n// changed\n")
    assert bench._traffic_for("select_kernel<fused>", "ice_select.cu", "llama8b_36k", 256) is None


def test_fused_kernel_follows_the_documented_cluster_rule():
    bench = _bench()
    # launches of up to 76 units run the cluster kernel, larger ones one block per unit
    assert bench.fused_kernel_of(8, 2)[0] == bench.CLUSTER_KERNEL
    assert bench.fused_kernel_of(76, 2)[0] == bench.CLUSTER_KERNEL
    assert bench.fused_kernel_of(77, 2)[0] == bench.FUSED_KERNEL
    assert bench.fused_kernel_of(256, 2)[0] == bench.FUSED_KERNEL
    assert bench.fused_kernel_of(8, 2, cluster_size=1)[0] == bench.FUSED_KERNEL
    assert bench.fused_kernel_of(256, 2, cluster_size=2)[0] == bench.CLUSTER_KERNEL
    assert bench.fused_kernel_of(60, 4)[0] == bench.FUSED_KERNEL  # 2 blocks < 4 composites


def test_binding_refuses_unpinned_cpu_memory():
    from semantic_paged_kv_head_gb300 import ice
    t = torch.zeros(16, 128, dtype=torch.bfloat16)
    assert not t.is_pinned()
    with pytest.raises(ValueError, match="page-locked"):
        ice._dev_ptr(t, torch.bfloat16, "q")
    with pytest.raises(ValueError):
        ice._dev_ptr(t, torch.bfloat16, "keys", host_ok=False)
    with pytest.raises(ValueError):
        ice._dev_ptr([1, 2, 3], None, "q")


def test_unknown_extra_is_refused_before_any_work():
    """A misspelt --extras name stops the benchmark while parsing its arguments (exit 2,
    the names it accepts in the message), before any device work."""
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--extras", "host_kv,recal"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2
    assert "recal" in r.stderr and "per_layer_serial" in r.stderr
