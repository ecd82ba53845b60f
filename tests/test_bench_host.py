"""Host-side logic of bench.py that needs no GPU: the source sets behind the
DRAM-traffic records and the staleness rule that keeps an old record out of
the bench line."""
import json
import os
import re

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "exact_io_aware_flash_gb300", "csrc")


def _includes(name):
    with open(os.path.join(CSRC, name), encoding="utf-8") as f:
        return {os.path.basename(m) for m in re.findall(r'#include\s+"([^"]+)"', f.read())
                if os.path.exists(os.path.join(CSRC, os.path.basename(m)))}


def test_kernel_sources_cover_every_included_header():
    for kernel in bench.KERNEL_FILES:
        srcs = bench.kernel_sources(kernel)
        assert srcs[0] == bench.KERNEL_FILES[kernel]
        # closed under the package's own #include lines
        for name in srcs:
            assert _includes(name) <= set(srcs), (kernel, name)
        assert "fa_internal.h" in srcs and "ptx.cuh" in srcs
    assert {"dkdv_body.cuh", "bwd_common.cuh"} <= set(bench.kernel_sources("fa_bwd_dq_kernel"))


def test_recorded_traffic_is_null_once_a_source_changes(tmp_path, monkeypatch):
    kernel = "fa_fwd_kernel"
    rec = {"dram_bytes_per_launch_full_workload": 123.0,
           "sources_digest": bench.kernel_sources_digest(kernel)}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / f"{kernel}_dram.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic(kernel) == 123.0
    rec["sources_digest"] = "0" * 16
    (tmp_path / "profiles" / f"{kernel}_dram.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic(kernel) is None
    assert bench.recorded_traffic_sum(("fa_fwd_kernel", "fa_bwd_dq_kernel")) is None
