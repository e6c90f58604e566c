"""Host-side pieces of bench.py (CPU only): the DRAM-traffic lookup, the algorithmic work per
launch and the JSON contract's fixed parts."""
import bench


def _table(tmp_path, rows):
    p = tmp_path / "traffic.md"
    lines = ["| roofline kernel | workload | capture | DRAM bytes | source hash |", "|---|---|---|---|---|"]
    lines += [f"| `{k}` | {w} | cap.md | {b} | {h} |" for k, w, b, h in rows]
    p.write_text("\n".join(lines) + "\n")
    return str(p)


def test_traffic_needs_same_workload_and_sources(tmp_path):
    gemm = bench.src_sha(*bench.KERNEL_SOURCES["prefill_gate_up_gemm"])
    dec = bench.src_sha(*bench.KERNEL_SOURCES["decode_layer"])
    path = _table(tmp_path, [
        ("prefill_gate_up_gemm", "T=4096 bias=none", 111, gemm),
        ("prefill_down_gemm", "T=4096 bias=none", 222, "0000000000000000"),  # stale sources
        ("decode_layer", "decode", 333, dec),
        ("not_a_kernel", "decode", 444, dec),
    ])
    assert bench.measured_traffic(4096, "none", path) == {"prefill_gate_up_gemm": 111, "decode_layer": 333}
    # another prefill size or router bias keeps only the decode row
    assert bench.measured_traffic(512, "none", path) == {"decode_layer": 333}
    assert bench.measured_traffic(4096, "zipf", path) == {"decode_layer": 333}
    assert bench.measured_traffic(4096, "none", str(tmp_path / "missing.md")) == {}


def test_committed_traffic_table_parses():
    """Every row of the committed table is well formed (matched or stale, never silently skipped
    for its format)."""
    import os
    import re
    text = open(os.path.join(bench.ROOT, "profiles", "dram_traffic.md")).read()
    rows = [ln for ln in text.splitlines() if ln.startswith("| `")]
    assert rows
    for ln in rows:
        assert re.match(r"\| `(\w+)` \| ([^|]+?) \| [^|]+ \| (\d+) \| ([0-9a-f]{16}) \|", ln), ln


def test_algorithmic_work_per_launch():
    """Counts of the scope table: decode reads the router plus k+1 experts of 1,769,472 B and x, y;
    the expert GEMMs count real rows only."""
    w = bench.algorithmic_work(d=2048, E=256, k=8, inter=512, T=4096)
    assert w["decode_layer"]["bytes"] == 256 * 2048 * 2 + 9 * 1769472 + 2 * 2048 * 2
    rows = 4096 * 8 + 4096
    assert w["prefill_gate_up_gemm"]["flop"] == 2.0 * rows * 2 * 512 * 2048
    assert w["prefill_down_gemm"]["flop"] == 2.0 * rows * 2048 * 512
    assert w["prefill_router_gemm"]["flop"] == 2.0 * 4096 * 256 * 2048
    eb = bench.expert_bytes(2048, 512)
    assert eb["gate_up"] + eb["down"] == 1769472


def test_device_info_never_raises():
    """The device record is informational: without a usable GPU it reports the error instead of
    failing the run."""
    import torch
    info = bench.device_info(torch.device("cuda", 0))
    if torch.cuda.is_available():
        assert {"name", "sms", "cc", "hbm_gib"} <= set(info)
    else:
        assert set(info) == {"error"}
