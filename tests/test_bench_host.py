"""Host logic of bench.py (no GPU): the algorithmic byte counts the roofline
divides by, and the lookup of per-launch DRAM traffic in the committed ncu
summaries under profiles/."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

H, E, K = 6144, 256, 8


def test_decode_fused_tail_bytes_by_hand():
    # one token of the router-less fused tail reads its k expert rows, the
    # shared-expert row and the residual row (BF16), its k map entries (int32)
    # and its E logits (FP32); it writes k ids + k weights and two BF16 rows
    # (residual_out, normed); gamma (FP32) is read once per launch
    per_token = K * H * 2 + H * 2 + H * 2 + K * 4 + E * 4 + K * (4 + 4) + 2 * H * 2
    assert bench.bytes_tail(64, H, K, E=E, route_out=True) == 64 * per_token + H * 4 == 9_533_440


def test_finalize_bytes_by_hand():
    # the finalize reads weights (FP32) in place of logits and writes no ids
    per_token = K * H * 2 + H * 2 + H * 2 + K * 4 + K * 4 + 2 * H * 2
    assert bench.bytes_tail(2048, H, K) == 2048 * per_token + H * 4
    # R partial buffers: R more BF16 rows per token; no expert rows, no shared
    per_token = 4 * H * 2 + H * 2 + 2 * H * 2
    assert bench.bytes_tail(64, H, 0, shared=False, R=4) == 64 * per_token + H * 4


def test_router_and_route_bytes_by_hand():
    assert bench.bytes_router(64, H, E) == E * H * 2 + 64 * H * 2 + 64 * E * 4 == 3_997_696
    assert bench.bytes_route(64, E, K) == 64 * E * 4 + 64 * K * (4 + 4)


def _write_profile(root, units, dram, files, digest):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "k_case.md"), "w") as f:
        f.write("# a kernel\n\nMachine-readable:\n\n")
        f.write(f"- kernel: `k<1>`\n- workload: `case`\n- units_per_launch: `{units}`\n")
        f.write(f"- dram_bytes_per_launch: `{dram}`\n- source_files: `{' '.join(files)}`\n")
        f.write(f"- source_sha256: `{digest}`\n")


def test_ncu_traffic_scales_per_unit_and_goes_stale(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "a.cu").write_text("kernel source\n")
    (tmp_path / "b.h").write_text("header\n")
    files = ["a.cu", "b.h"]
    _write_profile(str(tmp_path), 2048, 266_143_232, files, bench.source_digest(files))
    assert bench.ncu_traffic("k_case", 4096) == pytest.approx(2 * 266_143_232)
    assert bench.ncu_traffic("k_case", 1) == pytest.approx(266_143_232 / 2048)
    assert bench.ncu_traffic("absent", 1) is None
    (tmp_path / "b.h").write_text("header, changed\n")  # a listed source changed: the counters are stale
    assert bench.ncu_traffic("k_case", 4096) is None


def test_committed_profiles_are_complete():
    # every summary names the command that made it and carries a parsable
    # machine-readable block whose listed sources exist
    pdir = os.path.join(ROOT, "profiles")
    names = sorted(n for n in os.listdir(pdir) if n.endswith(".md"))
    assert names
    for n in names:
        text = open(os.path.join(pdir, n)).read()
        assert "ncu " in text and "--clock-control none" in text, n
        if n.startswith("launches_"):
            continue  # a launch list: shares, no per-kernel counters
        info = dict(re.findall(r"^- (\w+): `([^`]*)`$", text, flags=re.M))
        for key in ("kernel", "workload", "units_per_launch", "dram_bytes_per_launch", "source_files",
                    "source_sha256"):
            assert key in info, (n, key)
        assert int(info["units_per_launch"]) > 0 and int(info["dram_bytes_per_launch"]) > 0, n
        for f in info["source_files"].split():
            assert os.path.exists(os.path.join(ROOT, f)), (n, f)
        assert re.fullmatch(r"[0-9a-f]{16}", info["source_sha256"]), n
        # the counters were taken on the sources as they are now: bench.py
        # can quote them as the roofline traffic (a stale digest reads None)
        units = int(info["units_per_launch"])
        assert bench.ncu_traffic(n[:-3], units) == pytest.approx(int(info["dram_bytes_per_launch"])), (
            n, "stale: a listed source changed after the capture")
