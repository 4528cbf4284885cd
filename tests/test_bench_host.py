"""Host-side logic of bench.py that needs no GPU: the FLOP and byte counts the
reported rates divide by, the choice between the two end-to-end modes, and the
lookup of per-launch DRAM traffic in the committed ncu summaries."""
import hashlib
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_attn_flops_convention():
    # 4*B*H*N^2*d forward, 2.5x backward, halved for causal (the reported convention)
    f, b = bench.attn_flops(1, 32, 8192, 128, True)
    assert abs(f / 1e9 - 549.76) < 0.01 and abs(b / f - 2.5) < 1e-12
    f, b = bench.attn_flops(2, 16, 4096, 128, False)
    assert abs(f / 1e9 - 274.88) < 0.01 and abs(b / 1e9 - 687.19) < 0.01
    f, _ = bench.attn_flops(8, 16, 1024, 64, True)
    assert abs(f / 1e9 - 17.18) < 0.01


@pytest.mark.parametrize("N,W", [(1, 1), (5, 1), (7, 3), (16, 16), (33, 8), (40, 100)])
def test_attn_flops_window_counts_exact_pairs(N, W):
    pairs = sum(1 for i in range(N) for j in range(N) if i - W < j <= i)
    f, _ = bench.attn_flops(1, 1, N, 1, True, window=W)
    if W < N:
        assert f == 4.0 * pairs
    else:                                   # a window of N or more is plain causal
        assert f == bench.attn_flops(1, 1, N, 1, True)[0]


def test_decode_bytes_counts_rows_in_use():
    lens, H, Hkv, d = [3, 0, 5], 8, 2, 64
    kv = sum(lens) * Hkv * d * 2 * 2           # K and V rows, 16-bit
    qol = len(lens) * H * (d * 2 + d * 2 + 4)  # q read, O written, L written
    assert bench.decode_bytes(lens, H, Hkv, d) == kv + qol
    assert bench.decode_bytes(lens, H, Hkv, d, elem=1) == kv // 2 + qol


def test_e2e_pick_takes_the_faster_mode():
    ms, note, other = bench.e2e_pick(1.5, 4.0)
    assert ms == 1.5 and note == bench.E2E_NOTE and other == ("sequential", 4.0)
    ms, note, other = bench.e2e_pick(5.0, 4.0)
    assert ms == 4.0 and note == bench.E2E_SEQ_NOTE and other == ("pipelined", 5.0)


def test_traffic_lookup_follows_the_source(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("// kernel\n")
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "k_kernel__w.txt").write_text(
        f"source: k.cu\nsource_sha256: {sha}\ndram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "k_kernel", "k.cu")
    assert bench.traffic_from_profiles("k_kernel", "w") == 123456.0
    assert bench.traffic_from_profiles("k_kernel", "other") is None   # no capture
    src.write_text("// kernel, changed since the capture\n")
    assert bench.traffic_from_profiles("k_kernel", "w") is None


def test_committed_profiles_have_the_fields_the_bench_reads():
    names = [n for n in os.listdir(os.path.join(ROOT, "profiles")) if n.endswith(".txt")]
    assert names
    for n in names:
        kernel, workload = n[:-4].split("__")
        assert kernel in bench.KERNEL_SOURCES, n
        text = open(os.path.join(ROOT, "profiles", n)).read()
        src = re.search(r"^source:\s*(\S+)", text, re.M)
        assert src and src.group(1) == bench.kernel_source(kernel, workload), n
        assert re.search(r"source_sha256:\s*[0-9a-f]{64}", text), n
        assert re.search(r"dram_bytes_per_launch:\s*[0-9]+", text), n
        assert "--clock-control none" in text, n


def test_emit_prints_one_line_and_writes_it_with_json_out(tmp_path, capsys):
    out = {"metric": "m", "value": 1.5, "unit": "TFLOP/s"}
    bench.emit(out, bench.parse([]))
    lines = capsys.readouterr().out.splitlines()
    assert len(lines) == 1 and lines[0].startswith("{")
    path = tmp_path / "sub" / "line.json"
    bench.emit(out, bench.parse(["--json-out", str(path)]))
    printed = capsys.readouterr().out.strip()
    assert path.read_text().strip() == printed


def test_memory_report_matches_the_pages_sizes():
    # one head at 8K fp16: the 128 MiB score matrix the docs page prints (Fig. 2 and the
    # hero panel), against Q, K, V, O and L of that head
    r = bench.memory_report([8192], 1, 128, 2, 280 << 30, 0)
    assert r["score_matrix_bytes"] == 128 << 20
    assert r["linear_footprint_bytes"] == 4 * 8192 * 128 * 2 + 4 * 8192
    assert abs(r["score_over_linear"] - (128 << 20) / (8 << 20 | 32768)) < 1e-9
    # the score matrix alone fills the device at the N where B*H*N^2*2 reaches its size
    n = r["ordinary_attention_runs_out_at_N"]
    assert n * n * 2 <= 280 << 30 < (n + 1) * (n + 1) * 2
    # packed sequences add their own squares
    r2 = bench.memory_report([100, 300], 4, 64, 2, 1 << 30, 7)
    assert r2["score_matrix_bytes"] == 4 * 2 * (100 ** 2 + 300 ** 2)
    assert r2["peak_device_bytes_step"] == 7


def test_tensor_rate_at_clock():
    # 8192 FLOP per clock per SM: 152 SMs at 1807 MHz give the nominal 2.25 PFLOP/s
    assert abs(bench.tensor_rate_at_clock(152, 1807.0) - 2250.0) < 1.0
    assert bench.tensor_rate_at_clock(152, 1807.0, bits=8) == 2 * bench.tensor_rate_at_clock(152, 1807.0)


def test_profile_record_reads_tensor_activity(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel source")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "fwd_kernel__w.txt").write_text(
        f"source_sha256: {sha}\ndram_bytes_per_launch: 1234\n"
        "tensor pipeline (sm__pipe_tensor_cycles_active, elapsed)      66.2 %\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "fwd_kernel", "k.cu")
    assert bench.profile_record("fwd_kernel", "w") == (1234.0, 66.2)
    src.write_text("changed")
    assert bench.profile_record("fwd_kernel", "w") == (None, None)


def test_kernel_source_follows_the_head_dim():
    assert bench.kernel_source("bwd_dkdv_kernel", "n8k_causal_d128_bf16").endswith("fa_bwd128.cu")
    assert bench.kernel_source("bwd_dkdv_kernel", "gpt2m_causal_d64_fp16").endswith("fa_bwd64.cu")
    assert bench.kernel_source("bwd_dq_kernel", "ragged_causal_d32_fp16").endswith("fa_bwd64.cu")
    assert bench.kernel_source("fwd_kernel", "ragged_causal_d32_fp16").endswith("fa_fwd.cu")
