"""Host-side logic of bench.py, on the CPU: the ncu traffic record keyed by
the kernel source, the clock-sample parser, the roofline denominators, the
default timing arguments and the reference arm (the CPU oracle) end to end."""
import hashlib
import json
import os
import types

import numpy as np
import pytest

import bench


def _fake_tree(tmp_path, source="decode.cu", body=b"kernel v1"):
    csrc = tmp_path / "paged_kv_decode_05_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / source).write_bytes(body)
    (csrc / "common.cuh").write_bytes(b"helpers")
    (tmp_path / "profiles").mkdir()
    return csrc, _hash(body)


def _hash(*bodies):
    """The expected hash: each source's code, then common.cuh's ("helpers")."""
    text = b"".join(bench.code_only(b) + b"\n" for b in bodies) + bench.code_only(b"helpers")
    return hashlib.sha256(text).hexdigest()[:16]


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    csrc, h = _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles" / "decode_split_kernel_gqa8b.md"
    prof.write_text(f"# summary\n\ntraffic_bytes_per_launch: 12345 source_sha256: {h}\n")
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") == 12345
    # another workload has no summary
    assert bench.recorded_traffic("decode_split_kernel", "mha7b") is None
    # the kernel changed since the capture: the figure no longer counts
    (csrc / "decode.cu").write_bytes(b"kernel v2")
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") is None
    # so does a change to the shared header
    (csrc / "decode.cu").write_bytes(b"kernel v1")
    (csrc / "common.cuh").write_bytes(b"helpers v2")
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") is None


def test_traffic_record_ignores_host_code_below_the_marker(tmp_path, monkeypatch):
    """Only the device code counts: an edit below the host-code marker (an
    entry point, an argument check) keeps the ncu record current; an edit
    above it (a kernel) does not."""
    device = b"__global__ void k() {}\n"
    host = b"// ------------------------------------------------ host ---\nint f() { return 1; }\n"
    csrc, _ = _fake_tree(tmp_path, body=device + host)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = _hash(device)
    assert bench.kernel_source_hash("decode.cu") == h
    prof = tmp_path / "profiles" / "decode_split_kernel_gqa8b.md"
    prof.write_text(f"traffic_bytes_per_launch: 99 source_sha256: {h}\n")
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") == 99
    (csrc / "decode.cu").write_bytes(device + host + b"int g() { return 2; }\n")
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") == 99
    (csrc / "decode.cu").write_bytes(b"__global__ void k2() {}\n" + host)
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") is None


def test_traffic_record_ignores_comments_and_formatting(tmp_path, monkeypatch):
    """A comment or a reformatting above the marker leaves the record current;
    a change inside a string literal (e.g. inline PTX) does not."""
    device = b'__global__ void k() { asm("mov.u32 %0, 1;"); }\n'
    csrc, h = _fake_tree(tmp_path, body=device)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles" / "decode_split_kernel_gqa8b.md"
    prof.write_text(f"traffic_bytes_per_launch: 7 source_sha256: {h}\n")
    (csrc / "decode.cu").write_bytes(b"// the kernel\n/* two\n lines */\n__global__ void k()\n{\n"
                                     b'    asm("mov.u32 %0, 1;");   // one move\n}\n')
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") == 7
    (csrc / "decode.cu").write_bytes(b'__global__ void k() { asm("mov.u32 %0, 2;"); }\n')
    assert bench.recorded_traffic("decode_split_kernel", "gqa8b") is None


def test_recorded_traffic_for_the_multiquery_source(tmp_path, monkeypatch):
    _, h = _fake_tree(tmp_path, source="mq.cu", body=b"mq kernels")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles" / "mq_tc_kernel_prefill_chunk.md"
    prof.write_text(f"traffic_bytes_per_launch: 777 source_sha256: {h}\n")
    assert bench.recorded_traffic("mq_tc_kernel", "prefill_chunk", "mq.cu") == 777
    # keyed on decode.cu it does not match (and decode.cu is absent here)
    assert bench.recorded_traffic("mq_tc_kernel", "prefill_chunk") is None


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines):
    s = bench.ClockSampler("GPU-0")
    s.proc = _Proc()
    s.thread = types.SimpleNamespace(join=lambda timeout=None: None)
    s.lines = lines
    return s


def test_clock_sampler_keeps_the_timed_window_and_reasons():
    lines = [
        (0.5, "1000, 2070, 300.0, Not Active, Not Active, Not Active, Not Active"),   # before
        (1.0, "2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active"),
        (1.1, "2055, 2070, 950.0, Not Active, Not Active, Not Active, Active"),
        (1.2, "2070, 2070, 940.0, Not Active, Not Active, Not Active, Not Active"),
        (1.3, "[N/A], 2070, 940.0, Not Active, Not Active, Not Active, Not Active"),  # unparsable
        (1.4, "2070, 2070"),                                                         # short line
        (9.0, "500, 2070, 100.0, Active, Not Active, Not Active, Not Active"),         # after
    ]
    c = _sampler(lines).stop(1.0, 2.0)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]   # the hw_slowdown sample lies outside the window


def test_clock_sampler_counts_the_timed_region_inside_its_window():
    lines = [(t / 10, "2070, 2070, 900.0, Not Active, Not Active, Not Active, Not Active")
             for t in range(10, 31)]   # samples at 1.0, 1.1, ... 3.0 s
    c = _sampler(lines).stop(1.0, 3.0, timed=(2.05, 2.25))
    assert c["samples"] == 21 and c["samples_in_timed_region"] == 2
    assert c["window_s"] == 2.0 and "timed" in c["window"]


def test_parity_report():
    want = {0: np.array([[1.0, -0.5], [0.1, 0.0]]), 3: np.array([[2.0, 0.25], [0.0, 0.0]])}
    got = {b: v + 1e-3 for b, v in want.items()}
    r = bench.parity_report(got, want, int8=False)
    assert r["pass"] and r["sequences"] == 2 and r["elements"] == 8
    assert abs(r["max_abs"] - 1e-3) < 1e-12
    assert abs(r["max_rel_where_abs_o_ge_0.2"] - 1e-3 / 0.25) < 1e-9
    got[3] = want[3] + np.array([[0.0, 0.0], [0.0, 3e-3]])   # beyond 2e-3 + 1e-2 * 0
    assert not bench.parity_report(got, want, int8=False)["pass"]
    assert bench.parity_report(got, want, int8=True)["pass"]   # INT8 bound 2e-2
    got[0] = want[0] + 0.03
    assert not bench.parity_report(got, want, int8=True)["pass"]


def test_kernel_source_hash_of_the_shipped_sources():
    """The committed profile summaries carry hashes of this form."""
    for src in ("decode.cu", ("mq_split.cuh", "mq.cu"), ("mq_split.cuh",)):
        h = bench.kernel_source_hash(src)
        assert len(h) == 16 and int(h, 16) >= 0


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler("GPU-0")
    c = s.stop(0.0, 1.0)
    assert c["sm_mhz"] is None and c["reasons"] == ["nvidia-smi unavailable"]


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    assert bench.load_tensor_peak() == (bench.FALLBACK_BF16_TFLOPS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6794.8, "bf16_tflops": 1919.9}))
    assert bench.load_peaks() == (6794.8, "measured")
    assert bench.load_tensor_peak() == (1919.9, "measured")


def test_default_timing_arguments():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1
    assert a.impl != "reference" and a.config == "gqa8b"
    b = bench.parse_args(["--impl", "reference", "--steps", "5", "--warmup", "3"])
    assert b.impl == "reference" and b.steps == 5 and b.warmup == 3


@pytest.mark.parametrize("argv", [["--config", "nope"], ["--op", "nope"]])
def test_unknown_choices_are_rejected(argv):
    with pytest.raises(SystemExit):
        bench.parse_args(argv)


def test_reference_arm_line_on_the_tiny_workload(capsys, monkeypatch):
    """The reference arm (the CPU oracle) runs here and prints one JSON line
    with the contract's keys; its config names the workload with the same
    keys as the native arm's line."""
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    bench.run_reference(bench.parse_args(["--impl", "reference", "--config", "tiny",
                                          "--steps", "4", "--warmup", "3"]))
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 4 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["metric"] == bench.METRIC
    c = d["config"]
    assert c["name"] == "tiny" and c["batch"] == 4 and c["total_context_tokens"] == 310
    for key in ("workload", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
                "algorithmic_bytes_per_batch"):
        assert key in c


def test_reference_arm_other_ranks_do_no_work(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--config", "tiny",
                                          "--steps", "2", "--warmup", "3"]))
    assert capsys.readouterr().out == ""


def test_error_figures_of_the_test_helper():
    from _pkv_helpers import assert_attention_close, error_figures
    want = np.array([1.0, -0.5, 0.1, 0.0, 0.25])
    got = want + np.array([1e-3, -2e-3, 1e-3, 1e-3, 0.0])
    max_abs, max_rel = error_figures(got, want)
    assert abs(max_abs - 2e-3) < 1e-12 and abs(max_rel - 4e-3) < 1e-12   # 2e-3 / 0.5
    assert assert_attention_close(got, want, False) == (max_abs, max_rel)
    with pytest.raises(AssertionError):
        assert_attention_close(want + 3e-3, want, False)        # 3e-3 > 2e-3 + 1e-2 * 0
    assert assert_attention_close(want + 1e-2, want, True)[0] < 2e-2


def test_multiquery_kernel_rule_matches_the_library():
    """bench.py names the multi-query kernel in its roofline by a mirror of
    the library's dispatch rule; the library's planner (a test hook, no GPU)
    must pick the same kernel for every cache type, head dim, group size and
    query count."""
    from paged_kv_decode_05_gb300 import binding as B
    from paged_kv_decode_05_gb300.build import build
    build()
    dt = {"bf16": B.PKV_BF16, "f16": B.PKV_F16, "i8": B.PKV_I8}
    for kv in ("bf16", "f16", "i8"):
        for d in (64, 128):
            for g in (1, 2, 4, 8):
                desc = B.CacheDesc(64, 16, 2, d, dt[kv])
                for nq in (1, 2, 3, 5, 6, 7, 8, 9, 12, 16, 24, 25, 31, 32, 33, 64, 128):
                    q_dtype = B.PKV_BF16 if kv == "i8" else dt[kv]
                    name, rt = B.pkv_testing_multiquery_kernel(4, 2 * g, nq, desc, q_dtype)
                    assert name == bench.mq_kernel_for(kv, d, nq * g)[0], (kv, d, g, nq)
                    rows = nq * g
                    if name == "mqt_split_kernel" or name == "mqt_i8_split_kernel":
                        assert rt == 8 * -(-rows // 8) and rt <= 24
                    elif name == "mq_tc_kernel":
                        assert rt == 128
                    else:
                        assert rt in (16, 32, 64)
