"""Host-side pieces of bench.py (no GPU): throttle-reason decoding and the
nvidia-smi clock parser, the packed one-copy input buffer, and the rule that
reports an ncu DRAM figure only for the kernel sources it was taken on."""
import json
import os

import pytest
import torch

import bench


def test_clock_reasons_decode_and_median():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.nvml, c.max_mhz = None, 2070.0
    c.samples = []
    assert c.summary()["reasons"] == ["unsampled"]
    # power cap alone, then a hardware slowdown with thermal slowdown
    c.samples = [(2070.0, 0x0), (1980.0, 0x4), (2070.0, 0x0), (1500.0, 0x8 | 0x40)]
    s = c.summary()
    assert s["sm_mhz"] == 2025.0 and s["samples"] == 4 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert s["source"] == "nvidia-smi"
    c.samples = [(2070.0, 0x1 | 0x2)]        # idle / application clocks: not throttling
    assert c.summary()["reasons"] == []


def test_nvidia_smi_lines_parse():
    text = "\n".join(["2070, 2070, 0x0000000000000000",
                      "1965, 2070, 0x0000000000000004",
                      "[N/A], 2070, 0x0",             # a line that cannot be read is skipped
                      "",
                      "2070, 2070, 0x0000000000000020"])
    samples, mx = bench.ClockSampler.parse_smi(text)
    assert samples == [(2070.0, 0), (1965.0, 4), (2070.0, 0x20)] and mx == 2070.0
    assert bench.ClockSampler.parse_smi("") == ([], None)


def test_sampler_without_nvml_or_smi_reports_unsampled(monkeypatch):
    monkeypatch.setattr(bench.shutil, "which", lambda name: None)
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.index, c.samples, c.max_mhz, c.nvml, c.smi = 0, [], None, None, None
    c.stop = bench.threading.Event()
    with c:
        pass
    assert c.summary()["reasons"] == ["unsampled"]


def test_packed_inputs_are_one_buffer_at_256_byte_offsets():
    ts = [torch.arange(7, dtype=torch.int32), torch.randn(3, 5, dtype=torch.float32),
          torch.arange(4, dtype=torch.int64).reshape(2, 2), torch.ones(1, dtype=torch.bfloat16)]
    buf, views = bench.packed(ts, "cpu")
    assert buf.dtype == torch.uint8 and buf.numel() == 4 * 256
    for t, v in zip(ts, views):
        assert torch.equal(t, v) and v.dtype == t.dtype and v.shape == t.shape
        off = v.data_ptr() - buf.data_ptr()
        assert off % 256 == 0 and off + v.numel() * v.element_size() <= buf.numel()


def test_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "attention_traffic.json")))
    entry = d["qwen_gqa_bf16"]
    fresh = entry["kernel_sha"] == bench.kernel_source_hash("decode")
    got = bench.traffic_for("qwen_gqa_bf16", "decode_tc_kernel (split-K merge fused)")
    assert got == (entry["dram_bytes_per_launch"] if fresh else None)
    # another kernel, or sources changed since the counters: no figure
    assert bench.traffic_for("qwen_gqa_bf16", "decode_simt_kernel") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda family: "0" * 16)
    assert bench.traffic_for("qwen_gqa_bf16", "decode_tc_kernel (split-K merge fused)") is None
    assert bench.traffic_for("no_such_workload", "decode_tc_kernel") is None


@pytest.mark.parametrize("family", ["decode", "prefill"])
def test_kernel_source_hash_covers_its_files(family):
    h = bench.kernel_source_hash(family)
    assert len(h) == 16 and int(h, 16) >= 0
    for n in bench.KERNEL_SOURCES[family]:
        assert os.path.exists(os.path.join(bench.ROOT, "paged_kv_cache_137_gb300", "csrc", n))


def test_every_traffic_entry_names_its_kernel_family():
    """Each committed DRAM figure says which source family it was taken on; the
    shared-prefix call (a prefill-kernel pass and the decode kernel) is the
    decode family, so a change to either kernel's sources retires the figure."""
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "attention_traffic.json")))
    for name, e in d.items():
        assert e["family"] in bench.KERNEL_SOURCES, name
        assert e["dram_bytes_per_launch"] > 0
    assert d["prefix_fork_bf16"]["family"] == "decode"
    for n in ("attention_prefill_umma.cuh", "attention_shared_prefix.cu"):
        assert n in bench.KERNEL_SOURCES["decode"]
    import workloads as W
    e = d["prefix_fork_bf16"]
    label = bench.attention_kernels("auto", W.get("prefix_fork_bf16"), 1, shared_prefix=True)
    fresh = e["kernel_sha"] == bench.kernel_source_hash("decode")
    assert bench.traffic_for("prefix_fork_bf16", label) == (e["dram_bytes_per_launch"] if fresh else None)
