"""Host-side arithmetic of bench.py's roofline objects, on CPU: the prefill flop count, the three prefill
fractions, and the gating of ncu-derived numbers by the kernel source they were captured from."""
import math
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_prefill_useful_flops_per_head_token():
    # chunk 64, d = 128: five C x d products per token (A, Qk, W, U', Qk U), three d x d (W S, Q+ S, Ktil^T U),
    # and the triangular inverse, 2 C^2 / 3 per token
    assert bench.PREFILL_FLOPS_PER_HEAD_TOKEN == pytest.approx(81920 + 98304 + 8192 / 3, rel=1e-12)


def test_prefill_roofline_fractions_are_consistent():
    ms, head_tokens, io = 1.646, 22528 * 32, 1.4995e9
    r = bench.prefill_roofline(ms, head_tokens, io, "no_such_profile")
    hbm, bf16, _, _ = bench.measured_peaks()
    flops = bench.PREFILL_FLOPS_PER_HEAD_TOKEN * head_tokens
    assert r["useful_tflops"] == pytest.approx(flops / (ms / 1000) / 1e12, rel=1e-12)
    assert r["useful_flop_frac"] == pytest.approx(r["useful_tflops"] / bf16, rel=1e-12)
    assert r["byte_frac"] == pytest.approx(io / (ms / 1000) / 1e9 / hbm, rel=1e-12)
    assert r["flop_per_byte"] == pytest.approx(flops / io, rel=1e-12)
    # at 88 flop per byte the byte roofline is the lower one, and then the attainable fraction is the byte one
    assert r["bound"] == "hbm"
    assert r["attainable_tflops"] == pytest.approx(r["flop_per_byte"] * hbm / 1000, rel=1e-12)
    assert r["attainable_frac"] == pytest.approx(r["byte_frac"], rel=1e-12)
    # without a matching capture, no ncu-derived numbers
    assert r["tensor_pipe_frac"] is None and r["traffic"] is None


def test_compute_bound_case_takes_the_tensor_peak():
    # a call with very few bytes per flop: the attainable rate is the bf16 peak
    r = bench.prefill_roofline(1.0, 1 << 20, 1e6, "no_such_profile")
    _, bf16, _, _ = bench.measured_peaks()
    assert r["bound"] == "tensor"
    assert r["attainable_tflops"] == pytest.approx(bf16)
    assert r["attainable_frac"] == pytest.approx(r["useful_flop_frac"])


@pytest.mark.parametrize("name", ["kda_decode", "kda_decode_bf16", "kda_decode_multi", "kda_prefill_varlen4",
                                  "kda_prefill_long"])
def test_profile_numbers_are_read_only_for_their_own_kernel_source(name):
    path = os.path.join(ROOT, "profiles", f"{name}_traffic.txt")
    recorded = [ln.split(":", 1)[1].strip() for ln in open(path) if ln.startswith("kernel_source_sha:")]
    assert len(recorded) == 1
    sha = recorded[0]
    kv = bench.profiled_values(name, sha)
    assert kv["kernel_source_sha"] == sha
    assert bench.profiled_values(name, "0" * 16) == {}
    if "dram_bytes_per_launch" in kv:
        assert bench.profiled_traffic(name, sha) == float(kv["dram_bytes_per_launch"])
        assert bench.profiled_traffic(name, "0" * 16) is None
    for k, v in kv.items():
        if k.startswith("tensor_pipe_frac_"):
            assert 0.0 < float(v) < 1.0
        if k.startswith("dram_bytes"):
            assert float(v) > 0 and math.isfinite(float(v))


def test_file_sha_covers_every_source_in_order():
    a = "hybrid_linear_attention_decode_gb300/csrc/kda_decode.cu"
    b = "hybrid_linear_attention_decode_gb300/csrc/kda_device.cuh"
    assert bench.file_sha(a, b) != bench.file_sha(a) != bench.file_sha(b)
    assert bench.file_sha(a, b) != bench.file_sha(b, a)
    assert len(bench.file_sha(a)) == 16
