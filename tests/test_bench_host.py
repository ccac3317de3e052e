"""Host-side arithmetic of bench.py on CPU: algorithmic bytes, the roofline
object, peaks per dtype, workload names and the recorded-traffic guard.  No
GPU and no GEMM: problems are described by their shapes only."""
import json
from types import SimpleNamespace

import pytest

import bench

PK = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0}


def shape(M, N, K, dtype="f16", beta=0.0, bias=False, aux=False):
    return SimpleNamespace(M=M, N=N, K=K, a_dtype=dtype, beta=beta,
                           bias=object() if bias else None, aux=object() if aux else None)


def test_algorithmic_bytes_of_the_named_workloads():
    # fp16 4096^3 with beta != 0: A, B, C, D of 32 MiB each
    assert bench.algorithmic_bytes([shape(4096, 4096, 4096, beta=0.5)]) == 4 * 32 * 2 ** 20
    # e4m3 8192^3, beta 0: A, B one byte per element, D bf16
    assert bench.algorithmic_bytes([shape(8192, 8192, 8192, "e4m3")]) == (64 + 64 + 128) * 2 ** 20
    # fp16 256 x 256 x 65536, beta 1: the HBM-bound stream-K shape
    b = bench.algorithmic_bytes([shape(256, 256, 65536, beta=1.0)])
    assert b == 2 * 256 * 65536 * 2 + 2 * 256 * 256 * 2
    # bias adds N output elements, an auxiliary tensor M x N
    assert (bench.algorithmic_bytes([shape(512, 1024, 768, bias=True)])
            - bench.algorithmic_bytes([shape(512, 1024, 768)])) == 1024 * 2
    assert (bench.algorithmic_bytes([shape(64, 128, 32, aux=True)])
            - bench.algorithmic_bytes([shape(64, 128, 32)])) == 64 * 128 * 2
    # a group or a batch is the sum of its members
    members = [shape(m, 4096, 2048, beta=1.0) for m in (64, 1000, 4096)]
    assert bench.algorithmic_bytes(members) == sum(bench.algorithmic_bytes([p]) for p in members)


def test_tensor_peak_per_dtype():
    assert bench.tensor_peak("f16", PK) == bench.tensor_peak("bf16", PK) == 2000.0
    assert bench.tensor_peak("e4m3", PK) == 4000.0
    assert bench.tensor_peak("bf16", PK, sustained=True) == 1700.0


def test_roofline_picks_the_roof_met_first():
    # ridge = 2000e12 / 8000e9 = 250 flop/byte
    big = shape(4096, 4096, 4096, beta=0.5)
    flops, ab = 2.0 * 4096 ** 3, bench.algorithmic_bytes([big])
    r = bench.roofline_entry(flops, ab, 0.1, "f16", PK, "measured", 12345)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(flops / 1e-4 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["traffic"] == 12345 and r["algorithmic_bytes"] == ab
    # decode-size GEMM: intensity ~ M, far below the ridge
    thin = shape(16, 8192, 8192, "bf16")
    flops, ab = 2.0 * 16 * 8192 * 8192, bench.algorithmic_bytes([thin])
    r = bench.roofline_entry(flops, ab, 0.05, "bf16", PK, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 8000.0
    assert r["achieved"] == pytest.approx(ab / 5e-5 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 8000.0)
    assert r["traffic"] is None
    # fp8 takes twice the bf16 peak, which also moves its ridge point up
    f8 = shape(8192, 8192, 8192, "e4m3")
    flops, ab = 2.0 * 8192 ** 3, bench.algorithmic_bytes([f8])
    r = bench.roofline_entry(flops, ab, 0.3, "e4m3", PK, "fallback", None)
    assert r["bound"] == "tensor" and r["peak"] == 4000.0 and "x2 (e4m3" in r["peak_source"]
    assert r["peak_source"].startswith("fallback")


def test_roofline_bound_switches_exactly_at_the_ridge():
    ab = 1_000_000
    below = bench.roofline_entry(249.0 * ab, ab, 1.0, "f16", PK, "measured", None)
    above = bench.roofline_entry(251.0 * ab, ab, 1.0, "f16", PK, "measured", None)
    assert below["bound"] == "hbm" and above["bound"] == "tensor"


def test_named_workloads_cover_the_five_configs():
    names = set(bench.workloads())
    assert bench.DEFAULT_WORKLOAD in names and bench.BATCHED_WORKLOAD in names
    for n in ("fp16_1024_uniform", "fp16_1024_ones", "fp16_grouped_32", "e4m3_8192",
              "fp16_bias_relu_512x1024x768", "fp16_streamk_256x256x65536",
              "fp16_streamk_1536x1536x16384", "fp16_streamk_3000x5000x7000"):
        assert n in names, n
    for layer in ("qkv", "o_proj", "gate_up", "down"):
        for m in (16, 128, 1024, 4096, 8192):
            assert "bf16_llama70b_%s_m%d" % (layer, m) in names


def test_custom_workload_names_parse():
    (p,) = bench.custom_workload("custom_bf16_72x136x40_b0.5_tanh_bias_acol")
    assert (p.M, p.N, p.K, p.beta, p.act) == (72, 136, 40, 0.5, "tanh")
    assert p.a_dtype == "bf16" and p.a_col_major and not p.b_col_major
    assert p.bias is not None and tuple(p.bias.shape) == (136,)
    assert tuple(p.A.shape) == (40, 72) and tuple(p.B.shape) == (40, 136)  # A stored K x M
    (q,) = bench.custom_workload("custom_f16_8x16x32_relu_bcol")
    assert q.relu and q.act == "relu" and q.beta == 0.0 and q.b_col_major and q.bias is None


def test_recorded_traffic_needs_the_same_kernel_sources(tmp_path, monkeypatch):
    real = bench.kernel_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"w": {"dram_bytes_per_launch": 777, "kernel_hash": real}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda: real)
    assert bench.recorded_traffic("w") == 777
    assert bench.recorded_traffic("other") is None
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("w") is None


def test_committed_traffic_entries_are_well_formed():
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for name, e in d.items():
        assert name in bench.workloads() or name.startswith("custom_"), name
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"]
        assert len(e["kernel_hash"]) == 16


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    src = 'x = 1; // one\n/* block\n comment */ asm("max.NaN.f32 %0, %1; // kept");\n'
    assert bench.code_only(src) == 'x = 1; asm("max.NaN.f32 %0, %1; // kept");'
    assert bench.code_only("a  /* c */b\n\n'/'") == "a b '/'"
    import shutil
    csrc = tmp_path / "dense_gemm_15_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        shutil.copy(bench.os.path.join(bench.ROOT, "dense_gemm_15_gb300", "csrc", f), csrc / f)
    real = bench.kernel_hash()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_hash() == real
    k = csrc / "gemm_kernel.cuh"
    k.write_text("// a new comment line\n" + k.read_text(encoding="utf-8"), encoding="utf-8")
    assert bench.kernel_hash() == real
    k.write_text(k.read_text(encoding="utf-8") + "\nint one_more_line;\n", encoding="utf-8")
    assert bench.kernel_hash() != real


def test_block_scaled_peaks_and_bytes():
    """fp4 against 6 x the bf16 peak (the nominal 13.5 / 2.25 PFLOP/s ratio),
    fp8 against 2 x; fp4 operands are half a byte, and each scale block adds a
    byte per row of A and per column of B."""
    assert bench.tensor_peak("e2m1", PK) == 12000.0 and bench.tensor_peak("e5m2", PK) == 4000.0
    p = shape(8192, 8192, 8192, "e2m1")
    p.block_scales = (None, None, "e4m3", 16)
    assert bench.algorithmic_bytes([p]) == 2 * 8192 * 4096 + 8192 * 8192 * 2 + 2 * 8192 * 512


@pytest.mark.parametrize("name", ["custom_f16_96x264x128_b0.5_relu_bias",
                                  "custom_bf16_40x136x192_bcol_acol"])
def test_cpu_sample_is_a_block_of_the_full_result(name):
    """The CPU baseline's sample (rows 0..r, columns 0..c of D) computes exactly
    that block of the full problem: the column views of B, C and the bias line
    up with the rows the oracle is asked for."""
    import numpy as np
    import oracle
    from dense_gemm_15_gb300 import inputs as I
    p = bench.get_workload(name)[0]
    full = oracle.gemm(I.bits(p.A), p.a_dtype, I.bits(p.B), p.b_dtype,
                       I.bits(p.C) if p.C is not None and p.beta != 0.0 else None, p.c_dtype,
                       alpha=p.alpha, beta=p.beta, act=p.act,
                       bias=I.bits(p.bias) if p.bias is not None else None,
                       bias_dtype=p.d_dtype, a_col_major=p.a_col_major,
                       b_col_major=p.b_col_major)
    rows, cols = 17, 40
    b, c, bv, scales = bench._column_sample(p, cols)
    part = oracle.gemm(I.bits(p.A), p.a_dtype, b, p.b_dtype, c, p.c_dtype, alpha=p.alpha,
                       beta=p.beta, act=p.act, bias=bv, bias_dtype=p.d_dtype,
                       a_col_major=p.a_col_major, b_col_major=p.b_col_major, rows=(0, rows),
                       scales=scales)
    assert np.array_equal(part, full[:rows, :cols])


def test_cpu_sample_grows_to_its_budget():
    r = bench.cpu_oracle_sample(bench.get_workload("custom_f16_64x4096x256")[0:1], budget_s=0.2)
    flops_s, cores, desc, secs, rows, cols = r
    assert flops_s > 0 and cores >= 1 and 1 <= rows <= 64 and 1 <= cols <= 4096
    assert ("rows 0..%d x columns 0..%d" % (rows, cols)) in desc
