"""The bench's byte accounting without a GPU.  The roofline figures divide
these bytes by kernel time, so each count is checked against the per-token
and per-call bytes worked out by hand from the tensors a call reads and
writes once:

  per token  2*tp*H (partials) + 8H (streams in) + 8H (streams out)
             + 2H (layer input) + 16 + 64 (post, comb in) + 16 + 64 (out)
             MoE: tp*K*2H (routed rows) + tp*2H (shared) + tp*K*4 (indices)
                  + K*4 (weights) in place of the partials
             MXFP8: + H (values) + H/32 (scales)
  per call   384H (FP32 prenorm weight) + 2H (norm weight) + 12 + 96
             (scale, base); MXFP8 adds the scales of the padding rows.
"""
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("name,m,per_token,total", [
    # GLM-style, H = 6144, tp = 4
    ("glm", 256, 159_904, 256 * 159_904 + 384 * 6144 + 2 * 6144 + 108),
    # decode, H = 5120, tp = 8
    ("decode", 64, 174_240, 64 * 174_240 + 384 * 5120 + 2 * 5120 + 108),
    # MoE finalize, H = 5120, tp = 8, K = 8
    ("moe", 256, 829_888, 256 * 829_888 + 384 * 5120 + 2 * 5120 + 108),
    # large, H = 6144, tp = 8, MXFP8; 4096 tokens are 32 full 128-row tiles
    ("large_mxfp8", 4096, 215_392, 4096 * 215_392 + 384 * 6144 + 2 * 6144 + 108),
])
def test_call_bytes_match_the_hand_count(name, m, per_token, total):
    w = bench.workload(name, m)
    b = bench.call_bytes(w)
    assert b["total"] == total
    assert b["stage"] + b["finish"] + b["mixes"] == b["total"]
    # one token more costs exactly the per-token bytes (no padding row here)
    w1 = bench.workload(name, m + 128 if w.mxfp8 else m + 1)
    step = 128 if w.mxfp8 else 1
    assert bench.call_bytes(w1)["total"] - b["total"] == step * per_token


def test_headline_call_is_884_6_megabytes():
    assert bench.call_bytes(bench.workload("large_mxfp8", None))["total"] == 884_617_324


def test_mxfp8_padding_rows_add_only_their_scales():
    # 4095 tokens: one padding row, whose H/32 scale bytes are still written
    w, w1 = bench.workload("large_mxfp8", 4096), bench.workload("large_mxfp8", 4095)
    d = bench.call_bytes(w)["total"] - bench.call_bytes(w1)["total"]
    assert d == 215_392 - 6144 // 32


def test_weight_bytes_follow_its_type():
    # the BF16 weight [24][4H] is half the FP32 one
    f32 = bench.call_bytes(bench.workload("glm", 256))["stage"]
    bf16 = bench.call_bytes(bench.workload("glm_bf16fn", 256))["stage"]
    assert f32 - bf16 == 4 * 6144 * 24 * 2


def test_consumer_and_owner_reduce_bytes():
    H, tp, m = 6144, 8, 4096
    direct = bench.call_bytes(bench.workload("large_mxfp8", m))
    consumer = bench.call_bytes(bench.workload("consume", m))
    # no weight, no mixes, no MXFP8: pre [m][4] read instead of post/comb written
    assert consumer["total"] == m * (2 * tp * H + 18 * H + 16 + 64 + 16) + 2 * H
    residual_only = bench.call_bytes(bench.workload("residual_only", m))
    assert residual_only["total"] == m * (2 * tp * H + 16 * H + 80)
    owner = bench.call_bytes(bench.workload("owner_reduce", m))
    # the owners' sums: written once, read back once
    assert owner["total"] - direct["total"] == m * 4 * H


def test_traffic_is_read_only_for_the_same_workload_and_source(tmp_path, monkeypatch):
    import hashlib
    csrc = tmp_path / "mhc_residual_boundary_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k_stage_tc.cu").write_bytes(b"// kernel source\n")
    sha = hashlib.sha256(b"// kernel source\n").hexdigest()[:12]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k_stage_tc_large.md").write_text(
        f"traffic: workload=large_mxfp8 tokens=4096 kernel=k_stage_tc source_sha={sha} bytes_per_launch=123\n"
        f"traffic: workload=glm tokens=256 kernel=k_stage_tc source_sha=000000000000 bytes_per_launch=456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic(bench.workload("large_mxfp8", 4096)) == 123
    assert bench.kernel_traffic(bench.workload("large_mxfp8", 2048)) is None     # other size
    assert bench.kernel_traffic(bench.workload("glm", 256)) is None              # other source
    (csrc / "k_stage_tc.cu").write_bytes(b"// kernel source, edited\n")
    assert bench.kernel_traffic(bench.workload("large_mxfp8", 4096)) is None     # stale capture


def test_cpu_baseline_leg_times_the_oracle():
    from mhc_residual_boundary_gb300 import synth
    w = bench.workload("tiny", None)
    cpu = bench.cpu_baseline(w, synth.inputs_for(w))
    assert cpu["kind"] == "oracle" and cpu["unit"] == "tokens/s" and cpu["cores"] >= 1
    assert cpu["value"] > 0 and cpu["single_thread_value"] > 0
    assert f"all {w.m} tokens" in cpu["sample"]
