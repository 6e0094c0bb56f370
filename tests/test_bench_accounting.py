"""The benchmark's roofline accounting on the CPU: the algorithmic bytes and flops that bench.py
divides by its measured times, pinned to the per-unit counts worked out by hand from the chunk
algebra and the HBM layouts (d = 128, C = 64), and the ncu-traffic lookup that must drop a
capture once the kernel's source has changed."""
import json

import pytest

import bench

D, C = 128, 64


def test_prefill_bytes_per_token_head():
    # q, k, v in and out: 4 x 128 bf16 = 1024 B; alpha per channel fp32 = 512 B; beta fp32 = 4 B
    assert bench.prefill_bytes(1, 1, D, 0) == 1540
    assert bench.prefill_bytes(1, 1, D, 0, channel=False) == 1024 + 4 + 4   # scalar gate
    assert bench.prefill_bytes(1, 1, D, 0, linear=True) == 1024              # no gates
    assert bench.prefill_bytes(1, 1, D, 0, beta=False) == 1024 + 512         # gated linear
    # the states: S0 in and S_final out, fp32 d x d per (sequence, head)
    assert bench.prefill_bytes(0, 1, D, 1) == 2 * D * D * 4


def test_prefill_bytes_of_the_32_head_workload():
    # 1 x 32768 tokens, 32 heads: 1540 B per token-head plus one S0 and one S_final per head
    assert bench.prefill_bytes(32768, 32, D, 1) == 32768 * 32 * 1540 + 32 * 2 * D * D * 4
    assert bench.prefill_bytes(32768, 32, D, 1) == 1_619_001_344


def test_prefill_flops_per_token_head():
    # gated delta rule, 2 flops per multiply-add: W S, Q~ S, K^^T U (3 d^2), A over the strict
    # lower triangle ((C - 1) / 2 d), M with the diagonal ((C + 1) / 2 d), the solve applied to
    # [beta K~ | beta V] ((C - 1) / 2 2d), M U ((C + 1) / 2 d)
    assert bench.prefill_flops(1, 1, D) == pytest.approx(139_136)
    # linear attention: Q S and K^T V (2 d^2), the score triangle and its product with V
    assert bench.prefill_flops(1, 1, D, linear=True) == pytest.approx(82_176)
    # gated linear attention: as linear, the decay-weighted M over the same triangle
    assert bench.gated_linear_flops(1, 1, D) == pytest.approx(82_176)


def test_decode_accounting():
    # one read and one write of the fp32 state, q, k, v and out in bf16, alpha fp32, beta fp32
    assert bench.decode_bytes(1, 1, D) == 2 * D * D * 4 + 4 * D * 2 + D * 4 + 4
    assert bench.decode_bytes(1, 1, D) == 132_612
    assert bench.decode_flops(1, 1, D) == 2 * (3 * D * D + 2 * D)


def test_traffic_lookup_follows_the_source(tmp_path, monkeypatch):
    # a capture taken on the current source is returned; any other digest reads as no capture
    digest = bench.source_digest(bench.KERNEL_SOURCES["decode"])
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "decode": {"source_digest": digest, "dram_bytes_per_launch": 123},
        "prefill": {"source_digest": "0" * 16, "dram_bytes_per_launch": 456}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("decode") == 123
    assert bench.ncu_traffic("prefill") is None       # stale: taken on another source
    assert bench.ncu_traffic("linear_attn") is None   # not captured
    assert bench.ncu_traffic("no_such_kernel") is None


def test_committed_traffic_matches_current_sources():
    # every committed capture is on the current kernel sources (so the bench line reports it)
    for k in bench.KERNEL_SOURCES:
        t = bench.ncu_traffic(k)
        assert t is None or t > 0, k
