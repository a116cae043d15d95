"""Host-side accounting of the benchmark (CPU): the algorithmic bytes the roofline divides by, the
step's workload, and the rule that a recorded DRAM-traffic figure only counts for the source it was
measured on."""
import json

import bench


def test_linear_bytes_by_hand():
    # lm_head at M = 1: 128256 x 4096 packed nibbles, fp16 scale per 128 weights, bf16 x and y
    N, K = 128256, 4096
    assert bench.linear_bytes(1, N, K) == N * K // 2 + N * 32 * 2 + 4096 * 2 + N * 2 == 271_141_376
    # M only adds activation and output bytes
    assert bench.linear_bytes(4, N, K) - bench.linear_bytes(1, N, K) == 3 * (K * 2 + N * 2)


def test_verify_bytes_by_hand():
    B, g, V = 1, 3, 128256
    assert bench.verify_bytes(B, g, V, False) == 4 * V * 2                  # every target row once
    assert bench.verify_bytes(B, g, V, True) == 7 * V * 2 + 2 * V * 2       # target + draft rows, one row pair again


def test_step_workload():
    sb = bench.step_bytes()
    assert [n for n, _, _ in bench.LAYERS] == ["q", "k", "v", "o", "gate", "up", "down", "lm_head"]
    # every member of a group appears once, and the members of a group share K
    assert sorted(m for _, ms in bench.GROUPS for m in ms) == sorted(n for n, _, _ in bench.LAYERS)
    assert all(len({bench.SHAPE[m][1] for m in ms}) == 1 for _, ms in bench.GROUPS)
    # a grouped launch reads its input once: q, k, v and gate, up save 2 and 1 activation reads
    shared = lambda M: (2 + 1) * M * 4096 * 2
    assert sb["w4a4"] == bench.GAMMA * (sum(bench.linear_bytes(1, N, K) for _, N, K in bench.LAYERS) - shared(1))
    assert sb["w4a16"] == sum(bench.linear_bytes(bench.GAMMA + 1, N, K) for _, N, K in bench.LAYERS) - shared(4)
    assert sb["total"] == sb["w4a4"] + sb["w4a16"] + sb["verify"]
    assert 1.5e9 < sb["total"] < 1.6e9          # larger than L2 (129 MB): no flush needed between steps


def test_traffic_counts_only_for_the_measured_source(tmp_path, monkeypatch):
    fam = "linear_w4a4"
    good = {fam: {"dram_bytes_per_launch": 123, "source_sha256": bench.source_hash(bench.KERNEL_SOURCES[fam])}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(good))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda files: good[fam]["source_sha256"])  # sources as measured
    assert bench.kernel_traffic(fam) == 123
    monkeypatch.setattr(bench, "source_hash", lambda files: "0" * 64)   # the kernel source changed
    assert bench.kernel_traffic(fam) is None
    assert bench.kernel_traffic("verify_greedy") is None                 # no record at all


def test_committed_traffic_matches_current_sources():
    for fam in bench.KERNEL_SOURCES:
        assert bench.kernel_traffic(fam) is not None, f"{fam}: traffic recorded on another source"
