"""Host-side helpers of bench.py that need no GPU."""

import hashlib

import bench


def test_traffic_lookup_only_matches_the_current_source(tmp_path, monkeypatch):
    # DRAM bytes recorded by ncu are reported only while the kernel source they
    # were taken on is unchanged: any edit to it makes the figure null
    csrc = tmp_path / "dense_fp32_gemm_major_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "tc_gemm.cu").write_bytes(b"kernel v1\n")
    (csrc / "ptx.cuh").write_bytes(b"helpers\n")
    (csrc / "simt_gemm.cu").write_bytes(b"simt\n")
    sha = hashlib.sha256(b"kernel v1\nhelpers\n").hexdigest()[:16]
    simt_sha = hashlib.sha256(b"simt\n").hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment\n\n"
        f"kernel=tc_pair_tma_3xtf32 workload=c4 mode=exact src_sha256={sha} dram_bytes_per_launch=123\n"
        f"kernel=tc_pair_tma_tf32 workload=c4 mode=tf32 src_sha256=0000000000000000 dram_bytes_per_launch=9\n"
        f"kernel=simt_gemm workload=c4 mode=exact_simt src_sha256={simt_sha} dram_bytes_per_launch=77\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_lookup("tc_pair_tma_3xtf32", "c4", "exact") == (123, sha)
    assert bench.traffic_lookup("tc_pair_tma_3xtf32", "c5b", "exact") == (None, sha)
    assert bench.traffic_lookup("tc_pair_tma_tf32", "c4", "tf32") == (None, sha)   # stale hash
    assert bench.traffic_lookup("simt_gemm", "c4", "exact_simt") == (77, simt_sha)
    (csrc / "tc_gemm.cu").write_bytes(b"kernel v2\n")
    assert bench.traffic_lookup("tc_pair_tma_3xtf32", "c4", "exact")[0] is None
