"""The tile scheduler on the host (no GPU): the stream-K partition that the
tensor-core kernels walk, built and checked by gemm_f32_schedule_check with
the kernels' own work-list code. Every k-block of every unit tile must be
computed exactly once, split tiles must have their parts in k order, and
partial-sum slots must never be shared, at every size, cluster count and
launch kind."""

import itertools

import pytest

KINDS = ["exact_pair", "tf32_pair", "exact_lsu", "tf32_lsu"]


@pytest.mark.parametrize("kind", KINDS)
def test_partition_is_exact_cover(gemm_lib, kind):
    ms = [1, 100, 256, 257, 1000, 2048, 4096, 8192, 12345]
    ns = [1, 128, 300, 1531, 4096, 11008]
    ks = [1, 31, 32, 777, 2048, 4096, 16384]
    workers = [76, 75, 64, 37, 2, 1]
    for m, n, k, w in itertools.product(ms, ns, ks, workers):
        st, stats = gemm_lib.gemm_f32_schedule_check(m, n, k, w, kind)
        assert st == gemm_lib.OK, f"{kind} {m}x{n}x{k} on {w}: check {st}"
        assert stats["clusters"] <= max(w, 1)
        assert stats["max_parts"] <= 8


def test_benchmark_workloads_schedule(gemm_lib):
    # 4096^3 on 76 CTA pairs: 256 unit tiles of 256 x 256, three waves dealt
    # whole, the last 28 tiles split over every pair
    st, s = gemm_lib.gemm_f32_schedule_check(4096, 4096, 4096, 76, "exact_pair")
    assert st == gemm_lib.OK
    assert (s["tiles"], s["k_blocks"], s["whole_tiles"], s["splits"]) == (256, 128, 228, 1)
    assert s["clusters"] == 76
    # 2048^3: 64 tiles on 76 pairs, short enough to be dealt whole
    st, s = gemm_lib.gemm_f32_schedule_check(2048, 2048, 2048, 76, "exact_pair")
    assert st == gemm_lib.OK
    assert (s["tiles"], s["whole_tiles"], s["splits"], s["clusters"]) == (64, 64, 0, 64)
    # 8192 x 11008 x 4096: 32 x 43 tiles, 18 whole waves and 8 tiles split
    st, s = gemm_lib.gemm_f32_schedule_check(8192, 11008, 4096, 76, "exact_pair")
    assert st == gemm_lib.OK
    assert (s["tiles"], s["whole_tiles"], s["splits"]) == (1376, 1368, 1)
    # one TF32 pass at 4096^3: whole waves, the last 28 tiles in chunks of at
    # least 2048 k (two per tile)
    st, s = gemm_lib.gemm_f32_schedule_check(4096, 4096, 4096, 76, "tf32_pair")
    assert st == gemm_lib.OK
    assert (s["whole_tiles"], s["splits"], s["max_parts"]) == (228, 1, 2)
    # 512^3: 4 tiles of 16 k-blocks on 76 pairs: four pairs of one cluster
    # share each tile (k-slices of 4 k-blocks), no workspace
    st, s = gemm_lib.gemm_f32_schedule_check(512, 512, 512, 76, "exact_pair")
    assert st == gemm_lib.OK
    assert (s["tiles"], s["cluster_split"], s["splits"], s["clusters"]) == (4, 4, 0, 16)
    # 1024^3: 16 tiles of 32 k-blocks, slices of 8 in both modes
    for kind in ("exact_pair", "tf32_pair"):
        st, s = gemm_lib.gemm_f32_schedule_check(1024, 1024, 1024, 76, kind)
        assert st == gemm_lib.OK
        assert (s["tiles"], s["cluster_split"], s["clusters"]) == (16, 4, 64), kind
    # 1000 x 1531 x 777: 24 tiles, three pairs per tile on 76 pairs
    st, s = gemm_lib.gemm_f32_schedule_check(1000, 1531, 777, 76, "exact_pair")
    assert st == gemm_lib.OK
    assert (s["tiles"], s["cluster_split"], s["clusters"]) == (24, 3, 72)
    # a split must save each pair at least 128 k of 3xTF32 work or 768 k of
    # one TF32 pass: one TF32 pass at 512^3 (384 k saved at best) and
    # 512 x 512 x 128 (96 k) are not split, 512 x 512 x 256 (192 k) is
    st, s = gemm_lib.gemm_f32_schedule_check(512, 512, 512, 76, "tf32_pair")
    assert st == gemm_lib.OK and s["cluster_split"] == 1
    st, s = gemm_lib.gemm_f32_schedule_check(512, 512, 128, 76, "exact_pair")
    assert st == gemm_lib.OK and s["cluster_split"] == 1
    st, s = gemm_lib.gemm_f32_schedule_check(512, 512, 256, 76, "exact_pair")
    assert st == gemm_lib.OK and s["cluster_split"] == 4
    # 40 tiles on 76 pairs: more than half as many tiles as pairs, so the
    # stream-K schedule applies (every tile split through the workspace)
    st, s = gemm_lib.gemm_f32_schedule_check(2048, 1280, 2048, 76, "exact_pair")
    assert st == gemm_lib.OK
    assert (s["tiles"], s["cluster_split"], s["splits"], s["clusters"]) == (40, 1, 1, 76)
    # one tile with a long k range: four pairs of one cluster
    st, s = gemm_lib.gemm_f32_schedule_check(256, 128, 4096, 76, "exact_pair")
    assert st == gemm_lib.OK and s["cluster_split"] == 4
    # the plain-load kernel never splits within a cluster
    st, s = gemm_lib.gemm_f32_schedule_check(256, 128, 4096, 152, "exact_lsu")
    assert st == gemm_lib.OK
    assert s["cluster_split"] == 1 and s["splits"] == 1 and 2 <= s["max_parts"] <= 8


def test_schedule_check_rejects_bad_arguments(gemm_lib):
    bad = [(0, 1, 1, 76, 0), (1, 0, 1, 76, 0), (1, 1, 0, 76, 0), (1, 1, 1, 0, 0),
           (1, 1, 1, 5000, 0), (1, 1, 1, 76, 4), (1, 1, 1, 76, -1), (1 << 31, 1, 1, 76, 0)]
    for args in bad:
        st, _ = gemm_lib.gemm_f32_schedule_check(*args)
        assert st == gemm_lib.ERR_INVALID_ARG, args


def test_partition_random_shapes_and_worker_counts(gemm_lib):
    # seeded random sizes (log-uniform up to 2^15 per side, so at most 2^25
    # tile k-blocks, inside the check's enumeration limit) on worker counts
    # from 1 to 152, all four launch kinds
    import numpy as np

    rng = np.random.default_rng(20261202)
    for i in range(2000):
        m, n, k = (int(x) for x in np.exp2(rng.uniform(0, 15, 3)).astype(np.int64))
        w = int(rng.integers(1, 153))
        kind = KINDS[i % 4]
        st, stats = gemm_lib.gemm_f32_schedule_check(m, n, k, w, kind)
        assert st == gemm_lib.OK, f"{kind} {m}x{n}x{k} on {w}: check {st}"
        assert stats["clusters"] <= w
        assert stats["max_parts"] <= 8
