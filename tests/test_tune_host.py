"""Host logic of the launch-shape tuner (no GPU): its byte counts agree with the bench's algorithmic bytes, which
set the HBM bound above which a timing counts as L2-served, and its candidate shapes are legal."""
import memory_bound_decoder_gb300.tune as tune
import workloads as wl

KINDS = {"add_rmsnorm": "add_rmsnorm", "add_rmsnorm_quant_fp8": "add_rmsnorm_q8",
         "add_rmsnorm_quant_nvfp4": "add_rmsnorm_nvfp4", "swiglu": "swiglu", "swiglu_quant_fp8": "swiglu_q8",
         "swiglu_quant_nvfp4": "swiglu_nvfp4"}


def test_algorithmic_bytes_match_the_bench():
    for kind, wkind in KINDS.items():
        for mode in (("static", "dynamic") if kind.endswith("fp8") else (None,)):
            for T, W in ((1, 5120), (1000, 13824), (2048, 53248)):
                c = wl.Call(wkind, T, W, wl.N01, 1e-5, mode)
                assert tune.algorithmic_bytes(kind, mode, T, W) == c.algorithmic_bytes(), (kind, mode, T, W)


def test_candidates_are_legal_shapes():
    for kind, mode, width in tune.DEFAULT_SHAPES:
        nvec = width // 8
        reduces = kind.startswith("add") or (kind == "swiglu_quant_fp8" and mode == "dynamic")
        cands = tune.candidates(kind, mode, width)
        assert cands
        for c, v, th in cands:
            assert v in (1, 2, 4, 8) and 32 <= th <= 512 and th % 32 == 0
            assert not reduces or c <= 8
            slice_ = -(-nvec // c)
            if kind.endswith("nvfp4") and slice_ % 2:
                slice_ += 1
            assert th * v >= slice_


def test_rotation_covers_three_l2_sizes_where_the_launch_count_allows():
    l2 = 126 * 2 ** 20
    for T, W in ((2048, 14336), (8192, 4096), (64, 1536)):
        b = tune.algorithmic_bytes("swiglu", None, T, W)
        n = max(1, min(tune.MAX_SETS, -(-tune.ROTATE_L2 * l2 // b)))
        assert n * b >= tune.ROTATE_L2 * l2 or n == tune.MAX_SETS


def test_ranking_keeps_l2_served_timings_out_only_under_a_short_rotation():
    gbps = lambda us: 1000.0 / us          # a point of 1000 "bytes" per microsecond unit
    bound = 1.05 * 100.0                   # 1.05 x a copy rate of 100
    rules = (1, 2, 256)
    # a faster candidate above the bound: excluded when the rotation is short, kept when it is full
    timed = [((2, 2, 128), 9.0), ((4, 1, 128), 9.8)]          # 111 and 102 GB/s
    best, us, above = tune.rank(rules, 10.5, timed, gbps, bound, full_rotation=False)
    assert best == (4, 1, 128) and us == 9.8 and above == [[2, 2, 128]]
    best, us, above = tune.rank(rules, 10.5, timed, gbps, bound, full_rotation=True)
    assert best == (2, 2, 128) and us == 9.0 and above == [[2, 2, 128]]
    # the rules stand unless a candidate is faster, even when their own timing is above the bound
    best, us, above = tune.rank(rules, 9.0, [((4, 1, 128), 9.8)], gbps, bound, full_rotation=False)
    assert best == rules and us == 9.0 and above == [[1, 2, 256]]
    best, us, above = tune.rank(rules, 10.0, [], gbps, bound, full_rotation=False)
    assert best == rules and us == 10.0 and above == []
