"""Host-side tests of the polymerizer (no GPU): the pages' worked example, the
cost formula's wave arithmetic, and the structural invariants of every plan."""
import ctypes
import json
import os

import numpy as np
import pytest

import micro_polymerization_gb300 as mp
from micro_polymerization_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "case_study_4096_1024_4096.json")


def a100_handle(Ta, Tb):
    """H and micro-kernels of the case study: 108 SMs, 864 warps per wave;
    GEMM-A (256,128,32) with 8 warps, GEMM-B (64,64,64) with 4 warps.  Ta and
    Tb are the pipeline-task times at K = 4096 (f_num = 128 and 64)."""
    hw = mp.MpHw(num_pe=108, warps_per_wave=864, local_mem_bytes=164 * 1024,
                 shared_mem_bytes=40 * 2 ** 20, hbm_gbs=0.0, l2_gbs=0.0, mma_tflops=0.0)
    ka = mp.MpKernelDesc(um=256, un=128, uk=32, warps=8, swap=0, fixed_us=0.0, per_step_us=Ta / 128)
    kb = mp.MpKernelDesc(um=64, un=64, uk=64, warps=4, swap=0, fixed_us=0.0, per_step_us=Tb / 64)
    return mp.mp_init_host(hw, [ka, kb])


def test_case_study_wave_arithmetic():
    gold = json.load(open(GOLDEN))
    M, N, K = gold["shape"]
    Ta, Tb = 10.0, 3.0
    h = a100_handle(Ta, Tb)
    single = mp.mp_evaluate_plan(h, 1, M, N, K, [dict(kernel=0, m0=0, n0=0, m_ext=M, n_ext=N)])
    r = single.region[0]
    assert r.f_parallel == gold["single_A"]["tasks"]
    assert r.f_parallel * 8 == gold["single_A"]["warps"]
    assert r.f_wave == gold["single_A"]["waves"]
    assert r.f_num == 128
    assert single.cost_us == pytest.approx(2 * Ta)

    cut = gold["polymerized"]["cut_rows"]
    poly = mp.mp_evaluate_plan(h, 1, M, N, K, [dict(kernel=0, m0=0, n0=0, m_ext=cut, n_ext=N),
                                               dict(kernel=1, m0=cut, n0=0, m_ext=M - cut, n_ext=N)])
    ra, rb = poly.region[0], poly.region[1]
    assert ra.f_parallel == gold["polymerized"]["region_A"]["tasks"]
    assert rb.f_parallel == gold["polymerized"]["region_B"]["tasks"]
    assert ra.f_parallel * 8 == gold["polymerized"]["region_A"]["warps"]
    assert rb.f_parallel * 4 == gold["polymerized"]["region_B"]["warps"]
    assert ra.f_parallel * 8 + rb.f_parallel * 4 == gold["polymerized"]["total_warps"]
    assert (ra.f_wave, rb.f_wave) == (1, 2)
    assert ra.f_wave + rb.f_wave == gold["polymerized"]["total_waves"]
    assert poly.cost_us == pytest.approx(Ta + 2 * Tb)
    # The page's conclusion: polymerization wins exactly when Ta > 2 Tb.
    assert (poly.cost_us < single.cost_us) == (Ta > 2 * Tb)
    h.close()


@pytest.mark.parametrize("Ta,Tb", [(10.0, 3.0), (10.0, 6.0), (10.0, 4.99), (10.0, 5.01), (8.0, 1.0)])
def test_search_is_never_worse_than_the_pages_strategies(Ta, Tb):
    h = a100_handle(Ta, Tb)
    p = mp.mp_plan(h, 4096, 1024, 4096)
    assert p.cost_us <= min(2 * Ta, Ta + 2 * Tb) + 1e-9
    assert p.evaluated >= 2
    h.close()


def test_split_k_factor_and_f_num():
    """K~ = K / splits: f_num = ceil(K~ / uk) and no split is empty."""
    h = a100_handle(10.0, 3.0)
    for K, splits in [(4096, 3), (100, 7), (64, 64), (65, 2)]:
        p = mp.mp_evaluate_plan(h, 1, 256, 128, K, [dict(kernel=0, m0=0, n0=0, m_ext=256, n_ext=128,
                                                         splits=splits)])
        r = p.region[0]
        kb = -(-K // 32)
        assert r.f_num == -(-kb // splits) or r.splits < splits
        assert (r.splits - 1) * r.f_num < kb <= r.splits * r.f_num
        assert r.f_parallel == r.splits
    h.close()


def gb300_handle():
    hw = mp.MpHw(num_pe=148, warps_per_wave=148 * 6, local_mem_bytes=232448,
                 shared_mem_bytes=126 * 2 ** 20, hbm_gbs=6684.0, l2_gbs=20000.0, mma_tflops=1974.0)
    return mp.mp_init_host(hw)


def check_tiling(p, M, N):
    cover = np.zeros((M, N), dtype=np.int32) if M * N <= 4_000_000 else None
    area = 0
    for r in p.regions():
        assert r.m_ext > 0 and r.n_ext > 0 and r.m0 >= 0 and r.n0 >= 0
        assert r.m0 + r.m_ext <= M and r.n0 + r.n_ext <= N
        assert r.n0 % 8 == 0 and r.splits >= 1
        area += r.m_ext * r.n_ext
        if cover is not None:
            cover[r.m0:r.m0 + r.m_ext, r.n0:r.n0 + r.n_ext] += 1
    assert area == M * N
    if cover is not None:
        assert np.all(cover == 1)


def test_plans_tile_the_output_exactly_once():
    h = gb300_handle()
    shapes = [(g.M, g.N, g.K) for name in ("stress", "dynamic_sequence", "dynamic_resolution", "merged_qkv")
              for g in wl.workload(name)]
    shapes += [(m, n, k) for m in (1, 7, 128, 129, 4095) for n in (1, 8, 200, 3072) for k in (0, 1, 64, 4097)]
    for (M, N, K) in shapes:
        p = mp.mp_plan(h, M, N, K)
        assert p.num_regions in (1, 2)
        check_tiling(p, M, N)
        assert p.cost_us > 0
    h.close()


def test_plan_cache_returns_the_same_plan():
    h = gb300_handle()
    p1 = mp.mp_plan(h, 777, 3072, 1024)
    p2 = mp.mp_plan(h, 777, 3072, 1024)
    assert bytes(p1) == bytes(p2)
    h.close()


def test_skinny_huge_k_gets_split():
    """(105, 1024, 12544): 8 tiles of 128x128 cannot fill 148 SMs without split-K."""
    h = gb300_handle()
    p = mp.mp_plan(h, 105, 1024, 12544)
    assert sum(r.f_parallel for r in p.regions()) >= 72
    assert any(r.splits > 1 for r in p.regions())
    h.close()


def test_forced_plan_and_errors():
    h = gb300_handle()
    _, ks = mp.mp_get_hw(h)
    for k in range(len(ks)):
        mp.mp_force_plan(h, k, 3)
        if ks[k].pair:
            # CTA pairs never split K: a forced split has no valid plan.
            with pytest.raises(mp.MPError):
                mp.mp_plan(h, 300, 500, 700)
            mp.mp_force_plan(h, k, 1)
            p = mp.mp_plan(h, 300, 500, 700)
            assert p.num_regions == 1 and p.region[0].kernel == k and p.region[0].pair == 1
            continue
        p = mp.mp_plan(h, 300, 500, 700)
        assert p.num_regions == 1 and p.region[0].kernel == k and p.region[0].splits == 3
    mp.mp_force_plan(h, -1, 0)
    with pytest.raises(mp.MPError):
        mp.mp_force_plan(h, len(ks), 0)
    with pytest.raises(mp.MPError):
        mp.mp_plan(h, -1, 5, 5)
    bad = mp.MpPlanInfo()
    bad.num_regions = 2
    for i, (m0, me) in enumerate([(0, 60), (50, 50)]):  # overlapping rows
        bad.region[i].kernel, bad.region[i].m0, bad.region[i].m_ext = 0, m0, me
        bad.region[i].n0, bad.region[i].n_ext, bad.region[i].splits = 0, 64, 1
    st = mp.library().mp_evaluate_plan(h.ptr, 1, 100, 64, 64, ctypes.byref(bad))
    assert st == mp.MP_ERR_PLAN
    h.close()


def test_empty_shapes_plan_to_nothing():
    h = gb300_handle()
    for M, N in [(0, 5), (5, 0), (0, 0)]:
        p = mp.mp_plan(h, M, N, 10)
        assert p.num_regions == 0 and p.total_tasks == 0
    h.close()


def test_pair_kernels_hold_two_sms_never_split_never_mix():
    """Pair micro-kernels (a 256-row tile on a CTA pair) take two SMs' worth
    of task slots, never split K, and never share a plan with one-CTA
    kernels; a mixed plan is refused."""
    h = gb300_handle()
    hw, ks = mp.mp_get_hw(h)
    pairs = [k for k, d in enumerate(ks) if d.pair]
    singles = [k for k, d in enumerate(ks) if not d.pair]
    assert pairs and all(ks[k].warps == 2 * ks[singles[0]].warps and ks[k].um == 256 for k in pairs)
    rng = np.random.default_rng(7)
    for _ in range(300):
        M, N, K = int(rng.integers(1, 9000)), 8 * int(rng.integers(1, 1200)), int(rng.integers(1, 9000))
        p = mp.mp_plan(h, M, N, K)
        check_tiling(p, M, N)
        assert len({r.pair for r in p.regions()}) == 1, (M, N, K)
        for r in p.regions():
            if r.pair:
                assert r.splits == 1 and r.um == 256 and not r.swap
    single = next(k for k in singles if not ks[k].swap and ks[k].un == 256)
    bad = mp.MpPlanInfo()
    bad.num_regions = 2
    for i, (k, m0, me) in enumerate([(pairs[0], 0, 512), (single, 512, 512)]):
        bad.region[i].kernel, bad.region[i].m0, bad.region[i].m_ext = k, m0, me
        bad.region[i].n0, bad.region[i].n_ext, bad.region[i].splits = 0, 256, 1
    assert mp.library().mp_evaluate_plan(h.ptr, 1, 1024, 256, 256, ctypes.byref(bad)) == mp.MP_ERR_PLAN
    h.close()


def test_enumeration_covers_the_search_and_tiles_exactly():
    """mp_enumerate_plans: every candidate tiles the output once, never mixes
    pair and one-CTA kernels, comes sorted by cost, and the cheapest costs no
    more than the heuristic search's choice."""
    h = gb300_handle()
    rng = np.random.default_rng(11)
    shapes = [(4096, 1024, 4096), (105, 1024, 12544), (1984, 2304, 768), (1, 3072, 1024)]
    shapes += [(int(rng.integers(1, 6000)), 8 * int(rng.integers(1, 700)), int(rng.integers(1, 6000))) for _ in range(12)]
    for (M, N, K) in shapes:
        plans = mp.mp_enumerate_plans(h, M, N, K)
        assert plans, (M, N, K)
        costs = [p.cost_us for p in plans]
        assert costs == sorted(costs)
        for p in plans[:200] + plans[-50:]:
            check_tiling(p, M, N)
            assert len({r.pair for r in p.regions()}) == 1
            for r in p.regions():
                if r.pair:
                    assert r.splits == 1
        best = mp.mp_plan(h, M, N, K)
        assert costs[0] <= best.cost_us * 1.005 + 1e-9, (M, N, K, costs[0], best.cost_us)
        assert any(p.pattern == 1 for p in plans)
    first3 = mp.mp_enumerate_plans(h, 4096, 1024, 4096, capacity=3)
    assert len(first3) == 3
    h.close()


def test_wave_and_pipe_cost_models():
    """The ablation models of the cost-model study: WAVE minimises the total
    wave count (large micro-kernels), PIPE the total pipeline-task time (small
    ones); the default model is restored by mode 0."""
    h = gb300_handle()
    for (M, N, K) in [(4096, 1024, 4096), (1984, 2304, 768), (300, 5000, 2000)]:
        ref = mp.mp_plan(h, M, N, K)
        cands = mp.mp_enumerate_plans(h, M, N, K)
        mp.mp_set_plan_mode(h, mp.MP_PLAN_WAVE)
        pw = mp.mp_plan(h, M, N, K)
        assert pw.cost_us == sum(r.f_wave for r in pw.regions())
        assert pw.cost_us <= min(sum(r.f_wave for r in c.regions()) for c in cands)
        mp.mp_set_plan_mode(h, mp.MP_PLAN_PIPE)
        pp = mp.mp_plan(h, M, N, K)
        assert abs(pp.cost_us - sum(r.f_pipe_us for r in pp.regions())) < 1e-9
        area = lambda p: min(r.um * r.un for r in p.regions())
        assert area(pw) >= area(ref) >= area(pp) or area(pw) >= area(pp)
        mp.mp_set_plan_mode(h, mp.MP_PLAN_MIKPOLY)
        assert _key(mp.mp_plan(h, M, N, K)) == _key(ref)
    with pytest.raises(mp.MPError):
        mp.mp_set_plan_mode(h, 7)
    h.close()


def _key(p):
    return [(r.kernel, r.m0, r.n0, r.m_ext, r.n_ext, r.splits) for r in p.regions()]


def _gb300_host_handle():
    hw = mp.MpHw(num_pe=152, warps_per_wave=152 * 6, local_mem_bytes=232448, shared_mem_bytes=132644864,
                 hbm_gbs=6684.0, l2_gbs=20000.0, mma_tflops=1974.0)
    return mp.mp_init_host(hw)


def test_plan_many_equals_one_plan_per_call():
    """mp_plan_many gives, shape by shape, the plan mp_plan gives (with and
    without a plan cache), and rejects bad dimensions."""
    shapes = [(g.M, g.N, g.K) for g in wl.workload("dynamic_sequence")] + [(1, 1, 1), (105, 1024, 12544),
                                                                           (5, 7, 0)]
    h = _gb300_host_handle()
    os.environ["MP_PLAN_CACHE"] = "0"
    try:
        h0 = _gb300_host_handle()
    finally:
        del os.environ["MP_PLAN_CACHE"]
    try:
        for hh in (h, h0):
            many = mp.mp_plan_many(hh, shapes)
            for s, p in zip(shapes, many):
                one = mp.mp_plan(hh, *s)
                assert ctypes.string_at(ctypes.addressof(p), ctypes.sizeof(p)) == \
                    ctypes.string_at(ctypes.addressof(one), ctypes.sizeof(one)), s
        assert mp.mp_plan_many(h, shapes, want_plans=False) is None
        bad = (ctypes.c_int64 * 3)(4, -1, 4)
        assert mp.library().mp_plan_many(h.ptr, 1, bad, None) == mp.MP_ERR_INVALID_ARG
        assert mp.library().mp_plan_many(h.ptr, -1, bad, None) == mp.MP_ERR_INVALID_ARG
        assert mp.library().mp_plan_many(h.ptr, 0, None, None) == mp.MP_OK
    finally:
        h.close()
        h0.close()


def test_tail_is_charged_once_per_plan():
    """A micro-kernel's tail_us enters Cost(S, H) once, not once per wave:
    cost = f_wave * g_predict(f_num) + tail (one region, no HBM floor)."""
    hw = mp.MpHw(num_pe=4, warps_per_wave=16, local_mem_bytes=1 << 17, shared_mem_bytes=1 << 22,
                 hbm_gbs=0.0, l2_gbs=0.0, mma_tflops=0.0)
    k = mp.MpKernelDesc(um=64, un=64, uk=64, warps=4, swap=0, fixed_us=1.0, per_step_us=0.5, tail_us=0.0)
    h = mp.mp_init_host(hw, [k])
    try:
        M, N, K = 64 * 8, 64, 64 * 10          # 8 tasks on 4 slots: 2 waves of 10 steps
        base = mp.mp_evaluate_plan(h, 1, M, N, K, [dict(kernel=0, m0=0, n0=0, m_ext=M, n_ext=N)])
        assert base.region[0].f_wave == 2
        assert base.cost_us == pytest.approx(2 * (1.0 + 0.5 * 10))
        mp.mp_set_kernel_model(h, 0, 1.0, 0.5, 3.0)
        with_tail = mp.mp_evaluate_plan(h, 1, M, N, K, [dict(kernel=0, m0=0, n0=0, m_ext=M, n_ext=N)])
        assert with_tail.cost_us == pytest.approx(base.cost_us + 3.0)
        assert mp.mp_plan(h, M, N, K).cost_us == pytest.approx(base.cost_us + 3.0)
        with pytest.raises(mp.MPError):
            mp.mp_set_kernel_model(h, 0, 1.0, 0.5, -1.0)
    finally:
        h.close()


def _split_handle():
    """4 PEs at 1000 GB/s of L2 (250 GB/s each), one 64 x 64 micro-kernel."""
    hw = mp.MpHw(num_pe=4, warps_per_wave=16, local_mem_bytes=1 << 17, shared_mem_bytes=1 << 22,
                 hbm_gbs=0.0, l2_gbs=1000.0, mma_tflops=0.0)
    k = mp.MpKernelDesc(um=64, un=64, uk=64, warps=4, swap=0, fixed_us=1.0, per_step_us=0.5, tail_us=0.0)
    return mp.mp_init_host(hw, [k])


def test_split_model_enters_each_split_task():
    """A tile split S ways costs g_predict(f_num) + sync_us + bytes_factor *
    (4 um un bytes at one PE's share of L2) per task; a host handle has no
    clusters, so the split goes through L2 (on_chip = 0)."""
    h = _split_handle()
    try:
        M, N, K = 64, 64, 64 * 12            # one tile, 12 K steps
        region = [dict(kernel=0, m0=0, n0=0, m_ext=M, n_ext=N, splits=4)]
        d_sync, d_factor = mp.mp_get_split_model(h, 0)
        pass_us = 4.0 * 64 * 64 / (250.0 * 1e3)
        p = mp.mp_evaluate_plan(h, 1, M, N, K, region)
        r = p.region[0]
        assert (r.splits, r.f_num, r.f_parallel, r.f_wave) == (4, 3, 4, 1)
        assert p.cost_us == pytest.approx(1.0 + 0.5 * 3 + d_sync + d_factor * pass_us)
        mp.mp_set_split_model(h, 0, 7.0, 2.0)
        assert mp.mp_get_split_model(h, 0) == (7.0, 2.0)
        assert mp.mp_get_split_model(h, 1, S=2) != (7.0, 2.0)     # the on-chip terms are apart
        p2 = mp.mp_evaluate_plan(h, 1, M, N, K, region)
        assert p2.cost_us == pytest.approx(1.0 + 0.5 * 3 + 7.0 + 2.0 * pass_us)
        # An unsplit plan does not see the split terms.
        one = [dict(kernel=0, m0=0, n0=0, m_ext=M, n_ext=N)]
        assert mp.mp_evaluate_plan(h, 1, M, N, K, one).cost_us == pytest.approx(1.0 + 0.5 * 12)
        # A cheap enough reduction makes the search split; a dear one does not.
        mp.mp_set_split_model(h, 0, 0.0, 0.0)
        assert mp.mp_plan(h, M, N, K).region[0].splits > 1
        mp.mp_set_split_model(h, 0, 100.0, 0.0)
        assert mp.mp_plan(h, M, N, K).region[0].splits == 1
        for bad in [(2, 1.0, 1.0, 0), (0, -1.0, 1.0, 0), (0, 1.0, float("nan"), 0), (0, 1.0, 1.0, 4),
                    (1, 1.0, 1.0, 1), (1, 1.0, 1.0, 9)]:
            with pytest.raises(mp.MPError):
                mp.mp_set_split_model(h, *bad[:3], S=bad[3])
        for on_chip, S in [(1, 0), (0, 3), (1, 9)]:
            with pytest.raises(mp.MPError):
                mp.mp_get_split_model(h, on_chip, S)
        # On chip: one cluster size, or every size at once.
        mp.mp_set_split_model(h, 1, 1.5, 0.5)
        assert all(mp.mp_get_split_model(h, 1, S) == (1.5, 0.5) for S in range(2, 9))
        mp.mp_set_split_model(h, 1, 6.0, 3.0, S=3)
        assert mp.mp_get_split_model(h, 1, 3) == (6.0, 3.0)
        assert mp.mp_get_split_model(h, 1, 4) == (1.5, 0.5)
    finally:
        h.close()


def test_calibration_table_is_parsed(tmp_path):
    """The table's kernel lines replace g_predict and its tail, its split lines
    the reduction terms; comments and lines naming no kernel are ignored."""
    h = _split_handle()
    try:
        path = tmp_path / "table.txt"
        path.write_text("# um un uk swap fixed_us per_step_us tail_us\n"
                        "64 64 64 0 2.5 0.25 0.75   # measured\n"
                        "128 256 64 0 9.0 9.0 9.0\n"
                        "split 0 3.25 1.5\n"
                        "split 1 0.5 0.125\n"
                        "split 1 2.75 0.625 2\n"
                        "split 1 9.0 9.0 9\n"
                        "split 2 9.0 9.0\n")
        mp.mp_load_calibration(h, str(path))
        _, ks = mp.mp_get_hw(h)
        assert (ks[0].fixed_us, ks[0].per_step_us, ks[0].tail_us) == (2.5, 0.25, 0.75)
        assert mp.mp_get_split_model(h, 0) == (3.25, 1.5)
        assert mp.mp_get_split_model(h, 1, 2) == (2.75, 0.625)
        assert all(mp.mp_get_split_model(h, 1, S) == (0.5, 0.125) for S in range(3, 9))
        # The plan cache does not keep costs of the replaced model.
        assert mp.mp_plan(h, 64, 64, 64 * 4).cost_us == pytest.approx(2.5 + 0.25 * 4 + 0.75)
        with pytest.raises(mp.MPError):
            mp.mp_load_calibration(h, str(tmp_path / "missing.txt"))
    finally:
        h.close()


def test_calibration_writer_round_trips_through_the_parser(tmp_path):
    """calibrate.write_table's text (both forms, with split lines) is what
    mp_load_calibration reads back: g_predict, tail and the split terms."""
    from micro_polymerization_gb300 import calibrate as cal
    assert cal.fit_line([1, 2, 3], [5.0, 7.0, 9.0]) == pytest.approx((3.0, 2.0))
    assert cal.fit_line([1, 2, 3], [9.0, 7.0, 5.0]) == pytest.approx((7.0, 0.0))  # slope clamped at 0
    hw = mp.MpHw(num_pe=152, warps_per_wave=912, local_mem_bytes=1 << 17, shared_mem_bytes=1 << 27,
                 hbm_gbs=6800.0, l2_gbs=20000.0, mma_tflops=1890.0)
    h = mp.mp_init_host(hw)
    try:
        _, ks = mp.mp_get_hw(h)
        rows = [(d, 1.0 + i, 0.25 + 0.01 * i, 4.0 + i, 5.0 + i, 0.5 + 0.01 * i, [(4, 9.0, 12.0)], (1, 1), (2, 1))
                for i, d in enumerate(ks)]
        split = {0: (4.25, 2.5, [(128, 256, 0, 12, 4, 14.5)]), 3: (2.125, 5.5, []), 8: (2.5, 2.75, [])}
        for form in ("waves", "one-wave"):
            path = tmp_path / f"{form}.txt"
            cal.write_table(str(path), hw, rows, form, split)
            h2 = mp.mp_init_host(hw)
            try:
                mp.mp_load_calibration(h2, str(path))
                _, k2 = mp.mp_get_hw(h2)
                for i, d in enumerate(k2):
                    want = (1.0 + i, 0.25 + 0.01 * i, 4.0 + i) if form == "waves" else (5.0 + i, 0.5 + 0.01 * i, 0.0)
                    assert (d.fixed_us, d.per_step_us, d.tail_us) == pytest.approx(want, abs=1e-4)
                assert mp.mp_get_split_model(h2, 0) == pytest.approx((4.25, 2.5))
                assert mp.mp_get_split_model(h2, 1, 3) == pytest.approx((2.125, 5.5))
                assert mp.mp_get_split_model(h2, 1, 8) == pytest.approx((2.5, 2.75))
            finally:
                h2.close()
    finally:
        h.close()


def test_waves_fit_and_refit(tmp_path):
    """fit_kernel on exact lines T1 = 6 + 0.5 t, T2 - T1 = 2 + 0.25 t: a later
    wave costs 2 us plus the one-wave rate, the first the whole T1 line
    (tail 4); --refit rewrites a table from its recorded points."""
    from micro_polymerization_gb300 import calibrate as cal
    pts = [(t, 6 + 0.5 * t, (6 + 0.5 * t) + (2 + 0.25 * t)) for t in (4, 12, 24)]
    assert cal.fit_kernel(pts) == pytest.approx((2.0, 0.5, 4.0, 6.0, 0.5))
    hw = mp.MpHw(num_pe=152, warps_per_wave=912, local_mem_bytes=1 << 17, shared_mem_bytes=1 << 27,
                 hbm_gbs=6800.0, l2_gbs=20000.0, mma_tflops=1890.0)
    h = mp.mp_init_host(hw)
    try:
        _, ks = mp.mp_get_hw(h)
        rows = [(d,) + cal.fit_kernel(pts) + (pts, (128, 256), (256, 256)) for d in ks]
        src = tmp_path / "waves.txt"
        cal.write_table(str(src), hw, rows, "waves", {0: (4.0, 2.0, [(128, 256, 0, 12, 4, 14.5)])})
        dst = tmp_path / "one.txt"
        cal.refit(str(src), str(dst), "one-wave")
        mp.mp_load_calibration(h, str(dst))
        _, k1 = mp.mp_get_hw(h)
        assert all((d.fixed_us, d.per_step_us, d.tail_us) == pytest.approx((6.0, 0.5, 0.0), abs=1e-4) for d in k1)
        assert mp.mp_get_split_model(h, 0) == pytest.approx((4.0, 2.0))
        cal.refit(str(dst), str(tmp_path / "back.txt"), "waves")
        mp.mp_load_calibration(h, str(tmp_path / "back.txt"))
        _, kw = mp.mp_get_hw(h)
        assert all((d.fixed_us, d.per_step_us, d.tail_us) == pytest.approx((2.0, 0.5, 4.0), abs=1e-4) for d in kw)
    finally:
        h.close()
