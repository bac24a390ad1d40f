"""The measured GB300 table is the planner's default model on the GPU."""
import os

import pytest

import micro_polymerization_gb300 as mp

TABLE = os.path.join(os.path.dirname(mp.__file__), "calib", "gb300.txt")


def _kernel_lines(path):
    out = {}
    for line in open(path):
        f = line.split("#")[0].split()
        if len(f) >= 6 and f[0] != "split":
            out[(int(f[0]), int(f[1]), int(f[3]))] = tuple(float(x) for x in f[4:7])
    return out


@pytest.mark.gpu
def test_mp_init_loads_the_shipped_table_by_default():
    assert os.path.exists(TABLE)
    want = _kernel_lines(TABLE)
    h, ha = mp.mp_init(0), mp.mp_init(0, "")
    try:
        _, ks = mp.mp_get_hw(h)
        _, ka = mp.mp_get_hw(ha)
        seen = 0
        for d, a in zip(ks, ka):
            key = (d.um, d.un, d.swap)
            if key in want:
                seen += 1
                assert (d.fixed_us, d.per_step_us, d.tail_us) == pytest.approx(want[key], abs=1e-4)
        assert seen >= 8
        # "" keeps the analytic model, which differs from the table.
        assert any(abs(d.fixed_us - a.fixed_us) > 1e-3 for d, a in zip(ks, ka))
        assert mp.mp_get_split_model(h, 0) != mp.mp_get_split_model(ha, 0)
        # A table that cannot be read leaves the analytic model.
        hm = mp.mp_init(0, os.path.join(os.path.dirname(TABLE), "no-such-table.txt"))
        try:
            _, km = mp.mp_get_hw(hm)
            assert [(k.fixed_us, k.per_step_us, k.tail_us) for k in km] == \
                [(k.fixed_us, k.per_step_us, k.tail_us) for k in ka]
        finally:
            hm.close()
    finally:
        h.close()
        ha.close()


@pytest.mark.gpu
def test_calibrate_writes_a_table_the_library_loads(tmp_path, monkeypatch):
    """calibrate.py end to end on a reduced grid (two K depths, one cluster
    size on chip, one split through L2): every micro-kernel gets a line with a
    positive rate, the split lines parse, and a handle planning with the
    table still produces valid plans."""
    from micro_polymerization_gb300 import calibrate as cal
    monkeypatch.setattr(cal, "STEPS", (4, 12))
    monkeypatch.setattr(cal, "SPLIT_STEPS", (4,))
    monkeypatch.setattr(cal, "SPLIT_ON_CHIP", (4,))
    monkeypatch.setattr(cal, "SPLIT_THROUGH_L2", (12,))
    out = tmp_path / "gb300.txt"
    assert cal.main(["--out", str(out)]) == 0
    lines = _kernel_lines(str(out))
    h = mp.mp_init(0, str(out))
    try:
        _, ks = mp.mp_get_hw(h)
        assert all((k.um, k.un, k.swap) in lines for k in ks)
        assert all(k.per_step_us > 0 and k.fixed_us >= 0 and k.tail_us >= 0 for k in ks)
        sync, factor = mp.mp_get_split_model(h, 0)
        assert sync >= 0 and factor >= 0
        for M, N, K in [(105, 1024, 12544), (2088, 2304, 768), (4096, 4096, 4096), (7, 9, 5)]:
            p = mp.mp_plan(h, M, N, K)
            assert p.num_regions >= 1 and p.cost_us > 0
    finally:
        h.close()
