"""SM -> die map (die locality, "7 · AMD et le monokernel" §7.4).  CPU: the two-group split
it relies on, against cases whose answer is fixed by construction.  GPU: the probe covers
every SM once, its round trips are positive, and the split is the two-means split of
those times."""
import ctypes

import numpy as np
import pytest


@pytest.fixture(scope="module")
def mk():
    import __graft_entry__
    __graft_entry__.build()
    import persistent_sm_decode_megakernel_gb300 as m
    return m


def _groups(mk, x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = np.zeros(len(x), dtype=np.int32)
    t = ctypes.c_float()
    st = mk.mk_two_groups(x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), len(x),
                          g.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), ctypes.byref(t))
    return st, g, t.value


def test_two_groups_separates_two_clusters(mk):
    rng = np.random.default_rng(7)
    near = 1000 + rng.normal(0, 15, 76)
    far = 1400 + rng.normal(0, 15, 76)
    x = np.concatenate([near, far])
    perm = rng.permutation(len(x))
    st, g, t = _groups(mk, x[perm])
    assert st == mk.MK_OK
    want = (perm >= 76).astype(np.int32)
    np.testing.assert_array_equal(g, want)
    assert 1100 < t < 1300


def test_two_groups_degenerate_cases(mk):
    st, g, _ = _groups(mk, [5.0, 5.0, 5.0])
    assert st == mk.MK_OK and not g.any()
    st, g, t = _groups(mk, [1.0, 3.0])
    assert st == mk.MK_OK and list(g) == [0, 1] and t == pytest.approx(2.0)
    st, _, _ = _groups(mk, [1.0])
    assert st == mk.MK_ERR_INVALID


def test_die_map_rejects_bad_arguments_before_any_device_call(mk):
    die = (ctypes.c_int * 8)()
    n = ctypes.c_int()
    assert mk.mk_die_map(3, 8, die, None, ctypes.byref(n)) == mk.MK_ERR_INVALID   # reps < 4
    assert mk.mk_die_map(16, 8, None, None, ctypes.byref(n)) == mk.MK_ERR_INVALID  # no output array
    st, _, _ = _groups(mk, [])
    assert st == mk.MK_ERR_INVALID


@pytest.mark.gpu
def test_die_map_covers_every_sm(mk):
    import torch
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    die = (ctypes.c_int * 1024)()
    rtt = (ctypes.c_float * 1024)()
    n = ctypes.c_int()
    st = mk.mk_die_map(16, 1024, die, rtt, ctypes.byref(n))
    assert st == mk.MK_OK, mk.mk_last_error()
    assert n.value == n_sm
    d = np.array(die[:1024])
    r = np.array(rtt[:1024])
    used = d >= 0
    assert used.sum() == n_sm
    assert set(np.unique(d[used])) <= {0, 1}
    assert (r[used] >= 0).all() and (r[used] > 0).sum() == n_sm - 1
    # the split is the two-means split of the measured times (reference SM at the minimum)
    x = r[used].copy()
    x[x == 0] = x[x > 0].min()
    _, g, _ = _groups(mk, x)
    np.testing.assert_array_equal(g, d[used])


def test_line_latency_arguments_checked_on_host():
    import ctypes
    import numpy as np
    import persistent_sm_decode_megakernel_gb300 as mk
    la = (ctypes.c_float * 2)()
    lb = (ctypes.c_float * 2)()
    for offs in ([0, 4096], [0, 1 << 20]):   # the second lies outside the 64 KB buffer
        o = np.array(offs, dtype=np.int64)
        st = mk.mk_line_latency(1 << 16, o.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), 2, 0, 1, 1, la, lb)
        assert st == mk.MK_ERR_INVALID   # reps < 2, then an offset out of range: nothing launched
    o = np.array([0, 2], dtype=np.int64)  # not 4-byte aligned
    st = mk.mk_line_latency(1 << 16, o.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), 2, 0, 1, 8, la, lb)
    assert st == mk.MK_ERR_INVALID


@pytest.mark.gpu
def test_line_latency_from_both_dies():
    """Every sampled line has a finite L2 latency from an SM of each group, and the lines
    split into ones nearer to the first SM and ones nearer to the second (the address ->
    die interleave)."""
    import ctypes
    import numpy as np
    import __graft_entry__
    __graft_entry__.build()
    import persistent_sm_decode_megakernel_gb300 as mk
    n_max = 512
    die = (ctypes.c_int * n_max)()
    nsm = ctypes.c_int()
    assert mk.mk_die_map(6, n_max, die, None, ctypes.byref(nsm)) == mk.MK_OK, mk.mk_last_error()
    groups = [[i for i in range(nsm.value) if die[i] == g] for g in (0, 1)]
    assert groups[0] and groups[1]
    offs = np.arange(0, 1 << 20, 256, dtype=np.int64)
    la = (ctypes.c_float * len(offs))()
    lb = (ctypes.c_float * len(offs))()
    st = mk.mk_line_latency(1 << 20, offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(offs), groups[0][1],
                            groups[1][1], 8, la, lb)
    assert st == mk.MK_OK, mk.mk_last_error()
    a, b = np.array(la[:]), np.array(lb[:])
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b)), "a probe SM measured nothing"
    assert a.min() > 50 and b.min() > 50, f"latencies {a.min()}, {b.min()} cycles"
    d = a - b
    assert 0.1 < np.mean(d < 0) < 0.9, f"share of lines nearer the first SM {np.mean(d < 0):.3f}"
