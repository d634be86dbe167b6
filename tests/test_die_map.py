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
