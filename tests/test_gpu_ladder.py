"""Build ladder of "8 · Écrire son megakernel", §8.6, steps 1-4, on the GPU through the
C ABI (mk_selftest): a persistent kernel terminates; two-opcode dispatch keeps queue
order; counters order dependent instructions across CTAs with no deadlock; the page
pool streams many more TMA pages than it holds without corruption or leak.  Plus the
grid-barrier latency microbenchmark of "7 · AMD et le monokernel", §7.3."""
import ctypes

import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mk():
    import __graft_entry__
    __graft_entry__.build()
    import persistent_sm_decode_megakernel_gb300 as m
    return m


def _selftest(mk, kind):
    res = (ctypes.c_int64 * 8)()
    st = mk.mk_selftest(kind, res, 8)
    assert st == mk.MK_OK, mk.mk_last_error()
    return list(res)


def test_step1_persistent_kernel_terminates(mk):
    r = _selftest(mk, 1)
    assert r[0] == 1 and r[2] == 0 and r[1] >= 1


def test_step2_dispatch_keeps_order(mk):
    r = _selftest(mk, 2)
    assert r[0] == 1, r


def test_step3_counters_chain_and_fan_in(mk):
    r = _selftest(mk, 3)
    assert r[0] == 1, r
    assert r[3] == 7 + r[1]       # value passed through every CTA, then gathered


def test_step4_page_pool_no_corruption_no_leak(mk):
    r = _selftest(mk, 4)
    assert r[0] == 1 and r[3] == 0 and r[2] == 0, r


@pytest.mark.parametrize("mode", [0, 1])
def test_grid_barrier_latency(mk, mode):
    us = ctypes.c_double()
    st = mk.mk_barrier_bench(mode, 200, ctypes.byref(us))
    assert st == mk.MK_OK, mk.mk_last_error()
    assert 0.0 < us.value < 100.0
