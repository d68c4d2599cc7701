"""GPU parity of the int4 kernel's per-group accumulator form (opt-in with
LGT_GEMM_INT4_V2=1; used for at most 16 activation rows, group 128, splits
of whole groups, K-contiguous activation): codes expanded as 1024 + q /
64 + q without their scale, one TMEM accumulator per group, scaled in fp32
by the epilogue warps, and the term sum over g of s(n, g) (z(n, g) Ag[g][m]
+ Og[g][m]) taken off once per tile.  Same tolerances as the other int4
tests, against the fp64 oracle."""
import os

import numpy as np
import pytest

import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full, oracle_sample, run_case

pytestmark = pytest.mark.gpu

K = wl.K_CONTIG


def _case(M, N, Kd, split=1, zero=8.0):
    nm = f"int4groups_m{M}_n{N}_k{Kd}_s{split}_z{zero}"
    return wl.GemmCase(nm, M, N, Kd, K, K, wl.F16, wl.INT4, wl.F16, ("normal", 1.0), ("bytes",), split_k=split,
                       group_size=128, zero_value=zero)


@pytest.fixture(autouse=True)
def _groups_form():
    lib()
    old = os.environ.get("LGT_GEMM_INT4_V2")
    os.environ["LGT_GEMM_INT4_V2"] = "1"
    yield
    if old is None:
        del os.environ["LGT_GEMM_INT4_V2"]
    else:
        os.environ["LGT_GEMM_INT4_V2"] = old


@pytest.mark.parametrize("M", [1, 9, 16])
@pytest.mark.parametrize("N,Kd,split", [(256, 1024, 1), (300, 2048, 2), (640, 4096, 4), (384, 8192, 0)])
@pytest.mark.parametrize("zero", [8.0, None])
def test_groups_form_matches_oracle(M, N, Kd, split, zero):
    case = _case(M, N, Kd, split, zero)
    inp = wl.make_inputs(case, seed=M * 7 + N)
    c, g, _ = run_case(case, inp, reps=2)
    assert g.info.kernel == 1 and g.info.tile_m == 16
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


def test_groups_form_deterministic_split():
    m = lib()
    case = _case(16, 1024, 8192, split=8)
    inp = wl.make_inputs(case, seed=5)
    import helpers
    d = helpers.desc_for(m, case, 148)
    d.flags = m.GEMM_FLAG_DETERMINISTIC
    g = m.Gemm(d)
    c1, _, _ = run_case(case, inp, gemm=g)
    c2, _, _ = run_case(case, inp, gemm=g)
    assert np.array_equal(c1, c2)
    assert_close(c1, oracle_full(case, inp), case.name)
    g.close()


def test_groups_form_full_size_sampled():
    case = wl.INT4_DEQUANT
    inp = wl.make_inputs(case, seed=1)
    c, g, _ = run_case(case, inp, reps=2)
    rows, cols = wl.sample_indices(case.M, case.N, 1500, seed=3)
    assert_close(c[rows, cols], oracle_sample(case, inp, rows, cols), case.name)
    assert np.all(np.isfinite(c))
    g.close()
