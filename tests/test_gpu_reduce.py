"""GPU parity of the fp32 row reduction (include/reduce.h) against the fp64
oracle, through the C ABI.

Bound: a result of the library's fixed summation order is within
(chain + depth) * 2^-24 * sum|x| of the exact row sum, with chain <=
ceil(cols / 4096) + 1 and depth <= ceil(cols / 4096) + 18 whatever the split
plan (a row is split into at most ceil(cols / 4096) chunks; reduce.h gives the
derivation).  Integer-valued inputs whose partial sums stay below 2^24 are
summed exactly, so those cases compare bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import helpers
    return helpers.lib()


def _bound(x_cpu, rows, cols, ldx):
    c = math.ceil(cols / 4096)
    return oracle.reduce_rows_bound(oracle.reduce_rows_abs(x_cpu, rows, cols, ldx), c + 1, c + 18)


def _run(lib, x_dev, rows, cols, ldx=0, out=None):
    r = lib.RowReduce(rows, cols)
    out = torch.full((max(rows, 1),), float("nan"), dtype=torch.float32, device="cuda") if out is None else out
    r.run(x_dev, out, ldx=ldx)
    torch.cuda.synchronize()
    return out[:rows].cpu().numpy().astype(np.float64), r


def _check(lib, case, seed=0, offset=0):
    x = wl.make_reduce_input(case, seed)
    big = torch.full((x.numel() + offset,), float("nan"), dtype=torch.float32, device="cuda")
    dev = big[offset:]
    dev.copy_(x.cuda())
    got, r = _run(lib, dev, case.rows, case.cols, case.ldx)
    ref = oracle.reduce_rows(x, case.rows, case.cols, case.ldx)
    err = np.abs(got - ref)
    bound = _bound(x, case.rows, case.cols, case.ldx)
    assert np.all(np.isfinite(got)), case.name
    assert np.all(err <= bound), f"{case.name}: max err/bound {np.max(err / np.maximum(bound, 1e-300))}"
    return got, r


@pytest.mark.parametrize("case", [wl.REDUCE_VEC, wl.REDUCE_ROWS], ids=lambda c: c.name)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_page_cases(lib, case, seed):
    _check(lib, case, seed)


@pytest.mark.parametrize("rows,cols", [(1, 4096), (4, 4096), (3, 1 << 20), (1, (1 << 22) + 3)])
def test_integer_inputs_are_exact(lib, rows, cols):
    """All-ones rows sum to cols exactly; rows of small integers sum exactly
    (every partial sum is an integer below 2^24)."""
    ones = torch.ones(rows * cols, dtype=torch.float32, device="cuda")
    got, _ = _run(lib, ones, rows, cols)
    assert np.array_equal(got, np.full(rows, float(cols)))
    case = wl.ReduceCase("ints", rows, cols, ("ints", -3, 3))
    x = wl.make_reduce_input(case, 3)
    got, _ = _run(lib, x.cuda(), rows, cols)
    assert np.array_equal(got, oracle.reduce_rows(x, rows, cols))


RAGGED = [
    wl.ReduceCase("r1x1", 1, 1),
    wl.ReduceCase("r2x3_pad", 2, 3, ldx=7),
    wl.ReduceCase("r7x5_pad", 7, 5, ldx=9),
    wl.ReduceCase("r3x4097", 3, 4097),
    wl.ReduceCase("r5x12345_pad", 5, 12345, ldx=12350, dist=("uniform", -2.0, 2.0)),
    wl.ReduceCase("r1000x777_pad", 1000, 777, ldx=781),
    wl.ReduceCase("r2x1048583", 2, (1 << 20) + 7),
    wl.ReduceCase("r700x70000", 700, 70000, dist=("normal", 0.01)),
]


@pytest.mark.parametrize("case", RAGGED, ids=lambda c: c.name)
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_ragged_padded_unaligned(lib, case, offset):
    """Ragged lengths, padded pitches (NaN padding must not leak) and bases
    that are not 16-byte aligned (the head and tail elements)."""
    _check(lib, case, seed=offset, offset=offset)


def test_split_rows_reproducible_and_workspace_left_zero(lib):
    case = wl.ReduceCase("split", 2, (1 << 21) + 5)
    x = wl.make_reduce_input(case, 4).cuda()
    r = lib.RowReduce(case.rows, case.cols)
    assert r.ws_bytes > 0  # rows split across CTAs
    outs = []
    for _ in range(3):
        out = torch.empty(case.rows, dtype=torch.float32, device="cuda")
        r.run(x, out)
        outs.append(out.cpu())
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    counters = r.workspace[-4 * case.rows:].view(torch.int32)
    assert int(counters.abs().sum()) == 0


def test_full_size_sampled_rows(lib):
    """The 16384 x 16384 bandwidth workload: every output finite, sampled rows
    against the oracle, repeated runs bitwise equal."""
    case = wl.REDUCE_LARGE
    x = wl.make_reduce_input(case, 0)
    dev = x.cuda()
    got, r = _run(lib, dev, case.rows, case.cols)
    assert np.all(np.isfinite(got))
    rows = sorted(set([0, 1, case.rows - 1] + list(np.random.default_rng(0).integers(0, case.rows, 61))))
    xs = x.view(case.rows, case.cols)
    for row in rows:
        ref = oracle.reduce_rows(xs[row], 1, case.cols)[0]
        b = _bound(xs[row], 1, case.cols, 0)[0]
        assert abs(got[row] - ref) <= b, row
    again, _ = _run(lib, dev, case.rows, case.cols)
    assert np.array_equal(got, again)


def test_degenerate_and_errors(lib):
    x = torch.ones(64, dtype=torch.float32, device="cuda")
    out = torch.full((4,), 7.0, dtype=torch.float32, device="cuda")
    assert lib.reduce_rows_f32(x.data_ptr(), 0, 16, 0, out.data_ptr()) == lib.GEMM_OK
    assert lib.reduce_rows_f32(x.data_ptr(), 4, 0, 0, out.data_ptr()) == lib.GEMM_OK
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [0.0, 0.0, 0.0, 0.0]
    # a split plan without its workspace
    rows, cols = 1, 1 << 20
    big = torch.ones(cols, dtype=torch.float32, device="cuda")
    assert lib.reduce_rows_workspace_size(rows, cols) > 0
    assert lib.reduce_rows_f32(big.data_ptr(), rows, cols, 0, out.data_ptr()) == lib.GEMM_ERR_WORKSPACE
