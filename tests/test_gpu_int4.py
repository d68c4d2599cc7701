"""GPU parity of the int4-weight GEMM (dequantisation inside the mainloop)
against the fp64 oracle, through the C ABI.  Same tolerances as the dense
path.  Every test runs in both kernel forms where the shape allows: the
fp16 form (each weight expanded to fp16 q * s, rounded once; the zero point
z * s times the activation's group sums, in fp32) and the e4m3 form (codes as
exact e4m3 values, the activation as three e4m3 terms per 128-deep block,
all scales applied in fp32 after the MMA; activations of at most 16 rows,
K-contiguous, K and group multiples of 128).  `form` "default" takes the
planner's default (the fp16 form); "e4m3" asks for the e4m3 form
(LGT_GEMM_INT4_FORM=e4m3), which the planner grants where the shape allows."""
import numpy as np
import pytest
import torch

import helpers
import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full, oracle_sample, run_case

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG


def _case(M, N, Kd, al=K, split=1, group=128, zero=8.0, scale=("uniform", 0.005, 0.02), name=""):
    nm = f"int4_m{M}_n{N}_k{Kd}_{'a-kcontig' if al == K else 'a-mcontig'}_g{group}_s{split}{name}"
    return wl.GemmCase(nm, M, N, Kd, al, K, wl.F16, wl.INT4, wl.F16, ("normal", 1.0), ("bytes",), split_k=split,
                       group_size=group, zero_value=zero, scale_dist=scale)


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


@pytest.fixture(params=["default", "e4m3"])
def form(request, monkeypatch):
    if request.param == "e4m3":
        monkeypatch.setenv("LGT_GEMM_INT4_FORM", "e4m3")
    return request.param


def _check_form(g, form, case):
    want_f8 = (form == "e4m3" and case.M <= 16 and case.a_layout == K and case.K % 128 == 0
               and case.group_size % 128 == 0 and (g.info.k_per_split // 64) % 2 == 0)
    assert g.info.dequant_form == (2 if want_f8 else 1), (form, case.name)


@pytest.mark.parametrize("M", [1, 5, 16, 33])
@pytest.mark.parametrize("N,Kd", [(128, 128), (300, 640), (1000, 256)])
def test_int4_small(M, N, Kd, form):
    for zero in (8.0, None):
        case = _case(M, N, Kd, zero=zero)
        inp = wl.make_inputs(case, seed=M + N)
        c, g, _ = run_case(case, inp)
        assert g.info.kernel == 1 and g.info.swap_ab == 1
        _check_form(g, form, case)
        assert_close(c, oracle_full(case, inp), case.name)
        g.close()


@pytest.mark.parametrize("split", [2, 3, 8, 0])
def test_int4_split_k(split, form):
    case = _case(16, 700, 4096, split=split)
    inp = wl.make_inputs(case, seed=split + 1)
    c, g, _ = run_case(case, inp, reps=2)
    _check_form(g, form, case)
    if split:
        assert g.info.split_k == split
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


@pytest.mark.parametrize("group", [64, 256])
def test_int4_group_sizes(group, form):
    case = _case(9, 260, 1024, group=group, split=2)
    inp = wl.make_inputs(case, seed=group)
    c, g, _ = run_case(case, inp)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


@pytest.mark.parametrize("N,Kd,group,split", [(384, 8192, 64, 3), (300, 4096, 128, 5), (256, 16384, 512, 0),
                                                (640, 2048, 64, 7)])
def test_int4_scale_windows(N, Kd, group, split, form):
    """Scale reads along a run: the fp16 form loads each K block's scale two
    stages ahead by a walk over the same stages, the e4m3 form reads windows
    of 8 groups (16 bytes) of a row.  Runs that start and end inside a group
    or a window, short runs (split 7 over 5 tiles: one unit of 5 K blocks per
    CTA), rows beyond N, group 64 (two groups a stage) and 512 (a group every
    two stages)."""
    case = _case(16, N, Kd, group=group, split=split)
    inp = wl.make_inputs(case, seed=N + group)
    c, g, _ = run_case(case, inp, reps=2)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


def test_int4_unaligned_scale_rows(form):
    """A scale array that does not start on a 16-byte boundary cannot be
    read 16 bytes at a time: the per-K-block load path gives the same result."""
    case = _case(16, 384, 2048, group=64, split=2)
    inp = wl.make_inputs(case, seed=21)
    ref = oracle_full(case, inp)
    c_al, g, _ = run_case(case, inp)
    m = lib()
    A, B = inp.A.cuda(), inp.B.cuda()
    n_sc = inp.scales.numel()
    big = torch.zeros(n_sc + 8, dtype=inp.scales.dtype, device="cuda")
    big[1:1 + n_sc] = inp.scales.reshape(-1).cuda()
    sc = big[1:1 + n_sc]
    assert sc.data_ptr() % 16 != 0
    zr = inp.zeros.cuda() if inp.zeros is not None else None
    C = torch.full((case.M * inp.ldc,), float("nan"), dtype=wl.TORCH_DTYPE[case.c_dtype], device="cuda")
    g.run(A, B, C, sc, zr)
    assert g.sync_status() == m.GEMM_OK
    c_un = oracle.decode(C.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
    assert_close(c_un, ref, case.name + " (unaligned scales)")
    assert_close(c_al, ref, case.name)
    g.close()


def test_int4_activation_m_contiguous():
    case = _case(40, 512, 512, al=MN, split=2)
    inp = wl.make_inputs(case, seed=3)
    c, g, _ = run_case(case, inp)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


def test_int4_general_dequant_path(form):
    """Non-integer zero points and very small scales: the result must match
    the exact oracle, and also the oracle on fp16-rounded weights (what the
    fp16 form computes)."""
    case = _case(8, 384, 512, split=1, zero=7.5, scale=("uniform", 2e-4, 9e-4))
    inp = wl.make_inputs(case, seed=9)
    c, g, _ = run_case(case, inp)
    ref = oracle_full(case, inp)
    assert_close(c, ref, case.name)
    # and it is within tolerance of the oracle on fp16-rounded weights too
    a, b = oracle.logical_operands(case.M, case.N, case.K, inp.A, case.a_layout, inp.lda, case.a_dtype, inp.B,
                                   case.b_layout, 0, wl.INT4, inp.scales, inp.zeros, case.group_size)
    ref_rounded_w = a @ oracle.round_to(b, oracle.F16)
    assert_close(c, ref_rounded_w, case.name + " (rounded weights)")
    g.close()


def test_int4_closed_forms(form):
    m = lib()
    M, N, Kd = 4, 256, 256
    A = torch.empty(M * Kd, dtype=torch.float16).uniform_(-1, 1)
    a64 = oracle.decode(A, oracle.F16).reshape(M, Kd)
    desc = m.make_desc(M, N, Kd, a_dtype=m.GEMM_F16, b_dtype=m.GEMM_INT4, c_dtype=m.GEMM_F16, split_k=1,
                       num_sms=148)
    g = m.Gemm(desc)
    C = torch.empty(M * N, dtype=torch.float16, device="cuda")
    Ad = A.cuda()
    # all codes 8 with zero point 8 -> zero: in the fp16 form 8 s - 8 s is
    # exactly 0 per weight; in the e4m3 form 8 s (sum of the activation) less
    # s z Ag cancels to fp32 rounding.
    W = torch.full((N * Kd // 2,), 0x88, dtype=torch.uint8, device="cuda")
    s = torch.full((N, Kd // 128), 0.01, dtype=torch.float16, device="cuda")
    g.run(Ad, W, C, s, None)
    assert g.sync_status() == 0
    assert torch.max(torch.abs(C.float())).item() <= 1e-4
    # all codes 9, scale 1/64 -> C[m, n] = sum_k a[m, k] / 64
    W.fill_(0x99)
    s.fill_(1.0 / 64)
    g.run(Ad, W, C, s, None)
    assert g.sync_status() == 0
    got = oracle.decode(C.cpu(), oracle.F16).reshape(M, N)
    want = np.repeat((a64.sum(axis=1) / 64)[:, None], N, axis=1)
    assert_close(got, want, "codes 9")
    g.close()


def test_int4_full_size_sampled(form):
    case = wl.INT4_DEQUANT
    inp = wl.make_inputs(case, seed=0)
    c, g, _ = run_case(case, inp, reps=2)
    _check_form(g, form, case)
    assert g.info.split_k == oracle.splitk_factor(case.M, case.N, case.K, 128, 128, 64, 148)
    rows, cols = wl.sample_indices(case.M, case.N, 1500, seed=2)
    assert_close(c[rows, cols], oracle_sample(case, inp, rows, cols), case.name)
    assert np.all(np.isfinite(c))
    g.close()


def test_int4_full_size_repeats_bitwise(form):
    """Back-to-back runs of the full-size problem in deterministic mode give
    the same bits every time, over the whole output.  A weight stage handed
    back to its producer before every expander's loads of it had returned
    once showed here as a few columns of one tile changing from run to run
    (the stage refilled with the codes one ring lap further along K)."""
    m = lib()
    case = wl.INT4_DEQUANT
    inp = wl.make_inputs(case, seed=0)
    d = helpers.desc_for(m, case, 148)
    d.flags = m.GEMM_FLAG_DETERMINISTIC
    g = m.Gemm(d)
    _check_form(g, form, case)
    A, B = inp.A.cuda(), inp.B.cuda()
    sc, zr = inp.scales.cuda(), inp.zeros.cuda()
    first = None
    for _ in range(12):
        C = torch.full((case.M * inp.ldc,), float("nan"), dtype=torch.float16, device="cuda")
        g.run(A, B, C, sc, zr)
        assert g.sync_status() == m.GEMM_OK
        bits = C.view(torch.int16)
        if first is None:
            first = bits.clone()
            assert torch.isfinite(C).all()
        else:
            assert torch.equal(bits, first)
    rows, cols = wl.sample_indices(case.M, case.N, 500, seed=3)
    c = oracle.decode(C.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
    assert_close(c[rows, cols], oracle_sample(case, inp, rows, cols), case.name)
    g.close()
