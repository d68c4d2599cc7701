"""GPU parity: the tensor-core GEMM through the C ABI against the fp64 CPU
oracle, element by element.  Tolerances (the library's acceptance bound):
|C_gpu - C_ref| <= 2e-2 (|C_ref| + 1) elementwise and relative Frobenius
error <= 2e-3, with C_ref the unrounded fp64 sum."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full, oracle_sample, run_case

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG
F16, BF16 = wl.F16, wl.BF16


def _splitk_region_zero(g, M, N):
    """The fp32 partial sums and the per-tile counters (the start of the
    workspace) are left zero by every run; repacked operand copies follow."""
    pad = lambda x: (x + 255) // 256 * 256
    tiles = -(-M // g.info.tile_m) * -(-N // g.info.tile_n)
    n = pad(M * N * 4) + pad(tiles * 4)
    return torch.count_nonzero(g.workspace[:n]).item() == 0


def _case(M, N, Kd, al, bl, dt=BF16, split=1, lda=0, ldb=0, ldc=0, dist=("uniform", -1.0, 1.0)):
    name = wl.case_name(dt, M, N, Kd, al, bl, f"s{split}")
    return wl.GemmCase(name, M, N, Kd, al, bl, dt, dt, dt, dist, dist, split_k=split, lda=lda, ldb=ldb, ldc=ldc)


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


# ------------------------------------------------------------ 256^3, 4 layouts

@pytest.mark.parametrize("case", wl.small_layout_cases(), ids=lambda c: c.name)
def test_small_fp16_all_layouts(case):
    inp = wl.make_inputs(case, seed=0)
    c, g, _ = run_case(case, inp)
    ref = oracle_full(case, inp)
    assert_close(c, ref, case.name)
    g.close()


def test_small_layouts_agree_within_one_ulp():
    outs = []
    base = wl.small_layout_cases()[0]
    inp0 = wl.make_inputs(base, seed=1)
    a = oracle.a_logical(inp0.A, 256, 256, K, 256, F16)
    b = oracle.b_logical(inp0.B, 256, 256, K, 256, F16)
    for case in wl.small_layout_cases():
        # the same logical matrices, stored in this case's layouts
        A = torch.from_numpy((a if case.a_layout == K else a.T).copy().reshape(-1)).half()
        B = torch.from_numpy((b.T if case.b_layout == K else b).copy().reshape(-1)).half()
        inp = wl.GemmInputs(case, A, B, 256, 256, 256)
        c, g, _ = run_case(case, inp)
        outs.append(c)
        g.close()
    for o in outs[1:]:
        # fp16 values: one ulp of the larger magnitude
        ulp = np.spacing(np.maximum(np.abs(o), np.abs(outs[0])).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(o - outs[0]) <= ulp)


# ------------------------------------------------------------ ragged shapes

SHAPES = [(1, 1, 1), (1, 17, 33), (129, 130, 65), (200, 300, 1000), (257, 64, 192), (64, 513, 300),
          (130, 16, 17), (16, 16, 16), (300, 40, 128)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
def test_ragged_shapes(shape, al, bl):
    M, N, Kd = shape
    for dt in (F16, BF16):
        case = _case(M, N, Kd, al, bl, dt)
        inp = wl.make_inputs(case, seed=M + N + Kd)
        c, g, _ = run_case(case, inp)
        assert_close(c, oracle_full(case, inp), case.name)
        g.close()


@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
def test_padded_leading_dims(al, bl):
    M, N, Kd = 150, 200, 260
    lda = (Kd if al == K else M) + 24
    ldb = (Kd if bl == K else N) + 8
    case = _case(M, N, Kd, al, bl, BF16, lda=lda, ldb=ldb, ldc=N + 40)
    inp = wl.make_inputs(case, seed=5)
    c, g, _ = run_case(case, inp)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


@pytest.fixture(params=["kernel", "prepass"])
def realign_mode(request, monkeypatch):
    """How operands TMA cannot address are read: by the kernel's realigning
    loader (TMA boxes per row class, in the perpDim order, then a realigning
    pass in shared memory), or through the repacking pre-pass."""
    if request.param == "kernel":
        monkeypatch.setenv("LGT_GEMM_REALIGN", "1")
    return request.param


@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
def test_unaligned_leading_dims(al, bl, realign_mode):
    """Leading dimensions that are not a multiple of 8 elements (rows not on
    16-byte boundaries): realigned inside the kernel, or by the copy."""
    M, N, Kd = 131, 203, 517

    def odd_ld(base):
        ld = base + 1
        return ld + 1 if ld % 8 == 0 else ld

    lda = odd_ld(Kd if al == K else M)
    ldb = odd_ld(Kd if bl == K else N)
    case = _case(M, N, Kd, al, bl, F16, lda=lda, ldb=ldb, ldc=N)
    inp = wl.make_inputs(case, seed=6)
    c, g, _ = run_case(case, inp)
    prepass = realign_mode == "prepass"
    assert g.info.realign == (0 if prepass else 1)
    assert bool(g.info.repack_a) == prepass and bool(g.info.repack_b) == prepass
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


@pytest.mark.parametrize("shape", [(100, 120, 200), (40, 333, 130), (300, 129, 64)], ids=lambda s: "x".join(map(str, s)))
def test_misaligned_base_pointers(shape, realign_mode):
    M, N, Kd = shape
    for al, bl in ((MN, K), (K, MN)):
        case = _case(M, N, Kd, al, bl, BF16)
        inp = wl.make_inputs(case, seed=7)
        c, g, _ = run_case(case, inp, seed_offsets=(1, 3))
        assert_close(c, oracle_full(case, inp), case.name)
        g.close()


def test_realigned_bits_match_tma_layout(monkeypatch):
    """The same operand through TMA (aligned copy) and through the realigning
    loader (the copy at a 2-byte offset): every element of C is the same
    bits, for K- and M-contiguous A, swapped and not."""
    monkeypatch.setenv("LGT_GEMM_REALIGN", "1")
    m = lib()
    for M, N, Kd, al in ((1000, 520, 320, MN), (1000, 520, 320, K), (40, 700, 960, K), (40, 700, 960, MN)):
        case = _case(M, N, Kd, al, K, BF16)
        inp = wl.make_inputs(case, seed=11)
        c0, g0, C0 = run_case(case, inp)
        c1, g1, C1 = run_case(case, inp, seed_offsets=(1, 0), gemm=g0)
        assert g0.info.realign == 1
        assert torch.equal(C0.view(torch.int16), C1.view(torch.int16)), case.name
        g0.close()


# ------------------------------------------------------------ split-K and swap

@pytest.mark.parametrize("split", [2, 3, 7, 16])
@pytest.mark.parametrize("shape", [(200, 300, 1000), (64, 1000, 2048), (16, 700, 4000), (129, 65, 777)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_k(shape, split):
    M, N, Kd = shape
    for al, bl in ((K, K), (MN, MN)):
        case = _case(M, N, Kd, al, bl, BF16, split=split)
        inp = wl.make_inputs(case, seed=split)
        c, g, _ = run_case(case, inp, reps=2)   # second run reuses the self-cleaned workspace
        assert g.info.split_k == split
        assert_close(c, oracle_full(case, inp), case.name)
        assert _splitk_region_zero(g, M, N)
        g.close()


def test_split_k_with_empty_splits():
    # 5 K blocks over 8 splits: three splits have no work
    case = _case(100, 150, 320, K, MN, F16, split=8)
    inp = wl.make_inputs(case, seed=3)
    c, g, _ = run_case(case, inp)
    assert_close(c, oracle_full(case, inp), case.name)
    assert _splitk_region_zero(g, 100, 150)
    g.close()


@pytest.mark.parametrize("M", [1, 7, 16, 33, 64])
@pytest.mark.parametrize("al", [K, MN])
def test_swap_ab_skinny(M, al):
    for bl in (K, MN):
        case = _case(M, 1000, 700, al, bl, BF16)
        inp = wl.make_inputs(case, seed=M)
        c, g, _ = run_case(case, inp)
        assert g.info.swap_ab == 1
        assert_close(c, oracle_full(case, inp), case.name)
        g.close()


def test_k_zero_and_empty():
    m = lib()
    case = _case(33, 44, 0, K, K, F16)
    g = m.Gemm(m.make_desc(33, 44, 0, a_dtype=m.GEMM_F16, num_sms=148))
    C = torch.full((33 * 44,), 7.0, dtype=torch.float16, device="cuda")
    A = torch.zeros(1, dtype=torch.float16, device="cuda")
    g.run(A, A, C)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0
    g.close()
    g = m.Gemm(m.make_desc(0, 44, 10, a_dtype=m.GEMM_F16, num_sms=148))
    g.run(A, A, C)
    g.close()
    del case


def test_auto_split_matches_rule_and_oracle():
    case = _case(64, 2048, 8192, K, K, BF16, split=0, dist=("normal", 0.1))
    inp = wl.make_inputs(case, seed=11)
    c, g, _ = run_case(case, inp)
    assert g.info.split_k == oracle.splitk_factor(64, 2048, 8192, 128, 128, 64, 148)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


# ------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("case", [wl.SQUARE_BF16, wl.SKINNY_SPLITK, wl.IRREGULAR], ids=lambda c: c.name)
def test_full_size_sampled(case):
    inp = wl.make_inputs(case, seed=0)
    c, g, _ = run_case(case, inp, reps=2)
    rows, cols = wl.sample_indices(case.M, case.N, 3000, seed=1)
    ref = oracle_sample(case, inp, rows, cols)
    assert_close(c[rows, cols], ref, case.name)
    assert np.all(np.isfinite(c))
    g.close()


def test_skinny_full_oracle():
    # small enough for the full fp64 oracle: every element checked
    case = wl.SKINNY_SPLITK
    inp = wl.make_inputs(case, seed=2)
    c, g, _ = run_case(case, inp)
    assert g.info.split_k == 128
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


# ------------------------------------------------------------ integer helpers

def test_magic_division_on_device():
    m = lib()
    rng = np.random.default_rng(1)
    n = np.concatenate([np.arange(0, 1 << 16), rng.integers(0, 1 << 31, 1 << 20),
                        np.arange((1 << 31) - (1 << 16), 1 << 31)]).astype(np.uint32)
    nd = torch.from_numpy(n.view(np.int32)).cuda()
    q = torch.empty_like(nd)
    r = torch.empty_like(nd)
    for d in (1, 3, 7, 128, 148, 3000, 4095, (1 << 31) - 1):
        st = m.gemm_magic_divmod_device(nd.data_ptr(), n.size, d, q.data_ptr(), r.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
        assert st == m.GEMM_OK
        torch.cuda.synchronize()
        assert np.array_equal(q.cpu().numpy().view(np.uint32), n // np.uint32(d))
        assert np.array_equal(r.cpu().numpy().view(np.uint32), n % np.uint32(d))
