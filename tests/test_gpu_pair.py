"""GPU parity of the CTA-pair kernel (two CTAs of a cluster share a 256 x w
tile, w in 128..256, through one cta_group::2 MMA) against the fp64 oracle.
The planner uses it for large problems; here LGT_GEMM_PAIR=1 selects it on
small and ragged shapes too (LGT_GEMM_PAIR_BN picks w), so that pair tiles
whose second half is partly or wholly outside the matrix, ragged K, split-K
through per-half counters, every tile width and every operand layout are
all exercised."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, desc_for, lib, oracle_full, run_case

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG
F16, BF16 = wl.F16, wl.BF16


WIDTHS = [256, 224, 192, 160, 128]


@pytest.fixture(autouse=True)
def _pairs(monkeypatch):
    lib()
    monkeypatch.setenv("LGT_GEMM_PAIR", "1")
    monkeypatch.setenv("LGT_GEMM_PAIR_BN", "256")
    monkeypatch.delenv("LGT_GEMM_BN", raising=False)


def _case(M, N, Kd, al, bl, dt=BF16, split=1, dist=("uniform", -1.0, 1.0)):
    name = wl.case_name(dt, M, N, Kd, al, bl, f"pair_s{split}")
    return wl.GemmCase(name, M, N, Kd, al, bl, dt, dt, dt, dist, dist, split_k=split)


def _run(case, seed=0, reps=1, width=256):
    inp = wl.make_inputs(case, seed=seed)
    c, g, _ = run_case(case, inp, reps=reps)
    assert g.info.kernel == 2 and g.info.tile_m == 256 and g.info.tile_n == width, "pair kernel not selected"
    return inp, c, g


@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
@pytest.mark.parametrize("dt", [F16, BF16])
def test_pair_layouts(al, bl, dt):
    case = _case(512, 512, 512, al, bl, dt)
    inp, c, g = _run(case)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


@pytest.mark.parametrize("width", WIDTHS)
@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
def test_pair_widths(width, al, bl, monkeypatch):
    # N spans two tiles and a ragged third for every width
    monkeypatch.setenv("LGT_GEMM_PAIR_BN", str(width))
    case = _case(384, 2 * width + 40, 328, al, bl)
    inp, c, g = _run(case, seed=width, width=width)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


# (M, N, K): the second CTA's half partly (300, 129+) or wholly (M = 200:
# rows 128..199 only; M = 100: the second half holds no row) outside C,
# N not a multiple of the tile, K not a multiple of 64.
SHAPES = [(300, 260, 200), (129, 513, 64), (200, 256, 1000), (100, 384, 136), (777, 1000, 520)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
def test_pair_ragged(shape, al, bl):
    M, N, Kd = shape
    case = _case(M, N, Kd, al, bl)
    inp, c, g = _run(case, seed=M)
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


@pytest.mark.parametrize("mode", ["kernel", "prepass"])
def test_pair_with_unaligned_operands(mode, monkeypatch):
    # odd leading dimensions: read in place by the realigning loader of both
    # CTAs of each pair, or copied to 16-byte pitches first
    if mode == "kernel":
        monkeypatch.setenv("LGT_GEMM_REALIGN", "1")
    # (pitches in bytes: 600 / 406, 406 / 1044, 1208 / 1060: none a multiple of 16)
    for shape, al, bl in (((300, 260, 203), MN, K), ((600, 522, 203), K, MN), ((604, 530, 330), MN, MN)):
        case = _case(*shape, al, bl)
        inp, c, g = _run(case, seed=5)
        assert g.info.kernel == 2
        assert g.info.repack_b == (1 if mode == "prepass" else 0)
        assert g.info.realign == (0 if mode == "prepass" else 1)
        assert_close(c, oracle_full(case, inp), case.name)
        g.close()


@pytest.mark.parametrize("split", [2, 3, 8])
@pytest.mark.parametrize("shape", [(512, 512, 2048), (300, 700, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_pair_split_k(shape, split):
    M, N, Kd = shape
    case = _case(M, N, Kd, K, MN, split=split)
    inp, c, g = _run(case, seed=split, reps=3)
    assert g.info.split_k == split
    assert_close(c, oracle_full(case, inp), case.name)
    # partial sums and the per-half arrival counters are left zero
    pad = lambda x: (x + 255) // 256 * 256
    tiles = -(-M // 256) * -(-N // 256)
    n = pad(M * N * 4) + pad(2 * tiles * 4)
    assert torch.count_nonzero(g.workspace[:n]).item() == 0
    g.close()


def test_pair_matches_single_cta_kernel(monkeypatch):
    """Same inputs through the pair kernel and the single-CTA 128 x 256
    kernel: both within tolerance of the oracle and of each other."""
    case = _case(1024, 768, 1536, MN, MN, F16)
    inp, c_pair, g = _run(case, seed=11)
    g.close()
    monkeypatch.setenv("LGT_GEMM_PAIR", "0")
    monkeypatch.setenv("LGT_GEMM_BN", "256")
    c_single, g1, _ = run_case(case, inp)
    assert g1.info.kernel == 0 and g1.info.tile_m == 128
    g1.close()
    ref = oracle_full(case, inp)
    assert_close(c_pair, ref, "pair")
    assert_close(c_single, ref, "single")
    assert_close(c_pair, c_single, "pair vs single")


def test_pair_static_scratch():
    m = lib()
    case = _case(512, 512, 1024, K, K, split=2)
    inp = wl.make_inputs(case, seed=3)
    g = m.Gemm(desc_for(m, case))
    assert g.info.kernel == 2
    A, B = inp.A.cuda(), inp.B.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        C = torch.full((case.M * case.N,), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = m.gemm_run_static_scratch(g.plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), stream)
        assert st == m.GEMM_OK, m.gemm_status_string(st)
        assert g.sync_status() == m.GEMM_OK
        got = oracle.decode(C.cpu(), case.c_dtype).reshape(case.M, case.N)
        assert_close(got, oracle_full(case, inp), case.name)
    g.close()


def test_planner_choice_without_overrides(monkeypatch):
    """Without overrides: the large workloads go to CTA pairs with a width
    that fills whole waves; a problem with about one wave of 128 x 256 tiles
    stays on the single-CTA kernel (pairs would need two waves)."""
    monkeypatch.delenv("LGT_GEMM_PAIR")
    monkeypatch.delenv("LGT_GEMM_PAIR_BN")
    m = lib()
    for case in (wl.SQUARE_BF16, wl.IRREGULAR):
        g = m.Gemm(desc_for(m, case))
        assert g.info.kernel == 2 and g.info.split_k == 1 and g.info.tile_n in WIDTHS
        g.close()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one_wave = _case(128 * sms // 8, 256 * 8, 512, K, K)
    g = m.Gemm(desc_for(m, one_wave))
    assert g.info.kernel == 0 and g.info.tile_n == 256
    g.close()
