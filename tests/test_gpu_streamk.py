"""GPU parity of the stream-K tail: with no K split, the tiles of a last
partial wave are cut into single K blocks spread evenly over all persistent
CTAs (or CTA pairs) and reduced through the fp32 workspace.  Checked against
the fp64 oracle on both tensor-core kernels, with ragged edges, repeated
runs on one workspace (it must come back zero-filled), and against the
GEMM_FLAG_DETERMINISTIC plan, which runs every tile whole and reproduces its
output bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full, run_case

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG
BF16, F16 = wl.BF16, wl.F16


@pytest.fixture(autouse=True)
def _env(monkeypatch):
    lib()
    for v in ("LGT_GEMM_BN", "LGT_GEMM_PAIR_BN", "LGT_GEMM_STREAMK"):
        monkeypatch.delenv(v, raising=False)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _case(M, N, Kd, al, bl, dt=BF16):
    name = wl.case_name(dt, M, N, Kd, al, bl, "streamk")
    return wl.GemmCase(name, M, N, Kd, al, bl, dt, dt, dt, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0),
                       split_k=1)


def _desc(m, case, flags=0):
    l_a, l_b, l_c = case.dense_ld()
    return m.make_desc(case.M, case.N, case.K, case.a_layout, case.b_layout, case.a_dtype, case.b_dtype,
                       case.c_dtype, lda=l_a, ldb=l_b, ldc=l_c, split_k=case.split_k, num_sms=148, flags=flags)


def _tail_region_zero(g, M, N, tiles):
    pad = lambda x: (x + 255) // 256 * 256
    n = pad(M * N * 4) + pad(tiles * 4)
    return torch.count_nonzero(g.workspace[:n]).item() == 0


def _single_cta_shape():
    # 128 x 128 tiles (LGT_GEMM_BN=128): three whole waves of the SMs plus
    # about 1/8 of a wave (the tail needs three whole waves before it);
    # ragged M and N edges; 4 K blocks with a ragged last one
    s = _sms()
    rows = 8
    cols = -(-(3 * s + s // 8) // rows)
    return rows * 128 - 5, cols * 128 - 3, 3 * 64 + 40


@pytest.mark.parametrize("al", [K, MN])
@pytest.mark.parametrize("bl", [K, MN])
def test_streamk_tail_single_cta(al, bl, monkeypatch):
    monkeypatch.setenv("LGT_GEMM_PAIR", "0")
    monkeypatch.setenv("LGT_GEMM_BN", "128")
    M, N, Kd = _single_cta_shape()
    case = _case(M, N, Kd, al, bl)
    inp = wl.make_inputs(case, seed=al * 2 + bl)
    c, g, _ = run_case(case, inp, reps=3)
    assert g.info.kernel == 0 and g.info.split_k == 1 and g.info.streamk_tiles > 0
    assert_close(c, oracle_full(case, inp), case.name)
    tiles = -(-M // g.info.tile_m) * -(-N // g.info.tile_n)
    assert _tail_region_zero(g, M, N, 2 * tiles)  # arrival and finished-row counters
    g.close()


@pytest.mark.parametrize("al,bl,dt", [(K, MN, BF16), (MN, MN, BF16), (K, K, F16), (MN, K, F16)])
def test_streamk_tail_pairs(al, bl, dt, monkeypatch):
    monkeypatch.setenv("LGT_GEMM_PAIR", "1")
    monkeypatch.setenv("LGT_GEMM_PAIR_BN", "256")
    # 256 x 256 pair tiles: 11 x 22 = 242 tiles, three whole waves of 74..76
    # CTA pairs plus 14..20 tiles; ragged edges and a ragged last K block
    case = _case(11 * 256 - 7, 22 * 256 - 100, 3 * 64 + 40, al, bl, dt)
    inp = wl.make_inputs(case, seed=7)
    c, g, _ = run_case(case, inp, reps=2)
    assert g.info.kernel == 2 and g.info.split_k == 1
    tiles = -(-case.M // 256) * -(-case.N // 256)
    if g.info.streamk_tiles == 0:
        pytest.skip(f"{tiles} pair tiles fill whole waves on this device")
    assert_close(c, oracle_full(case, inp), case.name)
    assert _tail_region_zero(g, case.M, case.N, 4 * tiles)  # two counters per half-tile
    g.close()


def test_deterministic_flag_reproduces_and_agrees(monkeypatch):
    monkeypatch.setenv("LGT_GEMM_PAIR", "0")
    monkeypatch.setenv("LGT_GEMM_BN", "128")
    m = lib()
    M, N, Kd = _single_cta_shape()
    case = _case(M, N, Kd, K, MN)
    inp = wl.make_inputs(case, seed=21)
    gd = m.Gemm(_desc(m, case, flags=m.GEMM_FLAG_DETERMINISTIC))
    assert gd.info.streamk_tiles == 0
    c1, _, C1 = run_case(case, inp, gemm=gd)
    c2, _, C2 = run_case(case, inp, gemm=gd)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    gd.close()
    c_sk, g, _ = run_case(case, inp)
    assert g.info.streamk_tiles > 0
    g.close()
    ref = oracle_full(case, inp)
    assert_close(c1, ref, "deterministic")
    assert_close(c_sk, ref, "stream-K tail")
    assert_close(c_sk, c1, "stream-K tail vs deterministic")


def test_streamk_full_size_square():
    """The 4096^3 workload: planner's choice (CTA pairs, stream-K tail where
    the last wave is partial), sampled against the oracle."""
    case = wl.SQUARE_BF16
    inp = wl.make_inputs(case, seed=0)
    c, g, _ = run_case(case, inp, reps=2)
    assert g.info.kernel == 2
    from helpers import oracle_sample
    rows, cols = wl.sample_indices(case.M, case.N, 3000, seed=5)
    assert_close(c[rows, cols], oracle_sample(case, inp, rows, cols), case.name)
    assert np.all(np.isfinite(c))
    g.close()


@pytest.mark.parametrize("shape,split,pair", [((300, 700, 4000), 3, "0"), ((64, 4096, 16384), 0, "0"),
                                              ((16, 700, 4000), 7, "0"), ((512, 512, 2048), 4, "1"),
                                              ((129, 65, 777), 16, "0")],
                         ids=lambda x: str(x))
def test_deterministic_split_k(shape, split, pair, monkeypatch):
    """GEMM_FLAG_DETERMINISTIC with a split factor above 1: per-run partial
    slots summed in run order -- two runs are bitwise identical, and both
    are within tolerance of the oracle and of the atomic-reduction plan."""
    monkeypatch.setenv("LGT_GEMM_PAIR", pair)
    m = lib()
    M, N, Kd = shape
    case = wl.GemmCase(wl.case_name(BF16, M, N, Kd, K, K, f"det_s{split}"), M, N, Kd, K, K, BF16, BF16, BF16,
                       ("normal", 0.1), ("normal", 0.1), split_k=split)
    inp = wl.make_inputs(case, seed=split + 3)
    gd = m.Gemm(_desc(m, case, flags=m.GEMM_FLAG_DETERMINISTIC))
    assert gd.info.split_k > 1
    c1, _, C1 = run_case(case, inp, gemm=gd)
    c2, _, C2 = run_case(case, inp, gemm=gd)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    gd.close()
    c_at, g, _ = run_case(case, inp)
    g.close()
    ref = oracle_full(case, inp)
    assert_close(c1, ref, "deterministic")
    assert_close(c_at, ref, "atomic")


def test_deterministic_int4_split_k():
    m = lib()
    case = wl.GemmCase("int4_det_m16_n700_k4096", 16, 700, 4096, K, K, F16, wl.INT4, F16, ("normal", 1.0), ("bytes",),
                       split_k=8, group_size=128, zero_value=8.0)
    inp = wl.make_inputs(case, seed=4)
    l_a, l_b, l_c = case.dense_ld()
    desc = m.make_desc(case.M, case.N, case.K, K, K, F16, wl.INT4, F16, lda=l_a, ldb=0, ldc=l_c, split_k=8,
                       group_size=128, num_sms=148, flags=m.GEMM_FLAG_DETERMINISTIC)
    gd = m.Gemm(desc)
    c1, _, C1 = run_case(case, inp, gemm=gd)
    c2, _, C2 = run_case(case, inp, gemm=gd)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    assert_close(c1, oracle_full(case, inp), case.name)
    gd.close()
