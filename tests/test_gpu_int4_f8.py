"""GPU parity of the int4 kernel's e4m3 form (activations of at most 16
rows, K-contiguous, K and group size multiples of 128): the codes enter the
tensor core as exact e4m3 values q * 2^-9, the fp16 activation as three e4m3
terms per 128-deep block (exact for every element within 2^-14 of its
block's largest magnitude), and the scales, zero points and activation
scales are applied per block in fp32 after the MMA.  Same tolerances as the
other int4 tests, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import helpers
import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full, run_case

pytestmark = pytest.mark.gpu

K = wl.K_CONTIG


def _case(M, N, Kd, split=1, zero=8.0, group=128, scale=("uniform", 0.005, 0.02), name=""):
    nm = f"int4f8_m{M}_n{N}_k{Kd}_g{group}_s{split}_z{zero}{name}"
    return wl.GemmCase(nm, M, N, Kd, K, K, wl.F16, wl.INT4, wl.F16, ("normal", 1.0), ("bytes",), split_k=split,
                       group_size=group, zero_value=zero, scale_dist=scale)


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


@pytest.fixture(autouse=True)
def _e4m3(monkeypatch):
    monkeypatch.setenv("LGT_GEMM_INT4_FORM", "e4m3")


@pytest.mark.parametrize("M", [1, 9, 16])
@pytest.mark.parametrize("N,Kd,split,group", [(128, 128, 1, 128), (256, 1024, 1, 128), (300, 2048, 2, 256),
                                                (640, 4096, 4, 128), (384, 8192, 0, 512), (1000, 3072, 3, 128)])
@pytest.mark.parametrize("zero", [8.0, None, 7.5])
def test_f8_form_matches_oracle(M, N, Kd, split, group, zero):
    case = _case(M, N, Kd, split, zero, group)
    inp = wl.make_inputs(case, seed=M * 7 + N + group)
    c, g, _ = run_case(case, inp, reps=2)
    assert g.info.kernel == 1 and g.info.dequant_form == 2
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


def test_f8_form_activation_dynamic_range():
    """Blocks whose elements span many binades (1e-5 next to 1e3), an
    all-zero block, a block with one nonzero element, fp16 subnormals and the
    fp16 maximum: each block gets its own power-of-two scale."""
    m = lib()
    case = _case(16, 512, 1024, split=1, zero=8.0)
    inp = wl.make_inputs(case, seed=11)
    a = inp.A.clone().reshape(16, 1024).float()
    a[0, 0:128] = 0.0                               # all-zero block
    a[1, 128:256] = 0.0
    a[1, 200] = 3.0                                 # a single nonzero
    a[2, 256:384] *= 1e-5                           # tiny block (fp16 subnormals among them)
    a[3, 384:512] = torch.logspace(-5, 3, 128)      # 1e-5 .. 1e3 in one block
    a[4, 512:640] = 3.0e3 * torch.sign(a[4, 512:640])  # large (C stays within fp16)
    a[5, 640:768] = 2.0 ** -24                      # the smallest fp16 subnormal
    inp.A = a.to(torch.float16).reshape(-1)
    c, g, _ = run_case(case, inp)
    assert g.info.dequant_form == 2
    ref = oracle_full(case, inp)
    assert_close(c, ref, case.name)
    assert np.all(np.isfinite(c))
    g.close()


def test_f8_form_deterministic_split():
    m = lib()
    case = _case(16, 1024, 8192, split=8)
    inp = wl.make_inputs(case, seed=5)
    d = helpers.desc_for(m, case, 148)
    d.flags = m.GEMM_FLAG_DETERMINISTIC
    g = m.Gemm(d)
    assert g.info.dequant_form == 2
    c1, _, C1 = run_case(case, inp, gemm=g)
    c2, _, C2 = run_case(case, inp, gemm=g)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    assert_close(c1, oracle_full(case, inp), case.name)
    g.close()


def test_f8_and_fp16_forms_agree(monkeypatch):
    """The same problem through both forms: each within tolerance of the
    oracle, and of each other."""
    case = _case(12, 768, 4096, split=4, zero=None)
    inp = wl.make_inputs(case, seed=8)
    c8, g8, _ = run_case(case, inp)
    assert g8.info.dequant_form == 2
    g8.close()
    monkeypatch.setenv("LGT_GEMM_INT4_FORM", "fp16")
    c16, g16, _ = run_case(case, inp)
    assert g16.info.dequant_form == 1
    g16.close()
    ref = oracle_full(case, inp)
    assert_close(c8, ref, case.name + " e4m3")
    assert_close(c16, ref, case.name + " fp16")
    assert_close(c8, c16.astype(np.float64), case.name + " e4m3 vs fp16")


def test_f8_form_chained_without_sync():
    """Several runs of the e4m3 form back to back in one stream, on different
    activations, with no synchronisation between them: the pre-pass of run
    i + 1 overwrites the prepared activation only after run i has read it."""
    m = lib()
    case = _case(16, 2048, 4096, split=0)
    g = m.Gemm(helpers.desc_for(m, case, 148))
    inputs = [wl.make_inputs(case, seed=40 + i) for i in range(3)]
    B = inputs[0].B.cuda()
    sc = inputs[0].scales.cuda()
    zr = inputs[0].zeros.cuda()
    outs = []
    for inp in inputs:
        C = torch.empty(case.M * case.N, dtype=torch.float16, device="cuda")
        g.run(inp.A.cuda(), B, C, sc, zr)
        outs.append(C)
    assert g.sync_status() == m.GEMM_OK
    for inp, C in zip(inputs, outs):
        inp.B, inp.scales, inp.zeros = inputs[0].B, inputs[0].scales, inputs[0].zeros
        c = oracle.decode(C.cpu(), wl.F16).reshape(case.M, case.N)
        assert_close(c, oracle_full(case, inp), case.name)
    g.close()
