"""Failure detection on the GPU without a fault: a bounded wait that runs out.

A plan made with GEMM_FLAG_TEST_WITHHOLD_STAGE withholds, in its first run,
the first pipeline stage of one CTA (no copy is issued for it), so the MMA
issuer's wait on that stage gives up after the plan's wait limit (here 20 ms,
from LGT_GEMM_WAIT_LIMIT_MS at gemm_create).  The kernel records
GEMM_ERR_TIMEOUT in the plan's status word, lets every copy it did issue land,
frees its TMEM and returns; gemm_sync_status reports the timeout and clears
it.  The next run of the same plan, on the same buffers, is normal and must
match the oracle: the context is still usable."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full

pytestmark = pytest.mark.gpu


def _plan(m, case, monkeypatch, flags):
    monkeypatch.setenv("LGT_GEMM_WAIT_LIMIT_MS", "20")
    l_a, l_b, l_c = case.dense_ld()
    desc = m.make_desc(case.M, case.N, case.K, case.a_layout, case.b_layout, case.a_dtype, case.b_dtype,
                       case.c_dtype, lda=l_a, ldb=l_b, ldc=l_c, split_k=1, num_sms=148, flags=flags)
    g = m.Gemm(desc)
    monkeypatch.delenv("LGT_GEMM_WAIT_LIMIT_MS")
    return g


@pytest.mark.parametrize("al,bl", [(wl.K_CONTIG, wl.K_CONTIG), (wl.MN_CONTIG, wl.MN_CONTIG)])
def test_withheld_stage_times_out_then_next_run_is_correct(monkeypatch, al, bl):
    m = lib()
    case = wl.GemmCase(wl.case_name(wl.F16, 256, 256, 256, al, bl, "withhold"), 256, 256, 256, al, bl,
                       wl.F16, wl.F16, wl.F16, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), split_k=1)
    inp = wl.make_inputs(case, seed=3)
    g = _plan(m, case, monkeypatch, m.GEMM_FLAG_TEST_WITHHOLD_STAGE)
    assert g.info.kernel == 0 and g.info.split_k == 1 and g.info.streamk_tiles == 0 and g.info.cluster_size == 0
    A, B = inp.A.cuda(), inp.B.cuda()
    C = torch.full((case.M * inp.ldc,), float("nan"), dtype=torch.float16, device="cuda")
    g.run(A, B, C)
    assert g.sync_status() == m.GEMM_ERR_TIMEOUT
    assert g.sync_status() == m.GEMM_OK  # reading the status cleared it
    g.run(A, B, C)
    assert g.sync_status() == m.GEMM_OK
    torch.cuda.synchronize()
    c = oracle.decode(C.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()


def test_other_plans_unaffected_by_short_limit_and_flag(monkeypatch):
    """A plan without the flag, made while the short limit is set, runs
    normally: the limit alone never fires on a healthy run."""
    m = lib()
    case = wl.small_layout_cases()[0]
    inp = wl.make_inputs(case, seed=4)
    g = _plan(m, case, monkeypatch, 0)
    A, B = inp.A.cuda(), inp.B.cuda()
    C = torch.empty(case.M * inp.ldc, dtype=wl.TORCH_DTYPE[case.c_dtype], device="cuda")
    for _ in range(3):
        g.run(A, B, C)
    assert g.sync_status() == m.GEMM_OK
    c = oracle.decode(C.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()
