"""gemm_run_static_scratch: the entry point for callers that cannot allocate
device memory when they run the GEMM (no workspace to pass).  It must give
the same results as gemm_run with a workspace, call after call, while the
split-K partial sums live in the library's fixed device scratch array.

Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, desc_for, lib, oracle_full

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG

CASES = [
    # skinny, split chosen by the SM-waste rule (swapped MMA)
    wl.GemmCase("scratch_bf16_m64_n4096_k8192_splitk-auto", 64, 4096, 8192, K, K, wl.BF16, wl.BF16, wl.BF16,
                ("normal", 0.1), ("normal", 0.1), split_k=0),
    # ragged tiles, explicit split, both operands non-K-contiguous
    wl.GemmCase("scratch_f16_m104_n320_k1000_split3", 104, 320, 1000, MN, MN, wl.F16, wl.F16, wl.F16,
                ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), split_k=3),
    # split 1: no scratch needed at all
    wl.GemmCase("scratch_bf16_m256_n256_k512_split1", 256, 256, 512, K, MN, wl.BF16, wl.BF16, wl.BF16,
                ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), split_k=1),
]


def _decode(C, case):
    return oracle.decode(C.cpu(), case.c_dtype).reshape(case.M, case.N)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_static_scratch_matches_workspace_entry_point(case):
    m = lib()
    inp = wl.make_inputs(case, seed=4)
    g = m.Gemm(desc_for(m, case))
    A, B = inp.A.cuda(), inp.B.cuda()
    stream = torch.cuda.current_stream().cuda_stream

    C_ws = torch.full((case.M * case.N,), float("nan"), dtype=wl.TORCH_DTYPE[case.c_dtype], device="cuda")
    g.run(A, B, C_ws)
    assert g.sync_status() == m.GEMM_OK
    ref_existing = _decode(C_ws, case)

    for _ in range(2):  # two calls in a row share (and must re-clear) the scratch
        C = torch.full((case.M * case.N,), float("nan"), dtype=wl.TORCH_DTYPE[case.c_dtype], device="cuda")
        st = m.gemm_run_static_scratch(g.plan, A.data_ptr(), B.data_ptr(), C.data_ptr(), stream)
        assert st == m.GEMM_OK, m.gemm_status_string(st)
        assert g.sync_status() == m.GEMM_OK
        got = _decode(C, case)
        assert np.all(np.isfinite(got))
        assert_close(got, ref_existing, case.name + " vs gemm_run")
    assert_close(got, oracle_full(case, inp), case.name + " vs oracle")
    g.close()


def test_static_scratch_rejects_what_it_cannot_hold():
    m = lib()
    # 2048 x 2048 fp32 partial sums = 16 MiB > the 8 MiB array
    big = m.Gemm(m.make_desc(2048, 2048, 1024, split_k=2, num_sms=148))
    t = torch.zeros(2048 * 2048, dtype=torch.bfloat16, device="cuda")
    st = m.gemm_run_static_scratch(big.plan, t.data_ptr(), t.data_ptr(), t.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == m.GEMM_ERR_WORKSPACE
    big.close()
    # a leading dimension that needs a realigned copy has no room in the scratch
    odd = m.Gemm(m.make_desc(100, 128, 257, lda=257, ldb=257, split_k=2, num_sms=148))
    st = m.gemm_run_static_scratch(odd.plan, t.data_ptr(), t.data_ptr(), t.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == m.GEMM_ERR_UNSUPPORTED
    odd.close()
