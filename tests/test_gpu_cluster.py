"""GPU parity of split-K within a cluster (skinny, swapped problems whose
tiles are few: each tile's K range is split over the CTAs of one cluster and
the fp32 partials are added through distributed shared memory) against the
fp64 oracle, element by element, and against the split-K path through the
workspace.  Same tolerances as the other GEMM tests."""
import os

import numpy as np
import pytest
import torch

import workloads as wl
from helpers import assert_close, desc_for, lib, oracle_full, run_case

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG


def _case(M, N, Kd, split, al=K, bl=K, dt=wl.BF16, dist=("uniform", -1.0, 1.0)):
    name = wl.case_name(dt, M, N, Kd, al, bl, f"s{split}")
    return wl.GemmCase(name, M, N, Kd, al, bl, dt, dt, dt, dist, dist, split_k=split)


CASES = [
    # (case, expected cluster size: None = any the device holds, including none)
    (_case(64, 4096, 8192, 16), 4),
    (_case(40, 4000, 4096 + 3 * 64, 8), 4),             # ragged M, N and K blocks
    (_case(16, 3900, 2048, 4, dt=wl.F16), 4),           # BN 16, 31 tiles
    (_case(8, 7680, 1024, 2, dt=wl.F16), 2),            # 60 tiles, two CTAs a tile
    (_case(64, 4096, 700, 8), 4),                       # trailing splits without K blocks
    (_case(48, 2048, 4096, 16), None),                  # clusters of 8 where the device holds 16 of them
    (_case(64, 4096, 4096, 8, al=MN, bl=K), 4),         # A M-contiguous (the MMA's B operand MN-major)
    (_case(33, 4096, 2048, 8, al=K, bl=MN), 4),         # B N-contiguous (the MMA's A operand MN-major)
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


@pytest.mark.parametrize("case,want", CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_cluster_split_matches_oracle_and_is_reproducible(case, want):
    inp = wl.make_inputs(case, seed=2)
    c, g, C = run_case(case, inp, num_sms=148)
    cl = g.info.cluster_size
    if want is not None:
        assert cl == want, f"cluster size {cl}, expected {want}"
    if cl > 1 and not (g.info.repack_a or g.info.repack_b):
        assert g.ws_bytes == 0  # partials added in shared memory: no split-K region
    assert_close(c, oracle_full(case, inp), case.name)
    if cl > 1:
        c2, g2, _ = run_case(case, inp, num_sms=148, gemm=g)
        assert np.array_equal(c, c2), "cluster split-K is not reproducible"
    g.close()


def test_cluster_split_agrees_with_workspace_split():
    m = lib()
    case = _case(64, 4096, 8192, 16, dist=("normal", 1.0))
    inp = wl.make_inputs(case, seed=3)
    c1, g1, _ = run_case(case, inp, num_sms=148)
    assert g1.info.cluster_size > 1
    old = os.environ.get("LGT_GEMM_CLUSTER")
    os.environ["LGT_GEMM_CLUSTER"] = "0"
    try:
        g0 = m.Gemm(desc_for(m, case, 148))
    finally:
        if old is None:
            del os.environ["LGT_GEMM_CLUSTER"]
        else:
            os.environ["LGT_GEMM_CLUSTER"] = old
    assert g0.info.cluster_size == 0
    c0, _, _ = run_case(case, inp, num_sms=148, gemm=g0)
    ref = oracle_full(case, inp)
    assert_close(c0, ref, "workspace split")
    assert_close(c1, ref, "cluster split")
    # both round fp32 sums that differ only in summation order: they agree
    # to about a bf16 ulp of the result's scale
    assert np.linalg.norm(c1 - c0) <= 2 ** -8 * np.linalg.norm(ref)
    assert np.max(np.abs(c1 - c0)) <= 2 ** -7 * np.max(np.abs(ref))
    g0.close()
    g1.close()


def test_cluster_split_full_size_skinny():
    """The 64 x 4096 x 16384 skinny workload (split 128 by the SM-waste rule
    at 148 SMs) takes the cluster path on this GPU; every output checked."""
    case = wl.SKINNY_SPLITK
    inp = wl.make_inputs(case, seed=0)
    c, g, _ = run_case(case, inp, num_sms=148)
    assert g.info.split_k == 128 and g.info.cluster_size == 4
    assert_close(c, oracle_full(case, inp), case.name)
    g.close()
