"""Kernels are launched with programmatic stream serialization: the next
kernel's prologue may run while the previous kernel finishes, and each
kernel waits (griddepcontrol.wait) before touching global memory.  These
tests chain GEMMs in one stream with no synchronisation in between, each
reading the previous one's output, and compare the last result with the
oracle applied step by step (rounding each intermediate C as the GPU
stores it)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, lib

pytestmark = pytest.mark.gpu

K, MN = wl.K_CONTIG, wl.MN_CONTIG


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


def _rand(n, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, generator=g) * scale).to(wl.TORCH_DTYPE[dtype])


@pytest.mark.parametrize("M,N,split", [(256, 256, 1), (64, 1024, 0), (512, 768, 4)])
def test_chain_of_gemms_reading_previous_output(M, N, split):
    """C1 = A B1, C2 = C1 B2, C3 = C2 B3 (B2, B3 N x N, K-contiguous); one
    stream, no sync between launches."""
    m = lib()
    dt = wl.BF16
    Kd = 512
    A = _rand(M * Kd, dt, 1, 0.5)
    Bs = [_rand(N * Kd, dt, 2, 0.05)] + [_rand(N * N, dt, 3 + i, 0.05) for i in range(2)]
    plans = [m.Gemm(m.make_desc(M, N, Kd, K, K, dt, dt, dt, split_k=split, num_sms=148))]
    plans += [m.Gemm(m.make_desc(M, N, N, K, K, dt, dt, dt, split_k=split, num_sms=148)) for _ in range(2)]
    Cs = [torch.empty(M * N, dtype=wl.TORCH_DTYPE[dt], device="cuda") for _ in range(3)]
    Ad = A.cuda()
    Bd = [b.cuda() for b in Bs]
    torch.cuda.synchronize()
    for rep in range(3):  # repeated, so that each plan's workspace is reused right behind its last use
        plans[0].run(Ad, Bd[0], Cs[0])
        plans[1].run(Cs[0], Bd[1], Cs[1])
        plans[2].run(Cs[1], Bd[2], Cs[2])
    torch.cuda.synchronize()
    for p in plans:
        assert p.sync_status() == 0
    # each step against the oracle applied to the stored output of the
    # previous one (a kernel that read it before it was final would not match)
    ins = [A] + [Cs[i].cpu() for i in range(2)]
    ks = [Kd, N, N]
    for i in range(3):
        ref = oracle.gemm(M, N, ks[i], ins[i], K, ks[i], dt, Bs[i], K, ks[i], dt)
        got = oracle.decode(Cs[i].cpu(), dt).reshape(M, N)
        assert_close(got, ref, f"chain step {i} M={M} N={N} split={split}")
    for p in plans:
        p.close()


def test_int4_after_producer_kernel():
    """The int4 path's pre-pass reads an activation written by the kernel
    launched just before it (a torch fill), with no sync in between."""
    m = lib()
    M, N, Kd = 16, 512, 1024
    W = torch.randint(0, 256, (N * Kd // 2,), dtype=torch.uint8, generator=torch.Generator().manual_seed(5))
    s = (torch.rand(N * (Kd // 128), generator=torch.Generator().manual_seed(6)) * 0.01 + 0.005).to(torch.float16)
    g = m.Gemm(m.make_desc(M, N, Kd, K, K, wl.F16, wl.INT4, wl.F16, split_k=0, group_size=128, num_sms=148))
    Ad = torch.empty(M * Kd, dtype=torch.float16, device="cuda")
    C = torch.empty(M * N, dtype=torch.float16, device="cuda")
    Wd, sd = W.cuda(), s.cuda()
    torch.cuda.synchronize()
    for v in (0.25, -0.5, 1.0):
        Ad.fill_(v)  # a kernel writing A, then the GEMM reading it
        g.run(Ad, Wd, C, sd, None)
    torch.cuda.synchronize()
    assert g.sync_status() == 0
    A = torch.full((M * Kd,), 1.0, dtype=torch.float16)
    ref = oracle.gemm(M, N, Kd, A, K, Kd, wl.F16, W, K, 0, wl.INT4, scales=s, zeros=None, group=128)
    got = oracle.decode(C.cpu(), wl.F16).reshape(M, N)
    assert_close(got, ref, "int4 after a producer kernel")
    g.close()
