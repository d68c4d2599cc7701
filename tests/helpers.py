"""Shared test plumbing: run one case through the C ABI on the GPU and
compare with the oracle.  Marshalling only."""
import numpy as np
import torch

import oracle
import workloads as wl


def lib():
    import __graft_entry__
    __graft_entry__.build()
    import layout_general_tensor_gb300 as m
    return m


def desc_for(m, case, num_sms=148, lda=None, ldb=None, ldc=None):
    l_a, l_b, l_c = case.dense_ld()
    return m.make_desc(case.M, case.N, case.K, case.a_layout, case.b_layout, case.a_dtype, case.b_dtype,
                       case.c_dtype, lda=l_a if lda is None else lda, ldb=(0 if case.b_dtype == wl.INT4 else l_b)
                       if ldb is None else ldb, ldc=l_c if ldc is None else ldc, split_k=case.split_k,
                       group_size=case.group_size if case.b_dtype == wl.INT4 else 0, num_sms=num_sms)


def to_dev(t, offset_elems=0):
    """Copy a flat CPU tensor to the GPU, optionally at an element offset
    inside a larger allocation (to test base-pointer alignment)."""
    if offset_elems == 0:
        return t.cuda(), t.cuda()
    big = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device="cuda")
    view = big[offset_elems:]
    view.copy_(t.cuda())
    return view, big


def run_case(case, inputs, seed_offsets=(0, 0), num_sms=148, reps=1, gemm=None):
    """Returns (C as fp64 numpy M x N, the Gemm object, C storage)."""
    m = lib()
    g = gemm or m.Gemm(desc_for(m, case, num_sms))
    A, _ka = to_dev(inputs.A, seed_offsets[0])
    B, _kb = to_dev(inputs.B, seed_offsets[1])
    ldc = inputs.ldc
    C = torch.full((max(case.M, 1) * ldc,), float("nan"), dtype=wl.TORCH_DTYPE[case.c_dtype], device="cuda")
    sc = inputs.scales.cuda() if inputs.scales is not None else None
    zr = inputs.zeros.cuda() if inputs.zeros is not None else None
    ws, wsb = None, None
    if seed_offsets != (0, 0):
        wsb = max(g.ws_bytes, _misaligned_ws(m, g))
        ws = torch.zeros(max(wsb, 1), dtype=torch.uint8, device="cuda")
    for _ in range(reps):
        g.run(A, B, C, sc, zr, workspace=ws, workspace_bytes=wsb)
    st = g.sync_status()
    assert st == m.GEMM_OK, m.gemm_status_string(st)
    torch.cuda.synchronize()
    c = oracle.decode(C.cpu(), case.c_dtype).reshape(max(case.M, 1), ldc)[: case.M, : case.N]
    return c, g, C


def _misaligned_ws(m, g):
    # both operands repacked: rows * roundup(row, 8) * 2 each, plus the split-K region
    d = g.desc
    a_rows, a_row = (d.K, d.M) if d.a_layout == m.GEMM_MN_CONTIG else (d.M, d.K)
    b_rows, b_row = (d.K, d.N) if d.b_layout == m.GEMM_MN_CONTIG else (d.N, d.K)
    pad = lambda x: (x + 255) // 256 * 256
    return g.ws_bytes + pad(a_rows * ((a_row + 7) // 8 * 8) * 2) + pad(b_rows * ((b_row + 7) // 8 * 8) * 2)


def oracle_full(case, inputs):
    return oracle.gemm(case.M, case.N, case.K, inputs.A, case.a_layout, inputs.lda, case.a_dtype, inputs.B,
                       case.b_layout, inputs.ldb, case.b_dtype, scales=inputs.scales, zeros=inputs.zeros,
                       group=case.group_size)


def oracle_sample(case, inputs, rows, cols):
    return oracle.gemm_elements(rows, cols, case.M, case.N, case.K, inputs.A, case.a_layout, inputs.lda,
                                case.a_dtype, inputs.B, case.b_layout, inputs.ldb, case.b_dtype,
                                scales=inputs.scales, zeros=inputs.zeros, group=case.group_size)


def assert_close(c_gpu, c_ref, what=""):
    ok, viol, rel = oracle.check_close(c_gpu, c_ref)
    assert ok, f"{what}: max elementwise violation {viol:.3g} (<=1), rel Frobenius {rel:.3g} (<=2e-3)"
    return viol, rel
