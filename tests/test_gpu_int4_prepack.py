"""Pre-packed int4 weights (gemm_int4_prepack + GEMM_FLAG_INT4_PREPACKED).

The BitBLAS page ("Relevant Issues") asks for a ladder-style basic layout of
the quantised weights, prepared offline, so that the dequantising producer
reads whole conflict-free vectors.  Here the layout is the kernel's own
stage: per 128-row tile and 256-deep stage, the swizzled codes and then the
stage's scales.  The packed bytes are pinned to the layout gemm.h states,
rebuilt here in numpy from that statement; the GEMM on packed weights must
give the same bits as on the plain layout (same expansion, same order), and
both stay within the oracle's tolerance."""
import numpy as np
import pytest
import torch

import helpers
import oracle
import workloads as wl
from helpers import assert_close, lib, oracle_full, oracle_sample

pytestmark = pytest.mark.gpu

K = wl.K_CONTIG


def _case(M, N, Kd, split=1, group=128, zero=8.0, name=""):
    nm = f"int4pre_m{M}_n{N}_k{Kd}_g{group}_s{split}{name}"
    return wl.GemmCase(nm, M, N, Kd, K, K, wl.F16, wl.INT4, wl.F16, ("normal", 1.0), ("bytes",), split_k=split,
                       group_size=group, zero_value=zero, scale_dist=("uniform", 0.005, 0.02))


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


def _expected_pack(B, scales, N, Kd, group, ldb):
    """The packed buffer as gemm.h describes it, from the plain weights."""
    S = -(-Kd // 256)
    T = -(-N // 128)
    slots = 256 // group if group < 256 else 1
    blk = 128 * 128 + slots * 128 * 2
    out = np.zeros((T, S, blk), dtype=np.uint8)
    G = Kd // group
    w = B.reshape(N, ldb)[:, : Kd // 2]
    sc = scales.reshape(N, G).view(np.uint16)
    for t in range(T):
        for s in range(S):
            codes = np.zeros((128, 128), dtype=np.uint8)
            rows = w[t * 128: min(N, t * 128 + 128), s * 128: s * 128 + 128]
            codes[: rows.shape[0], : rows.shape[1]] = rows
            sw = np.zeros_like(codes)
            for r in range(128):
                for c in range(8):
                    sw[r, (c ^ (r % 8)) * 16: (c ^ (r % 8)) * 16 + 16] = codes[r, c * 16: c * 16 + 16]
            out[t, s, : 128 * 128] = sw.reshape(-1)
            sl = np.zeros((slots, 128), dtype=np.uint16)
            for slot in range(slots):
                g = s * (256 // group) + slot if group < 256 else (s * 256) // group
                if g < G:
                    n1 = min(N, t * 128 + 128)
                    sl[slot, : n1 - t * 128] = sc[t * 128: n1, g]
            out[t, s, 128 * 128:] = sl.reshape(-1).view(np.uint8)
    return out.reshape(-1)


@pytest.mark.parametrize("N,Kd,group", [(300, 640, 64), (256, 1024, 128), (130, 1280, 256), (200, 1536, 512)])
def test_prepack_bytes_match_stated_layout(N, Kd, group):
    m = lib()
    case = _case(4, N, Kd, group=group)
    inp = wl.make_inputs(case, seed=N + Kd)
    nbytes = m.gemm_int4_prepack_bytes(N, Kd, group)
    slots = 256 // group if group < 256 else 1
    assert nbytes == -(-N // 128) * -(-Kd // 256) * (128 * 128 + slots * 256)
    packed = m.int4_prepack(inp.B.cuda(), inp.scales.cuda(), N, Kd, group)
    torch.cuda.synchronize()
    want = _expected_pack(inp.B.numpy(), inp.scales.numpy(), N, Kd, group, Kd // 2)
    got = packed.cpu().numpy()
    assert got.shape == want.shape
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


def test_prepack_padded_rows():
    """A row pitch beyond K / 2 (ldb a multiple of 16): only the first K / 2
    bytes of each row are taken."""
    m = lib()
    N, Kd, group, ldb = 260, 512, 128, 272
    case = _case(4, N, Kd, group=group)
    inp = wl.make_inputs(case, seed=5)
    Bp = torch.full((N, ldb), 0xAB, dtype=torch.uint8)
    Bp[:, : Kd // 2] = inp.B.reshape(N, Kd // 2)
    packed = m.int4_prepack(Bp.reshape(-1).cuda(), inp.scales.cuda(), N, Kd, group, ldb=ldb)
    want = _expected_pack(Bp.reshape(-1).numpy(), inp.scales.numpy(), N, Kd, group, ldb)
    assert np.array_equal(packed.cpu().numpy(), want)


def test_prepack_rejects():
    m = lib()
    B = torch.zeros(256 * 512, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(256 * 8, dtype=torch.float16, device="cuda")
    out = torch.zeros(m.gemm_int4_prepack_bytes(256, 1024, 128), dtype=torch.uint8, device="cuda")
    assert m.gemm_int4_prepack(B.data_ptr() + 8, 0, sc.data_ptr(), 256, 1024, 128, out.data_ptr()) == \
        m.GEMM_ERR_ALIGNMENT
    assert m.gemm_int4_prepack(B.data_ptr(), 520, sc.data_ptr(), 256, 1024, 128, out.data_ptr()) == \
        m.GEMM_ERR_ALIGNMENT
    assert m.gemm_int4_prepack(B.data_ptr(), 0, sc.data_ptr(), 256, 1024, 128, 0) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_int4_prepack(B.data_ptr(), 0, sc.data_ptr(), 256, 1024, 192, out.data_ptr()) == \
        m.GEMM_ERR_INVALID_ARG


def _run(case, inp, packed=None, det=True, reps=2, split=None):
    m = lib()
    d = helpers.desc_for(m, case, 148)
    if split is not None:
        d.split_k = split
    d.flags = (m.GEMM_FLAG_DETERMINISTIC if det else 0) | (m.GEMM_FLAG_INT4_PREPACKED if packed is not None else 0)
    g = m.Gemm(d)
    assert g.info.dequant_form == 1
    A = inp.A.cuda()
    B = packed if packed is not None else inp.B.cuda()
    sc = inp.scales.cuda()
    zr = inp.zeros.cuda() if inp.zeros is not None else None
    C = torch.full((case.M * inp.ldc,), float("nan"), dtype=torch.float16, device="cuda")
    for _ in range(reps):
        g.run(A, B, C, sc, zr)
    assert g.sync_status() == m.GEMM_OK
    torch.cuda.synchronize()
    info = g.info
    g.close()
    return C, info


@pytest.mark.parametrize("M,N,Kd,group,split", [(1, 128, 256, 128, 1), (16, 300, 640, 64, 1), (9, 700, 4096, 128, 4),
                                                (16, 384, 8192, 64, 0), (5, 260, 2048, 256, 2),
                                                (16, 256, 16384, 512, 0), (33, 640, 3072, 128, 3)])
def test_prepacked_same_bits_as_plain(M, N, Kd, group, split):
    m = lib()
    for zero in (8.0, None):
        case = _case(M, N, Kd, split=split, group=group, zero=zero)
        inp = wl.make_inputs(case, seed=M * 7 + N)
        packed = m.int4_prepack(inp.B.cuda(), inp.scales.cuda(), N, Kd, group)
        c_pre, info = _run(case, inp, packed)
        if split:
            assert info.split_k == split
        assert (info.k_per_split // 64) % 4 == 0 or info.split_k == 1
        # (the same split factor: an auto factor may have been rounded to
        # whole stages, and the factor fixes the order of the fp32 sums)
        c_plain, _ = _run(case, inp, split=info.split_k)
        assert torch.equal(c_pre.view(torch.int16), c_plain.view(torch.int16)), case.name
        c = oracle.decode(c_pre.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
        assert_close(c, oracle_full(case, inp), case.name)


def test_prepacked_full_size():
    """The 16 x 16384 x 16384 int4 workload on pre-packed weights: the same
    bits as the plain layout in deterministic mode, sampled against the
    oracle, and the same planner decisions."""
    m = lib()
    case = wl.INT4_DEQUANT
    inp = wl.make_inputs(case, seed=0)
    packed = m.int4_prepack(inp.B.cuda(), inp.scales.cuda(), case.N, case.K, case.group_size)
    c_pre, info = _run(case, inp, packed, reps=3)
    c_plain, info_plain = _run(case, inp)
    assert info.split_k == info_plain.split_k == oracle.splitk_factor(case.M, case.N, case.K, 128, 128, 64, 148)
    assert torch.equal(c_pre.view(torch.int16), c_plain.view(torch.int16))
    c = oracle.decode(c_pre.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
    rows, cols = wl.sample_indices(case.M, case.N, 1500, seed=4)
    assert_close(c[rows, cols], oracle_sample(case, inp, rows, cols), case.name)
    # without the deterministic flag: within tolerance as well
    c_nd, _ = _run(case, inp, packed, det=False)
    c2 = oracle.decode(c_nd.cpu(), case.c_dtype).reshape(case.M, inp.ldc)[:, : case.N]
    assert_close(c2[rows, cols], oracle_sample(case, inp, rows, cols), case.name + " (atomic)")
