"""CPU tests of the C-ABI library: it loads, exports every entry point the
header declares, and its host-side integer logic (split-K rule, perpDim
permutation, magic division, planner decisions, argument validation) agrees
bit-exactly with the oracle and with plain integer division.  No GPU work."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import helpers
    return helpers.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*((?:gemm|reduce|attn)_[a-z0-9_]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"gemm_create", "gemm_run", "gemm_destroy", "gemm_workspace_size"} <= declared
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(raw, name), f"libgemm.so does not export {name}"
    assert set(lib.EXPORTS) == declared


def test_status_strings(lib):
    for code in range(7):
        assert lib.gemm_status_string(code).startswith("GEMM_")


def test_splitk_rule_matches_oracle(lib, golden_dir):
    rng = np.random.default_rng(3)
    for _ in range(5000):
        M, N, K = (int(x) for x in rng.integers(1, 70000, 3))
        sms = int(rng.integers(1, 300))
        bm, bn = int(rng.choice([64, 128, 256])), int(rng.choice([64, 128, 256]))
        bk = int(rng.choice([32, 64, 128]))
        assert lib.gemm_splitk_auto(M, N, K, bm, bn, bk, sms, 0.05) == \
            oracle.splitk_factor(M, N, K, bm, bn, bk, sms, 0.05)
    for line in open(os.path.join(golden_dir, "splitk_traces.txt")):
        if line.strip() and not line.startswith("#"):
            head, want = line.split("->")
            M, N, K, sms = map(int, head.split()[:4])
            assert lib.gemm_splitk_auto(M, N, K, 128, 128, 64, sms, 0.05) == int(want)


def test_perm_matches_oracle(lib):
    for B in range(1, 129):
        for S in range(1, B + 1):
            if B % S:
                continue
            count = 3 * B + B // 2          # two full blocks and a partial tail
            want = oracle.perm_apply(count, B, S)
            got = [lib.gemm_perm_fwd(i, count, B, S) for i in range(count)]
            assert got == want, (B, S)
            assert [lib.gemm_perm_inv(v, count, B, S) for v in got] == list(range(count))


def test_magic_division_bit_exact(lib):
    divisors = [1, 2, 3, 5, 7, 31, 64, 128, 148, 152, 1000, 3000, 4095, 65537, 1 << 20, (1 << 31) - 1, 1 << 30,
                12345679]
    rng = np.random.default_rng(9)
    top = 1 << 31
    for d in divisors:
        parts = [np.arange(0, 1 << 20, dtype=np.uint32),
                 np.arange(top - (1 << 20), top, dtype=np.uint32),
                 rng.integers(0, top, 1 << 20, dtype=np.uint32)]
        ks = np.arange(1, min(top // d, 1 << 16), dtype=np.uint64) if d > 1 else np.arange(1, 10, dtype=np.uint64)
        edges = np.concatenate([ks * d - 1, ks * d, ks * d + 1])
        parts.append(edges[edges < top].astype(np.uint32))
        n = np.concatenate(parts)
        q, r = lib.gemm_magic_divmod_host(n, d)
        assert np.array_equal(q, n // np.uint32(d)), d
        assert np.array_equal(r, n % np.uint32(d)), d
    # exhaustive over the full 31-bit range for one small divisor, in chunks
    d = 148
    for start in range(0, top, 1 << 27):
        n = np.arange(start, start + (1 << 27), dtype=np.uint32)
        q, r = lib.gemm_magic_divmod_host(n, d)
        assert np.array_equal(q, n // np.uint32(d))


def test_magic_division_rejects_out_of_range(lib):
    with pytest.raises(lib.GemmError):
        lib.gemm_magic_divmod_host(np.array([1 << 31], dtype=np.uint32), 3)
    with pytest.raises(lib.GemmError):
        lib.gemm_magic_divmod_host(np.array([5], dtype=np.uint32), 0)


def _plan_for(lib, case, num_sms=148):
    lda, ldb, ldc = case.dense_ld()
    desc = lib.make_desc(case.M, case.N, case.K, case.a_layout, case.b_layout, case.a_dtype, case.b_dtype,
                         case.c_dtype, lda=case.lda, ldb=case.ldb, ldc=case.ldc, split_k=case.split_k,
                         num_sms=num_sms)
    st, h = lib.gemm_create_status(desc)
    return st, h


@pytest.mark.parametrize("case", [c for c in wl.WORKLOADS if c.b_dtype != wl.INT4], ids=lambda c: c.name)
def test_planner_decisions(lib, case):
    st, h = _plan_for(lib, case)
    assert st == lib.GEMM_OK
    try:
        info = lib.gemm_query(h)
        want_split = case.split_k or oracle.splitk_factor(case.M, case.N, case.K, 128, 128, 64, 148)
        assert info.split_k == want_split
        assert info.swap_ab == (1 if case.M <= 64 else 0)
        lda, ldb, _ = case.dense_ld()
        # unaligned leading dimensions are repacked first (the in-kernel
        # realigning loader is opt-in)
        assert info.realign == 0
        assert info.repack_a == ((lda * 2) % 16 != 0)
        assert info.repack_b == ((ldb * 2) % 16 != 0)
        ws = lib.gemm_workspace_size(h)
        if info.split_k > 1:
            assert ws >= case.M * case.N * 4
        if info.repack_a:
            assert ws >= (case.K * ((case.M + 7) // 8 * 8) * 2 if case.a_layout == wl.MN_CONTIG
                          else case.M * ((case.K + 7) // 8 * 8) * 2)
        # K blocks per split follow Ks = ceil(K / (f * 64)) * 64
        assert info.k_per_split == -(-case.K // (info.split_k * 64)) * 64
    finally:
        lib.gemm_destroy(h)


def test_planner_int4(lib):
    case = wl.INT4_DEQUANT
    desc = lib.make_desc(case.M, case.N, case.K, a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_INT4, c_dtype=lib.GEMM_F16,
                         split_k=0, group_size=128, num_sms=148)
    h = lib.gemm_create(desc)
    info = lib.gemm_query(h)
    assert info.kernel == 1 and info.swap_ab == 1 and info.split_k == 32
    assert info.tile_m == 16 and info.tile_n == 128 and info.k_per_split == 512
    assert info.dequant_form == 1
    assert lib.gemm_workspace_size(h) >= case.M * case.N * 4
    lib.gemm_destroy(h)
    bad = [dict(group_size=96), dict(group_size=512, K=768), dict(a_dtype=lib.GEMM_BF16)]
    for kw in bad:
        args = dict(M=16, N=256, K=1024, a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_INT4, c_dtype=lib.GEMM_F16,
                    num_sms=148)
        args.update(kw)
        st, h = lib.gemm_create_status(lib.make_desc(**args))
        assert st == lib.GEMM_ERR_INVALID_ARG, kw
    st, h = lib.gemm_create_status(lib.make_desc(16, 256, 1024, a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_INT4,
                                                 c_dtype=lib.GEMM_F16, ldb=520, num_sms=148))
    assert st == lib.GEMM_ERR_UNSUPPORTED


def test_planner_int4_form(lib, monkeypatch):
    """Plans take the fp16 form unless LGT_GEMM_INT4_FORM=e4m3 asks for the
    e4m3 form, which needs at most 16 activation rows, a K-contiguous
    activation, K and the group multiples of 128 and splits of whole 128-deep
    blocks (everything else stays on the fp16 form)."""
    def form(M, N, K, group=128, split=1, a_layout=wl.K_CONTIG):
        d = lib.make_desc(M, N, K, a_layout=a_layout, a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_INT4,
                          c_dtype=lib.GEMM_F16, split_k=split, group_size=group, num_sms=148)
        h = lib.gemm_create(d)
        f = lib.gemm_query(h).dequant_form
        lib.gemm_destroy(h)
        return f
    assert form(16, 512, 1024) == 1 and form(1, 256, 128) == 1
    monkeypatch.setenv("LGT_GEMM_INT4_FORM", "e4m3")
    assert form(16, 512, 1024) == 2 and form(1, 256, 128) == 2 and form(9, 300, 2048, 256, 2) == 2
    assert form(17, 512, 1024) == 1                        # more than 16 activation rows
    assert form(16, 512, 1024, group=64) == 1              # group below 128
    assert form(16, 512, 1024, a_layout=wl.MN_CONTIG) == 1  # M-contiguous activation
    assert form(16, 512, 2048, split=7) == 1               # splits of 5 K blocks: not whole 128-deep blocks
    assert form(16, 512, 192 * 4, group=192) == 1          # group not a multiple of 128
    monkeypatch.setenv("LGT_GEMM_INT4_FORM", "fp16")
    assert form(16, 512, 1024) == 1
    h = lib.gemm_create(lib.make_desc(256, 256, 256, num_sms=148))
    assert lib.gemm_query(h).dequant_form == 0
    lib.gemm_destroy(h)


def test_planner_int4_prepacked(lib, monkeypatch):
    """GEMM_FLAG_INT4_PREPACKED: int4 plans only, the fp16 form (also when
    the e4m3 form is asked for), groups of 64 or 128 or multiples of 256,
    split ranges of whole 256-deep stages; the packed size is one block of
    codes and scale slots per 128-row tile and 256-deep stage."""
    monkeypatch.setenv("LGT_GEMM_INT4_FORM", "e4m3")
    base = dict(a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_INT4, c_dtype=lib.GEMM_F16, num_sms=148,
                flags=lib.GEMM_FLAG_INT4_PREPACKED, group_size=128)
    h = lib.gemm_create(lib.make_desc(16, 16384, 16384, split_k=0, **base))
    info = lib.gemm_query(h)
    assert info.dequant_form == 1 and info.split_k == 32 and (info.k_per_split // 64) % 4 == 0
    lib.gemm_destroy(h)
    # the rule's split ranges rounded up to whole 256-deep stages
    for M, N, K in [(16, 384, 8192), (16, 700, 4096), (1, 128, 640), (16, 4096, 2048)]:
        d = lib.make_desc(M, N, K, split_k=0, **base)
        h = lib.gemm_create(d)
        info = lib.gemm_query(h)
        lib.gemm_destroy(h)
        kb = -(-K // 64)
        rule = lib.gemm_splitk_auto(M, N, K, 128, 128, 64, 148, 0.05)
        want_kbps = -(-kb // rule)
        if rule > 1:
            want_kbps = -(-want_kbps // 4) * 4
        assert info.k_per_split == want_kbps * 64, (M, N, K)
        assert info.split_k == -(-kb // want_kbps), (M, N, K)
    for kw in [dict(M=16, N=512, K=2048, split_k=7), dict(M=16, N=512, K=768, group_size=192)]:
        args = dict(base)
        args.update(kw)
        st, _ = lib.gemm_create_status(lib.make_desc(**args))
        assert st == lib.GEMM_ERR_UNSUPPORTED, kw
    st, _ = lib.gemm_create_status(lib.make_desc(256, 256, 256, num_sms=148, flags=lib.GEMM_FLAG_INT4_PREPACKED))
    assert st == lib.GEMM_ERR_UNSUPPORTED
    for N, K, g in [(16384, 16384, 128), (300, 640, 64), (130, 1280, 256), (1, 512, 512)]:
        slots = 256 // g if g < 256 else 1
        assert lib.gemm_int4_prepack_bytes(N, K, g) == -(-N // 128) * -(-K // 256) * (128 * 128 + slots * 256)
    for N, K, g in [(0, 256, 128), (256, 0, 128), (256, 768, 192), (256, 100, 64), (256, 640, 256), (256, 1024, -256),
                    (256, 1024, -64), (1 << 31, 512, 128), (256, 1 << 32, 128)]:
        assert lib.gemm_int4_prepack_bytes(N, K, g) == 0, (N, K, g)
    # null pointers are refused before any launch
    assert lib.gemm_int4_prepack(0, 0, 0, 256, 1024, 128, 0) == lib.GEMM_ERR_INVALID_ARG


def test_planner_skinny_and_irregular_factors(lib):
    # the SM-waste rule's values at 148 SMs for the skinny bf16 and int4-shaped problems
    desc = lib.make_desc(64, 4096, 16384, split_k=0, num_sms=148)
    h = lib.gemm_create(desc)
    info = lib.gemm_query(h)
    assert info.split_k == 128
    import torch
    if not torch.cuda.is_available():
        # split-K inside clusters needs the device's cluster occupancy: never without one
        assert info.cluster_size == 0
        assert lib.gemm_workspace_size(h) >= 64 * 4096 * 4
    lib.gemm_destroy(h)
    desc = lib.make_desc(4095, 3000, 2880, wl.MN_CONTIG, wl.MN_CONTIG, split_k=0, num_sms=160)
    h = lib.gemm_create(desc)
    assert lib.gemm_query(h).split_k == 4
    lib.gemm_destroy(h)


def test_invalid_arguments(lib):
    bad = [
        lib.make_desc(-1, 4, 4, num_sms=148),
        lib.make_desc(4, 4, 4, a_layout=2, num_sms=148),
        lib.make_desc(4, 4, 4, lda=3, num_sms=148),
        lib.make_desc(4, 4, 4, a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_BF16, num_sms=148),
        lib.make_desc(4, 4, 4, c_dtype=lib.GEMM_F32, num_sms=148),
        lib.make_desc(4, 4, 4, flags=2, num_sms=148),
        lib.make_desc(4, 4, 4, split_k=-2, num_sms=148),
        lib.make_desc(4, 4, 4, a_dtype=lib.GEMM_BF16, b_dtype=lib.GEMM_INT4, c_dtype=lib.GEMM_F16, num_sms=148),
    ]
    for d in bad:
        st, h = lib.gemm_create_status(d)
        assert st == lib.GEMM_ERR_INVALID_ARG and h is None
    assert lib._lib.gemm_create(None, None) == lib.GEMM_ERR_INVALID_ARG
    assert lib._lib.gemm_query(None, None) == lib.GEMM_ERR_INVALID_ARG


def test_deterministic_flag(lib):
    # accepted with or without a K split (per-run partial slots replace the
    # fp32 atomics); never a stream-K tail
    h = lib.gemm_create(lib.make_desc(512, 512, 512, flags=lib.GEMM_FLAG_DETERMINISTIC, num_sms=148))
    info = lib.gemm_query(h)
    assert info.split_k == 1 and info.streamk_tiles == 0
    lib.gemm_destroy(h)
    h = lib.gemm_create(lib.make_desc(512, 512, 4096, split_k=4, flags=lib.GEMM_FLAG_DETERMINISTIC, num_sms=148))
    assert lib.gemm_query(h).split_k == 4
    lib.gemm_destroy(h)


def test_withhold_flag_only_where_no_cta_waits_on_another(lib):
    """The failure-path test aid is accepted only for plans whose CTAs never
    wait on each other (single-CTA kernel, whole tiles)."""
    W = lib.GEMM_FLAG_TEST_WITHHOLD_STAGE
    h = lib.gemm_create(lib.make_desc(256, 256, 256, a_dtype=lib.GEMM_F16, split_k=1, flags=W, num_sms=148))
    info = lib.gemm_query(h)
    assert info.kernel == 0 and info.split_k == 1 and info.streamk_tiles == 0
    lib.gemm_destroy(h)
    for d in (lib.make_desc(256, 256, 4096, split_k=4, flags=W, num_sms=148),
              lib.make_desc(16, 256, 1024, a_dtype=lib.GEMM_F16, b_dtype=lib.GEMM_INT4, c_dtype=lib.GEMM_F16,
                            flags=W, num_sms=148)):
        st, h = lib.gemm_create_status(d)
        assert st == lib.GEMM_ERR_UNSUPPORTED and h is None
    st, h = lib.gemm_create_status(lib.make_desc(256, 256, 256, flags=W | 8, num_sms=148))
    assert st == lib.GEMM_ERR_INVALID_ARG


def test_no_device_paths(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    st, h = lib.gemm_create_status(lib.make_desc(128, 128, 128, num_sms=0))
    assert st == lib.GEMM_ERR_CUDA and h is None
    h = lib.gemm_create(lib.make_desc(128, 128, 128, num_sms=148))
    assert lib.gemm_run(h, 16, 16, 16) == lib.GEMM_ERR_CUDA
    lib.gemm_destroy(h)


def test_reduce_host_checks(lib):
    """Workspace sizing and argument checks of the row reduction (host only)."""
    assert lib.reduce_rows_workspace_size(1, 4096, 148) == 0       # the IREE page's cases: one CTA a row
    assert lib.reduce_rows_workspace_size(4, 4096, 148) == 0
    assert lib.reduce_rows_workspace_size(16384, 16384, 148) == 0  # rows fill the GPU
    n = lib.reduce_rows_workspace_size(1, 1 << 22, 148)            # one long row: split across CTAs
    assert n >= 148 * 4 * 4 + 4
    assert lib.reduce_rows_workspace_size(0, 5, 148) == 0
    with pytest.raises(lib.GemmError):
        lib.reduce_rows_workspace_size(-1, 5, 148)
    F = lib.reduce_rows_f32
    assert F(4096, -1, 4, 0, 4096) == lib.GEMM_ERR_INVALID_ARG
    assert F(4096, 2, 8, 7, 4096) == lib.GEMM_ERR_INVALID_ARG       # ldx < cols
    assert F(0, 2, 8, 0, 4096) == lib.GEMM_ERR_INVALID_ARG          # NULL x
    assert F(4098, 2, 8, 0, 4096) == lib.GEMM_ERR_ALIGNMENT         # x not 4-byte aligned
    assert F(4096, 2, 8, 0, 4097) == lib.GEMM_ERR_ALIGNMENT         # out not 4-byte aligned
    assert F(4096, 0, 8, 0, 0) == lib.GEMM_OK                       # no rows: nothing to do


def test_reduce_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert lib.reduce_rows_f32(4096, 2, 8, 0, 4096) == lib.GEMM_ERR_CUDA
    st = lib._lib.reduce_rows_workspace_size(2, 8, 0, ctypes.byref(ctypes.c_size_t()))
    assert st == lib.GEMM_ERR_CUDA


def test_planner_realign_or_repack(lib, monkeypatch):
    """With LGT_GEMM_REALIGN=1 an unaligned leading dimension is realigned
    inside the kernel when the plan leaves the fixup warps free (no split-K
    through the workspace, no stream-K tail); else, and by default, it is
    repacked first."""
    def info(M, N, K, lda, split=1, al=wl.MN_CONTIG):
        d = lib.make_desc(M, N, K, al, wl.K_CONTIG, lib.GEMM_BF16, lda=lda, split_k=split, num_sms=148)
        h = lib.gemm_create(d)
        i = lib.gemm_query(h)
        ws = lib.gemm_workspace_size(h)
        lib.gemm_destroy(h)
        return i, ws
    i, ws = info(4095, 3000, 2880, 4095)   # pitch 8190 bytes: the default repacks
    assert i.realign == 0 and i.repack_a == 1 and ws >= 2880 * 4096 * 2
    monkeypatch.setenv("LGT_GEMM_REALIGN", "1")
    i, ws = info(4095, 3000, 2880, 4095)
    assert i.realign == 1 and i.repack_a == 0 and i.streamk_tiles == 0 and ws == 0
    i, _ = info(4095, 3000, 2880, 4096)    # aligned pitch: the same plan, nothing to realign
    assert i.realign == 1 and i.repack_a == 0
    i, ws = info(300, 400, 4096, 301, split=4)  # split-K through the workspace: pre-pass
    assert i.realign == 0 and i.repack_a == 1 and ws >= 4096 * 304 * 2


def test_attention_descriptor_checks(lib):
    """attn_create refuses shapes and types outside the header's contract
    before it touches a device."""
    bad = [dict(heads=0), dict(heads=70000), dict(seq_q=0), dict(seq_k=0), dict(head_dim=96), dict(head_dim=256),
           dict(dtype=lib.GEMM_F32), dict(scale=-1.0), dict(scale=float("inf")), dict(scale=float("nan"))]
    for kw in bad:
        args = dict(heads=2, seq_q=128, seq_k=128, head_dim=64, dtype=lib.GEMM_BF16, scale=0.0)
        args.update(kw)
        st, h = lib.attn_create_status(lib.attn_desc_t(**args))
        assert st == lib.GEMM_ERR_INVALID_ARG and h is None, kw


def test_binding_refuses_host_tensors(lib):
    """A host tensor's address never reaches a kernel or a tensor map: every
    run method of the binding raises before calling into the library."""
    import torch
    x = torch.zeros(64, dtype=torch.float16)
    g = object.__new__(lib.Gemm)
    g.plan, g.ws_bytes, g.workspace = None, 0, None
    with pytest.raises(ValueError, match="Gemm.run: A must be a CUDA tensor"):
        g.run(x, x, x)
    a = object.__new__(lib.Attention)
    a.plan = None
    with pytest.raises(ValueError, match="Attention.run: Q must be a CUDA tensor"):
        a.run(x, x, x, x)
    r = object.__new__(lib.RowReduce)
    r.rows, r.cols, r.ws_bytes, r.workspace = 1, 64, 0, None
    with pytest.raises(ValueError, match="RowReduce.run: x must be a CUDA tensor"):
        r.run(x.float(), torch.zeros(1))
    with pytest.raises(ValueError, match="int4_prepack: B must be a CUDA tensor"):
        lib.int4_prepack(torch.zeros(8, dtype=torch.uint8), x, 128, 256)
