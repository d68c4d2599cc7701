"""GPU parity of the fused attention forward (O = softmax(Q K^T scale) V per
head, the second product with V contiguous along head_dim: the non-TN second
dot of Flash Attention that the Triton inThreadTranspose page names) against
the fp64 oracle, through the C ABI.

Tolerance: elementwise |O - ref| <= 2e-2 (|ref| + 1) and a relative Frobenius
error of at most 2e-3 (fp16) or 4e-3 (bf16).  The kernel rounds the softmax
probabilities once to the input type for the second product and the output
once; each rounding is at most 2^-11 (fp16) or 2^-9 (bf16) relative per
term, so two of them stay below 2 x 2^-9 < 4e-3 for bf16, and the fp16 case
keeps the GEMM bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import lib

pytestmark = pytest.mark.gpu

F16, BF16 = wl.F16, wl.BF16


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


def _fro(dtype):
    return 2e-3 if dtype == F16 else 4e-3


def _run(case, q, k, v, reps=1):
    m = lib()
    a = m.Attention(case.heads, case.sq, case.sk, case.d, case.dtype, case.scale)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    O = torch.full((case.heads * case.sq * case.d,), float("nan"), dtype=wl.TORCH_DTYPE[case.dtype], device="cuda")
    for _ in range(reps):
        a.run(Q, K, V, O)
    assert a.sync_status() == m.GEMM_OK
    torch.cuda.synchronize()
    out = oracle.decode(O.cpu(), case.dtype).reshape(case.heads, case.sq, case.d)
    a.close()
    return out, O


def _check(out, ref, dtype, what):
    ok, viol, rel = oracle.check_close(out.reshape(-1, out.shape[-1]), ref.reshape(-1, ref.shape[-1]),
                                       fro_tol=_fro(dtype))
    assert ok, f"{what}: max elementwise violation {viol:.3g} (<=1), rel Frobenius {rel:.3g}"


@pytest.mark.parametrize("heads,sq,sk,d,dtype", [(1, 128, 128, 64, F16), (2, 128, 256, 128, F16),
                                                 (3, 200, 300, 128, F16), (2, 77, 1000, 64, BF16),
                                                 (1, 384, 129, 128, BF16), (2, 256, 640, 128, BF16),
                                                 (1, 130, 127, 64, F16)])
def test_attention_matches_oracle(heads, sq, sk, d, dtype):
    case = wl.attn_case(heads, sq, sk, d, dtype)
    q, k, v = wl.make_attn_inputs(case, seed=sq + sk)
    out, _ = _run(case, q, k, v)
    _check(out, oracle.attention(q, k, v, heads, sq, sk, d, dtype), dtype, case.name)


def test_attention_zero_queries_and_one_key():
    """Q = 0: the softmax is uniform and O is the mean of V's rows.  One key:
    O is V's row (probability 1, rounded exactly)."""
    case = wl.attn_case(2, 130, 300, 64, F16)
    _, k, v = wl.make_attn_inputs(case, seed=7)
    q = torch.zeros(case.heads * case.sq * case.d, dtype=torch.float16)
    out, _ = _run(case, q, k, v)
    vv = oracle.decode(v, F16).reshape(2, 300, 64)
    _check(out, np.repeat(vv.mean(axis=1)[:, None, :], 130, axis=1), F16, "zero queries")
    one = wl.attn_case(1, 128, 1, 128, BF16)
    q1, k1, v1 = wl.make_attn_inputs(one, seed=8)
    out1, _ = _run(one, q1, k1, v1)
    v1r = oracle.round_to(oracle.decode(v1, BF16).reshape(1, 1, 128), oracle.BF16)
    assert np.array_equal(out1, np.repeat(v1r, 128, axis=1))


def test_attention_peaked_softmax_rescales():
    """Logits of spread several tens: the running maximum moves between key
    blocks and the O accumulator is rescaled on the way."""
    case = wl.attn_case(2, 256, 1024, 128, F16, dist=("normal", 2.5), scale=0.5)
    q, k, v = wl.make_attn_inputs(case, seed=9)
    out, _ = _run(case, q, k, v)
    _check(out, oracle.attention(q, k, v, 2, 256, 1024, 128, F16, scale=0.5), F16, case.name)


def test_attention_repeats_bitwise_and_checks_alignment():
    m = lib()
    case = wl.attn_case(2, 256, 512, 128, BF16)
    q, k, v = wl.make_attn_inputs(case, seed=10)
    _, O1 = _run(case, q, k, v)
    _, O2 = _run(case, q, k, v, reps=3)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    a = m.Attention(2, 256, 512, 128, m.GEMM_BF16)
    Q = torch.zeros(case.heads * case.sq * case.d + 8, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros(case.heads * case.sk * case.d, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros(case.heads * case.sq * case.d, dtype=torch.bfloat16, device="cuda")
    assert m.attn_run(a.plan, Q.data_ptr() + 2, K.data_ptr(), K.data_ptr(), O.data_ptr()) == m.GEMM_ERR_ALIGNMENT
    assert m.attn_run(a.plan, Q.data_ptr(), K.data_ptr(), 0, O.data_ptr()) == m.GEMM_ERR_INVALID_ARG
    a.close()


def test_attention_full_size_sampled():
    """32 heads x 4096 queries x 4096 keys, head_dim 128, bf16: sampled rows
    (every head, first and last query tiles and the ragged-free middle)
    against the oracle one row at a time."""
    case = wl.ATTN_BF16
    q, k, v = wl.make_attn_inputs(case, seed=0)
    out, _ = _run(case, q, k, v)
    gen = np.random.default_rng(11)
    hs = gen.integers(0, case.heads, 48)
    rs = np.concatenate([[0, 127, 128, case.sq - 1], gen.integers(0, case.sq, 44)])
    ref = oracle.attention_rows(hs, rs, q, k, v, case.heads, case.sq, case.sk, case.d, BF16)
    _check(out[hs, rs], ref, BF16, case.name)
    assert np.all(np.isfinite(out))
