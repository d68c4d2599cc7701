"""Seeded synthetic inputs for the any-layout GEMM.

This module is shared by the tests, the benchmark and the CPU oracle's
checks.  It only *draws* storage buffers (random values of a given dtype,
laid out with a given leading dimension) and describes the workloads; it
holds none of the GEMM arithmetic, no layout decoding and no dequantisation.

Storage conventions (the library's operand layouts):

* A is logically M x K.  ``K_CONTIG``: M rows of ``lda >= K`` elements
  (row-major M x K).  ``MN_CONTIG``: K rows of ``lda >= M`` elements
  (column-major M x K).
* B is logically K x N.  ``K_CONTIG``: N rows of ``ldb >= K`` elements
  (B stored N x K).  ``MN_CONTIG``: K rows of ``ldb >= N`` elements
  (row-major K x N).
* C is M rows of ``ldc >= N`` elements (row-major M x N).
* int4 weights: N rows of K/2 bytes, two codes per byte.  Uniform codes in
  both nibbles are exactly uniform random bytes, so the generator draws
  bytes and never packs anything.

Padding between a row's logical end and the leading dimension is filled with
NaN so that any read of it shows up in the results.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

K_CONTIG = 0
MN_CONTIG = 1

F16 = 0
BF16 = 1
INT4 = 2
F32 = 3

TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}
DTYPE_NAME = {F16: "f16", BF16: "bf16", INT4: "int4", F32: "f32"}


@dataclasses.dataclass(frozen=True)
class GemmCase:
    """One GEMM problem: shapes, layouts, dtypes and the value recipe."""

    name: str
    M: int
    N: int
    K: int
    a_layout: int
    b_layout: int
    a_dtype: int
    b_dtype: int
    c_dtype: int
    a_dist: tuple          # ("uniform", lo, hi) | ("normal", std)
    b_dist: tuple          # same; for INT4 weights: ("bytes",)
    split_k: int = 1       # 0 = auto (SM-waste rule)
    lda: int = 0           # 0 = dense
    ldb: int = 0
    ldc: int = 0
    group_size: int = 128  # int4 only
    scale_dist: tuple = ("uniform", 0.005, 0.02)
    zero_value: Optional[float] = 8.0   # None -> pass a NULL zeros pointer

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def dense_ld(self):
        lda = self.lda or (self.K if self.a_layout == K_CONTIG else self.M)
        if self.b_dtype == INT4:
            ldb = self.K // 2
        else:
            ldb = self.ldb or (self.K if self.b_layout == K_CONTIG else self.N)
        ldc = self.ldc or self.N
        return lda, ldb, ldc


def _layout_name(op, layout):
    if op == "a":
        return "a-kcontig" if layout == K_CONTIG else "a-mcontig"
    return "b-kcontig" if layout == K_CONTIG else "b-ncontig"


def case_name(dtype, M, N, K, a_layout, b_layout, extra=""):
    s = f"gemm_{DTYPE_NAME[dtype]}_m{M}_n{N}_k{K}_{_layout_name('a', a_layout)}_{_layout_name('b', b_layout)}"
    return s + (f"_{extra}" if extra else "")


def small_layout_cases():
    """fp16 256^3 in all four layout combinations, U[-1,1], split 1."""
    out = []
    for al in (K_CONTIG, MN_CONTIG):
        for bl in (K_CONTIG, MN_CONTIG):
            out.append(GemmCase(case_name(F16, 256, 256, 256, al, bl), 256, 256, 256, al, bl,
                                F16, F16, F16, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), split_k=1))
    return out


SQUARE_BF16 = GemmCase(case_name(BF16, 4096, 4096, 4096, K_CONTIG, MN_CONTIG), 4096, 4096, 4096,
                       K_CONTIG, MN_CONTIG, BF16, BF16, BF16, ("normal", 1.0), ("normal", 1.0), split_k=1)

SKINNY_SPLITK = GemmCase(case_name(BF16, 64, 4096, 16384, K_CONTIG, K_CONTIG, "splitk-auto"), 64, 4096, 16384,
                         K_CONTIG, K_CONTIG, BF16, BF16, BF16, ("normal", 0.1), ("normal", 0.1), split_k=0)

IRREGULAR = GemmCase(case_name(BF16, 4095, 3000, 2880, MN_CONTIG, MN_CONTIG), 4095, 3000, 2880,
                     MN_CONTIG, MN_CONTIG, BF16, BF16, BF16, ("uniform", -2.0, 2.0), ("uniform", -2.0, 2.0),
                     split_k=1)

INT4_DEQUANT = GemmCase("gemm_int4w_m16_n16384_k16384_a-kcontig_b-kcontig_g128_splitk-auto", 16, 16384, 16384,
                        K_CONTIG, K_CONTIG, F16, INT4, F16, ("normal", 1.0), ("bytes",), split_k=0)

# The five workloads of the benchmark table, in order.
WORKLOADS = small_layout_cases() + [SQUARE_BF16, SKINNY_SPLITK, IRREGULAR, INT4_DEQUANT]


def _draw(n, dist, dtype, gen):
    kind = dist[0]
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        x = torch.rand(n, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    elif kind == "normal":
        x = torch.randn(n, generator=gen, dtype=torch.float32) * dist[1]
    elif kind == "ones":
        x = torch.ones(n, dtype=torch.float32)
    elif kind == "ints":
        x = torch.randint(dist[1], dist[2] + 1, (n,), generator=gen).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist}")
    return x.to(TORCH_DTYPE[dtype])


def strided_matrix(rows, row_len, ld, dist, dtype, gen):
    """A flat storage buffer of ``rows`` rows of ``row_len`` drawn values at
    stride ``ld``; padding columns hold NaN.  Returns a 1-D CPU tensor of
    ``rows * ld`` elements (the last row's padding is included so every row
    has the same length)."""
    assert ld >= row_len
    vals = _draw(rows * row_len, dist, dtype, gen).view(rows, row_len)
    if ld == row_len:
        return vals.reshape(-1).contiguous()
    buf = torch.full((rows, ld), float("nan"), dtype=TORCH_DTYPE[dtype])
    buf[:, :row_len] = vals
    return buf.reshape(-1).contiguous()


@dataclasses.dataclass
class GemmInputs:
    """Host (CPU) storage for one case. ``A``/``B`` are flat tensors in the
    case's layout; for int4, ``B`` is uint8 [N * K/2] and ``scales``/``zeros``
    are fp16 [N, K/group]."""

    case: GemmCase
    A: torch.Tensor
    B: torch.Tensor
    lda: int
    ldb: int
    ldc: int
    scales: Optional[torch.Tensor] = None
    zeros: Optional[torch.Tensor] = None


def make_inputs(case: GemmCase, seed: int = 0) -> GemmInputs:
    gen = torch.Generator().manual_seed(1_000_003 * seed + 17)
    lda, ldb, ldc = case.dense_ld()
    M, N, K = case.M, case.N, case.K
    if case.a_layout == K_CONTIG:
        A = strided_matrix(M, K, lda, case.a_dist, case.a_dtype, gen)
    else:
        A = strided_matrix(K, M, lda, case.a_dist, case.a_dtype, gen)
    scales = zeros = None
    if case.b_dtype == INT4:
        assert K % 2 == 0 and K % case.group_size == 0
        B = torch.randint(0, 256, (N * (K // 2),), generator=gen, dtype=torch.uint8)
        G = K // case.group_size
        scales = _draw(N * G, case.scale_dist, F16, gen).view(N, G).contiguous()
        if case.zero_value is not None:
            zeros = torch.full((N, G), case.zero_value, dtype=torch.float16)
    elif case.b_layout == K_CONTIG:
        B = strided_matrix(N, K, ldb, case.b_dist, case.b_dtype, gen)
    else:
        B = strided_matrix(K, N, ldb, case.b_dist, case.b_dtype, gen)
    return GemmInputs(case, A, B, lda, ldb, ldc, scales, zeros)


def sample_indices(M, N, count, seed=0):
    """Seeded (row, col) sample of output positions.  It always includes the
    four corners and the last eight positions of the last row and column
    (the ragged tails)."""
    gen = torch.Generator().manual_seed(seed + 99)
    r = torch.randint(0, M, (count,), generator=gen).tolist()
    c = torch.randint(0, N, (count,), generator=gen).tolist()
    fixed = [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]
    fixed += [(M - 1, max(0, N - 1 - j)) for j in range(8)]
    fixed += [(max(0, M - 1 - j), N - 1) for j in range(8)]
    rows = [p[0] for p in fixed] + r
    cols = [p[1] for p in fixed] + c
    import numpy as np
    return np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64)


def ceil_div(a, b):
    return -(-a // b)


def storage_elems(rows, ld):
    return rows * ld


# ---------------------------------------------------------------------------
# fp32 row reductions (the IREE page's multi_reduction cases)
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ReduceCase:
    """out[r] = sum of row r of a rows x cols fp32 matrix (row pitch ldx,
    0 = cols) with values drawn from ``dist``."""
    name: str
    rows: int
    cols: int
    dist: tuple = ("normal", 1.0)
    ldx: int = 0

    def pitch(self):
        return self.ldx or self.cols


# The IREE page's two verification cases (4096 -> 1 and 4 x 4096 -> 4), and
# a 1 GiB matrix (larger than L2) for the bandwidth measurement.
REDUCE_VEC = ReduceCase("reduce_f32_4096_to_1", 1, 4096)
REDUCE_ROWS = ReduceCase("reduce_f32_4x4096_to_4", 4, 4096)
REDUCE_LARGE = ReduceCase("reduce_f32_16384x16384_to_16384", 16384, 16384)


def make_reduce_input(case: ReduceCase, seed: int = 0) -> torch.Tensor:
    """Flat CPU fp32 storage of ``rows * pitch`` elements (NaN padding)."""
    gen = torch.Generator().manual_seed(1_000_003 * seed + 29)
    return strided_matrix(case.rows, case.cols, case.pitch(), case.dist, F32, gen)



# ---------------------------------------------------------------------------
# fused attention (the second product P.V with V contiguous along d)
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class AttnCase:
    """O = softmax(Q K^T * scale) V per head; Q (heads x sq x d), K and V
    (heads x sk x d), O (heads x sq x d), all [head][row][d] contiguous, with
    values drawn from ``dist``.  scale 0: 1 / sqrt(d)."""
    name: str
    heads: int
    sq: int
    sk: int
    d: int
    dtype: int = BF16
    dist: tuple = ("normal", 1.0)
    scale: float = 0.0

    def flops(self):
        return 4.0 * self.heads * self.sq * self.sk * self.d


def attn_case(heads, sq, sk, d, dtype=BF16, dist=("normal", 1.0), scale=0.0, extra=""):
    nm = f"attn_{DTYPE_NAME[dtype]}_h{heads}_sq{sq}_sk{sk}_d{d}" + (f"_{extra}" if extra else "")
    return AttnCase(nm, heads, sq, sk, d, dtype, dist, scale)


# 32 heads (e.g. batch 4 x 8 heads) of 4096 queries and keys, head dim 128.
ATTN_BF16 = attn_case(32, 4096, 4096, 128, BF16)


def make_attn_inputs(case: AttnCase, seed: int = 0):
    """(Q, K, V) as flat CPU tensors."""
    gen = torch.Generator().manual_seed(1_000_003 * seed + 43)
    q = _draw(case.heads * case.sq * case.d, case.dist, case.dtype, gen)
    k = _draw(case.heads * case.sk * case.d, case.dist, case.dtype, gen)
    v = _draw(case.heads * case.sk * case.d, case.dist, case.dtype, gen)
    return q, k, v
