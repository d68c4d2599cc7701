"""CPU oracle for the any-layout half-precision GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may call it.  It shares no code, table or constant with the CUDA path.

What it computes, and the passage each function follows:

* :func:`gemm` -- ``C[m,n] = sum_k a(m,k) * b(k,n)`` accumulated in fp64,
  with the operand element addressed by explicit index arithmetic for each
  storage layout (K-contiguous or M/N-contiguous).  The operand cases are
  those of the Triton inThreadTranspose page ("Feature description": a dot
  operand is either contiguous along K or not) and the plain definition of
  a matrix product.  A library matmul is used as the summation step.
* :func:`gemm_elements` -- the same sum for selected (m, n), one dot product
  per output, for full-size problems.
* :func:`dequant_int4` -- ``w(k,n) = (q(n,k) - z(n,g)) * s(n,g)`` with
  ``g = k // group``; the BitBLAS TileLang page ("Relevant Issues" and the
  dequantise copy example) is the setting; the pages give no formula, and
  this is the plainest reading (per-group fp16 scale and zero point, groups
  of 128 consecutive k by default, zero point 8 when none is given).
* :func:`splitk_factor` -- the SM-waste split-K rule of the BitBLAS page
  (the "SplitK Infer for dequantize cases" snippet).
* :func:`perm_forward` / :func:`perm_inverse` -- the perpendicular-dimension
  stride permutation of the hipBLASLt DTL page ("Add support for permuting
  perpDim": forward and inverse mappings).
* :func:`attention` / :func:`attention_rows` -- ``O = softmax(Q K^T * scale) V``
  per head, in fp64: the fused attention whose second product P.V the Triton
  inThreadTranspose page names as a non-TN dot ("Introduction": the second
  dotOp of Flash Attention, V contiguous along the output dimension).  The
  pages give no formula; this is the standard definition (row-wise softmax
  of the scaled logits, then the product with V), non-causal, with
  ``scale = 1 / sqrt(d)`` unless given, Q, K, V and O stored [head][row][d]
  contiguous.
* :func:`round_to` -- round-to-nearest-even of fp64 values to fp16 / bf16.
* :func:`reduce_rows` -- ``out[r] = sum_c x[r*ldx + c]`` in fp64, the
  reduction of the IREE page ("[LLVMGPUVectorDistribute] Add support for
  inter-subgroup multi_reduction": linalg.generic with arith.addf over the
  inner dimension, initial value 0, on 4096 and 4 x 4096 f32 inputs);
  :func:`reduce_rows_bound` is the first-order fp32 summation error bound a
  result computed by any fixed order of pairwise additions with sequential
  chains of at most ``chain`` terms and trees of total depth ``depth``
  must meet.

Readings taken where the pages are silent or garbled (all listed in the
design notes): split-K grid counts use ceiling division (floor gives zero
tiles for M < block_M and the page's ratio then divides by zero); int4 low
nibble holds the even k; zeros pointer NULL means z = 8; the permutation is
applied within whole blocks of B indices and a trailing partial block is the
identity; output rounding is round-to-nearest-even, once.
"""
from __future__ import annotations

import numpy as np

K_CONTIG = 0
MN_CONTIG = 1
F16 = 0
BF16 = 1
INT4 = 2
F32 = 3


# ---------------------------------------------------------------------------
# element decoding (exact)
# ---------------------------------------------------------------------------

def decode(storage, dtype) -> np.ndarray:
    """Storage (numpy array or CPU torch tensor) of fp16 / bf16 / fp32 values
    -> exact fp64 values.  bf16 is the upper half of an IEEE binary32, so the
    16 stored bits shifted left by 16 are that binary32's bits."""
    if hasattr(storage, "numpy"):
        import torch
        if storage.dtype == torch.bfloat16:
            storage = storage.view(torch.int16).numpy().view(np.uint16)
        elif storage.dtype == torch.float16:
            storage = storage.numpy()
        else:
            storage = storage.numpy()
    a = np.asarray(storage)
    if dtype == F16:
        return a.view(np.float16).astype(np.float64)
    if dtype == BF16:
        bits = a.view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == F32:
        return a.view(np.float32).astype(np.float64)
    raise ValueError(f"decode: unsupported dtype {dtype}")


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """Round fp64 values to the nearest fp16 / bf16 value, ties to even,
    returned as fp64.  bf16 is done from the significand directly (one
    rounding, no detour through binary32)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == F16:
        with np.errstate(over="ignore"):       # overflow to inf is the rounding result
            return x.astype(np.float16).astype(np.float64)
    if dtype == BF16:
        out = np.empty_like(x)
        finite = np.isfinite(x)
        xf = x[finite]
        # bf16: 8 significant bits, minimum normal exponent -126, subnormal
        # spacing 2^-133.
        mant, exp = np.frexp(xf)               # xf = mant * 2^exp, |mant| in [0.5, 1)
        exp = np.maximum(exp, -125)            # below 2^-126 the spacing is fixed
        scaled = np.ldexp(xf, 8 - exp)         # exact: a power-of-two scaling
        r = np.ldexp(np.rint(scaled), exp - 8)  # rint: ties to even
        big = np.abs(r) > 3.3895313892515355e38   # beyond the largest bf16
        r[big] = np.copysign(np.inf, r[big])
        out[finite] = r
        out[~finite] = x[~finite]
        return out
    if dtype == F32:
        return x.astype(np.float32).astype(np.float64)
    raise ValueError(f"round_to: unsupported dtype {dtype}")


# ---------------------------------------------------------------------------
# operand addressing: explicit index arithmetic per layout
# ---------------------------------------------------------------------------

def a_index(m, k, layout, lda):
    """Flat storage index of A's logical element (m, k).
    K-contiguous: row-major M x K, element at m*lda + k.
    M-contiguous: column-major M x K, element at k*lda + m."""
    if layout == K_CONTIG:
        return m * lda + k
    if layout == MN_CONTIG:
        return k * lda + m
    raise ValueError("bad A layout")


def b_index(k, n, layout, ldb):
    """Flat storage index of B's logical element (k, n).
    K-contiguous: B stored N x K row-major, element at n*ldb + k.
    N-contiguous: B stored K x N row-major, element at k*ldb + n."""
    if layout == K_CONTIG:
        return n * ldb + k
    if layout == MN_CONTIG:
        return k * ldb + n
    raise ValueError("bad B layout")


def a_logical(A, M, K, layout, lda, dtype) -> np.ndarray:
    """A as a dense fp64 M x K array, gathered element by element through
    :func:`a_index`."""
    vals = decode(A, dtype)
    m = np.arange(M, dtype=np.int64)[:, None]
    k = np.arange(K, dtype=np.int64)[None, :]
    return vals[a_index(m, k, layout, lda)]


def b_logical(B, K, N, layout, ldb, dtype) -> np.ndarray:
    """B as a dense fp64 K x N array, gathered through :func:`b_index`."""
    vals = decode(B, dtype)
    k = np.arange(K, dtype=np.int64)[:, None]
    n = np.arange(N, dtype=np.int64)[None, :]
    return vals[b_index(k, n, layout, ldb)]


# ---------------------------------------------------------------------------
# int4 weights
# ---------------------------------------------------------------------------

def int4_codes(W, N, K) -> np.ndarray:
    """Codes q(n, k) in 0..15 as an N x K int array.  Row n holds K/2 bytes;
    byte k//2 carries k's code in its low nibble for even k and in its high
    nibble for odd k."""
    if hasattr(W, "numpy"):
        W = W.numpy()
    W = np.asarray(W, dtype=np.uint8).reshape(-1)
    n = np.arange(N, dtype=np.int64)[:, None]
    k = np.arange(K, dtype=np.int64)[None, :]
    byte = W[n * (K // 2) + k // 2].astype(np.int64)
    return (byte >> (4 * (k & 1))) & 0xF


def dequant_int4(W, scales, zeros, N, K, group) -> np.ndarray:
    """The dequantised weight as a logical fp64 K x N matrix:
    b(k, n) = (q(n, k) - z(n, k // group)) * s(n, k // group), evaluated in
    fp64.  ``zeros`` None means z = 8 everywhere."""
    q = int4_codes(W, N, K).astype(np.float64)                  # N x K
    G = K // group
    s = decode(scales, F16).reshape(N, G)
    z = np.full((N, G), 8.0) if zeros is None else decode(zeros, F16).reshape(N, G)
    g = np.arange(K) // group
    w = (q - z[:, g]) * s[:, g]                                  # N x K
    return w.T                                                   # K x N


# ---------------------------------------------------------------------------
# the GEMM
# ---------------------------------------------------------------------------

def logical_operands(M, N, K, A, a_layout, lda, a_dtype, B, b_layout, ldb, b_dtype,
                     scales=None, zeros=None, group=128):
    a = a_logical(A, M, K, a_layout, lda, a_dtype)
    if b_dtype == INT4:
        if b_layout != K_CONTIG:
            raise ValueError("int4 weights are stored N x K (K-contiguous)")
        b = dequant_int4(B, scales, zeros, N, K, group)
    else:
        b = b_logical(B, K, N, b_layout, ldb, b_dtype)
    return a, b


def gemm(M, N, K, A, a_layout, lda, a_dtype, B, b_layout, ldb, b_dtype,
         scales=None, zeros=None, group=128) -> np.ndarray:
    """Unrounded fp64 C = A.B (M x N).  K = 0 gives zeros."""
    a, b = logical_operands(M, N, K, A, a_layout, lda, a_dtype, B, b_layout, ldb, b_dtype,
                            scales, zeros, group)
    return a @ b


def gemm_elements(rows, cols, M, N, K, A, a_layout, lda, a_dtype, B, b_layout, ldb, b_dtype,
                  scales=None, zeros=None, group=128) -> np.ndarray:
    """fp64 C[rows[i], cols[i]] as one dot product each, reading only the
    needed row of A and column of B -- for problems too large to form."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    avals = decode(A, a_dtype)
    k = np.arange(K, dtype=np.int64)
    out = np.empty(len(rows), dtype=np.float64)
    if b_dtype == INT4:
        W_bytes = np.asarray(B.numpy() if hasattr(B, "numpy") else B, dtype=np.uint8).reshape(-1)
        s_all = decode(scales, F16).reshape(N, K // group)
        z_all = None if zeros is None else decode(zeros, F16).reshape(N, K // group)
        g = k // group
        for i, (m, n) in enumerate(zip(rows, cols)):
            byte = W_bytes[n * (K // 2) + k // 2].astype(np.int64)
            q = ((byte >> (4 * (k & 1))) & 0xF).astype(np.float64)
            z = 8.0 if z_all is None else z_all[n, g]
            w = (q - z) * s_all[n, g]
            out[i] = np.dot(avals[a_index(m, k, a_layout, lda)], w)
        return out
    bvals = decode(B, b_dtype)
    for i, (m, n) in enumerate(zip(rows, cols)):
        out[i] = np.dot(avals[a_index(m, k, a_layout, lda)], bvals[b_index(k, n, b_layout, ldb)])
    return out


# ---------------------------------------------------------------------------
# attention (the fused second product P.V with V contiguous along d)
# ---------------------------------------------------------------------------

def _softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row-wise softmax in fp64: exp(s - row max) / row sum."""
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def attention(Q, K, V, heads, sq, sk, d, dtype, scale=None) -> np.ndarray:
    """fp64 O[h] = softmax(Q[h] K[h]^T * scale) V[h] for every head h, from
    flat storages laid out [head][row][d]; returns heads x sq x d."""
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    q = decode(Q, dtype).reshape(heads, sq, d)
    k = decode(K, dtype).reshape(heads, sk, d)
    v = decode(V, dtype).reshape(heads, sk, d)
    out = np.empty((heads, sq, d), dtype=np.float64)
    for h in range(heads):
        p = _softmax_rows((q[h] @ k[h].T) * scale)
        out[h] = p @ v[h]
    return out


def attention_rows(heads_idx, rows, Q, K, V, heads, sq, sk, d, dtype, scale=None) -> np.ndarray:
    """fp64 O[heads_idx[i], rows[i], :] one query row at a time, for problems
    too large to form whole; returns len(rows) x d."""
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    q = decode(Q, dtype).reshape(heads, sq, d)
    k = decode(K, dtype).reshape(heads, sk, d)
    v = decode(V, dtype).reshape(heads, sk, d)
    out = np.empty((len(rows), d), dtype=np.float64)
    for i, (h, r) in enumerate(zip(heads_idx, rows)):
        p = _softmax_rows((k[h] @ q[h, r]) * scale)
        out[i] = p @ v[h]
    return out


# ---------------------------------------------------------------------------
# split-K factor (SM-waste rule)
# ---------------------------------------------------------------------------

def splitk_factor(M, N, K, block_M, block_N, block_K, num_sms, threshold=0.05):
    """Start at 1; stop when the share of SMs left idle in the last wave
    (tiles*f mod num_sms, over tiles*f) is at most ``threshold``, or when the
    doubled factor times block_K would reach K; otherwise double.
    Tile counts use ceiling division (the page's floor division yields zero
    tiles for M < block_M)."""
    grid_m = -(-M // block_M)
    grid_n = -(-N // block_N)
    total = grid_m * grid_n
    if total == 0:
        return 1
    f = 1
    while True:
        t = total * f
        waste = t - (t // num_sms) * num_sms
        if waste / t <= threshold:
            break
        doubled = f * 2
        if doubled * block_K >= K:
            break
        f = doubled
    return f


def splitk_trace(M, N, K, block_M, block_N, block_K, num_sms, threshold=0.05):
    """The sequence of (factor, waste ratio) the rule visits, for reports."""
    grid_m = -(-M // block_M)
    grid_n = -(-N // block_N)
    total = grid_m * grid_n
    out = []
    f = 1
    while True:
        t = total * f
        ratio = (t % num_sms) / t
        out.append((f, ratio))
        if ratio <= threshold or 2 * f * block_K >= K:
            return out
        f *= 2


# ---------------------------------------------------------------------------
# perpendicular-dimension stride permutation
# ---------------------------------------------------------------------------

def perm_forward(i, block, stride):
    """Within blocks of ``block`` indices: S' = block / stride,
    i' = stride * (i mod S') + i div S' (the global-read mapping).  Indices
    in a trailing partial block map to themselves; ``stride`` must divide
    ``block``."""
    if block <= 0 or stride <= 0 or block % stride:
        raise ValueError("stride must divide block")
    base, r = divmod(i, block)
    sp = block // stride
    return base * block + stride * (r % sp) + r // sp


def perm_inverse(ip, block, stride):
    """The local-read mapping: with S' = block / stride,
    i = S' * (i' mod stride) + i' div stride."""
    if block <= 0 or stride <= 0 or block % stride:
        raise ValueError("stride must divide block")
    base, r = divmod(ip, block)
    sp = block // stride
    return base * block + sp * (r % stride) + r // stride


def perm_apply(count, block, stride):
    """The forward map over 0..count-1 (trailing partial block = identity)."""
    full = (count // block) * block
    return [perm_forward(i, block, stride) if i < full else i for i in range(count)]


# ---------------------------------------------------------------------------
# row reduction (IREE page: inter-subgroup multi_reduction)
# ---------------------------------------------------------------------------

def reduce_rows(x, rows, cols, ldx=0) -> np.ndarray:
    """out[r] = sum over c < cols of x[r*ldx + c], each fp32 input exact
    in fp64 and the sum accumulated in fp64 (ldx = 0 means cols).  Elements
    outside a row's first ``cols`` (padding) are never read."""
    ldx = cols if ldx == 0 else ldx
    vals = np.asarray(x.numpy() if hasattr(x, "numpy") else x, dtype=np.float32).astype(np.float64)
    out = np.zeros(rows, dtype=np.float64)
    for r in range(rows):
        idx = r * ldx + np.arange(cols, dtype=np.int64)
        out[r] = np.sum(vals[idx]) if cols else 0.0
    return out


def reduce_rows_abs(x, rows, cols, ldx=0) -> np.ndarray:
    """sum over c of |x[r*ldx + c]| per row, in fp64 (the scale of the
    rounding error of any fp32 summation of the row)."""
    return reduce_rows(np.abs(np.asarray(x.numpy() if hasattr(x, "numpy") else x, dtype=np.float32)), rows, cols, ldx)


def reduce_rows_bound(abs_sums, chain, depth):
    """First-order bound on |fp32 sum - exact sum| for a summation whose
    every term passes through at most ``chain`` sequential additions and
    trees of total depth ``depth``: (chain + depth) * 2^-24 * sum |x|
    (each addition rounds once with relative error at most 2^-24, and a term
    is affected only by the additions on its path to the result)."""
    return (chain + depth) * 2.0 ** -24 * np.asarray(abs_sums, dtype=np.float64)


# ---------------------------------------------------------------------------
# acceptance check
# ---------------------------------------------------------------------------

def check_close(c_gpu: np.ndarray, c_ref: np.ndarray, elem_tol=2e-2, fro_tol=2e-3):
    """Return (ok, max_violation, rel_fro): elementwise
    |c_gpu - c_ref| <= elem_tol * (|c_ref| + 1) and relative Frobenius error
    <= fro_tol (an all-zero reference requires an exact zero result)."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    c_ref = np.asarray(c_ref, dtype=np.float64)
    diff = np.abs(c_gpu - c_ref)
    bound = elem_tol * (np.abs(c_ref) + 1.0)
    viol = float(np.max(diff / bound)) if diff.size else 0.0
    denom = float(np.linalg.norm(c_ref))
    num = float(np.linalg.norm(c_gpu - c_ref))
    rel = num / denom if denom > 0 else (0.0 if num == 0 else float("inf"))
    ok = bool(np.all(np.isfinite(c_gpu)) and viol <= 1.0 and rel <= fro_tol)
    return ok, viol, rel
