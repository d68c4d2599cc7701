"""Python binding of the any-layout GEMM C ABI (``include/gemm.h``) and the
fp32 row reduction (``include/reduce.h``).

Argument marshalling only: every function forwards to the entry point of the
same name in ``_lib/libgemm.so``; all arithmetic runs in the library's CUDA
kernels.  Importing this package fails loudly when the library has not been
built -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgemm.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_ALIGNMENT = 3
GEMM_ERR_WORKSPACE = 4
GEMM_ERR_CUDA = 5
GEMM_ERR_TIMEOUT = 6

GEMM_FLAG_DETERMINISTIC = 1
GEMM_FLAG_INT4_PREPACKED = 4
GEMM_FLAG_TEST_WITHHOLD_STAGE = 1 << 30

GEMM_K_CONTIG = 0
GEMM_MN_CONTIG = 1

GEMM_F16 = 0
GEMM_BF16 = 1
GEMM_INT4 = 2
GEMM_F32 = 3

# Every entry point include/gemm.h and include/reduce.h declare.
EXPORTS = (
    "gemm_create", "gemm_workspace_size", "gemm_query", "gemm_run", "gemm_run_static_scratch",
    "gemm_sync_status", "gemm_destroy",
    "gemm_splitk_auto", "gemm_perm_fwd", "gemm_perm_inv", "gemm_perm_device", "gemm_magic_divmod_host",
    "gemm_magic_divmod_device", "gemm_status_string", "gemm_int4_prepack_bytes", "gemm_int4_prepack",
    "reduce_rows_workspace_size", "reduce_rows_f32",
    "attn_create", "attn_run", "attn_sync_status", "attn_destroy",
)


class gemm_desc_t(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("a_layout", ctypes.c_int32), ("b_layout", ctypes.c_int32),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
        ("a_dtype", ctypes.c_int32), ("b_dtype", ctypes.c_int32), ("c_dtype", ctypes.c_int32),
        ("split_k", ctypes.c_int32), ("group_size", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("flags", ctypes.c_int32),
    ]


class attn_desc_t(ctypes.Structure):
    _fields_ = [
        ("heads", ctypes.c_int32), ("seq_q", ctypes.c_int32), ("seq_k", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
    ]


class gemm_info_t(ctypes.Structure):
    _fields_ = [
        ("split_k", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
        ("tile_k", ctypes.c_int32), ("swap_ab", ctypes.c_int32), ("num_units", ctypes.c_int32),
        ("k_per_split", ctypes.c_int32), ("repack_a", ctypes.c_int32), ("repack_b", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("streamk_tiles", ctypes.c_int32), ("cluster_size", ctypes.c_int32), ("dequant_form", ctypes.c_int32),
        ("realign", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python layout_general_tensor_gb300/build.py` "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    sig = {
        "gemm_create": (ctypes.c_int, [ctypes.POINTER(gemm_desc_t), ctypes.POINTER(P)]),
        "gemm_workspace_size": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_size_t)]),
        "gemm_query": (ctypes.c_int, [P, ctypes.POINTER(gemm_info_t)]),
        "gemm_run": (ctypes.c_int, [P, P, P, P, P, P, P, ctypes.c_size_t, P]),
        "gemm_run_static_scratch": (ctypes.c_int, [P, P, P, P, P]),
        "gemm_sync_status": (ctypes.c_int, [P, P]),
        "gemm_destroy": (ctypes.c_int, [P]),
        "gemm_splitk_auto": (ctypes.c_int32, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double]),
        "gemm_perm_fwd": (ctypes.c_uint32, [ctypes.c_uint32] * 4),
        "gemm_perm_inv": (ctypes.c_uint32, [ctypes.c_uint32] * 4),
        "gemm_perm_device": (ctypes.c_int, [P, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                            ctypes.c_int32, P, P]),
        "gemm_magic_divmod_host": (ctypes.c_int, [P, ctypes.c_size_t, ctypes.c_uint32, P, P]),
        "gemm_magic_divmod_device": (ctypes.c_int, [P, ctypes.c_size_t, ctypes.c_uint32, P, P, P]),
        "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "gemm_int4_prepack_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]),
        "gemm_int4_prepack": (ctypes.c_int, [P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                             P, P]),
        "reduce_rows_workspace_size": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                      ctypes.POINTER(ctypes.c_size_t)]),
        "reduce_rows_f32": (ctypes.c_int, [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P,
                                           ctypes.c_size_t, P]),
        "attn_create": (ctypes.c_int, [ctypes.POINTER(attn_desc_t), ctypes.POINTER(P)]),
        "attn_run": (ctypes.c_int, [P, P, P, P, P, P]),
        "attn_sync_status": (ctypes.c_int, [P, P]),
        "attn_destroy": (ctypes.c_int, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


class GemmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {gemm_status_string(status)} ({status})")


def _check(status, what):
    if status != GEMM_OK:
        raise GemmError(status, what)


# ------------------------------------------------------------- thin wrappers

def gemm_status_string(status: int) -> str:
    return _lib.gemm_status_string(int(status)).decode()


def gemm_create(desc: gemm_desc_t) -> int:
    h = ctypes.c_void_p()
    _check(_lib.gemm_create(ctypes.byref(desc), ctypes.byref(h)), "gemm_create")
    return h.value


def gemm_create_status(desc: gemm_desc_t):
    """gemm_create returning (status, handle or None) without raising."""
    h = ctypes.c_void_p()
    st = _lib.gemm_create(ctypes.byref(desc), ctypes.byref(h))
    return st, h.value


def gemm_workspace_size(plan: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.gemm_workspace_size(plan, ctypes.byref(n)), "gemm_workspace_size")
    return n.value


def gemm_query(plan: int) -> gemm_info_t:
    info = gemm_info_t()
    _check(_lib.gemm_query(plan, ctypes.byref(info)), "gemm_query")
    return info


def gemm_run(plan: int, A: int, B: int, C: int, scales: int = 0, zeros: int = 0, workspace: int = 0,
             workspace_bytes: int = 0, stream: int = 0) -> int:
    """Raw entry point: integer device addresses; returns the status code."""
    return _lib.gemm_run(plan, A or None, B or None, C or None, scales or None, zeros or None, workspace or None,
                         workspace_bytes, stream or None)


def gemm_run_static_scratch(plan: int, A: int, B: int, C: int, stream: int = 0) -> int:
    """Run `plan` using the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate device memory when
    they run the GEMM).  Integer device addresses; returns the status."""
    return _lib.gemm_run_static_scratch(plan, A or None, B or None, C or None, stream or None)


def gemm_sync_status(plan: int, stream: int = 0) -> int:
    return _lib.gemm_sync_status(plan, stream or None)


def gemm_destroy(plan: int) -> None:
    _check(_lib.gemm_destroy(plan), "gemm_destroy")


def gemm_splitk_auto(M, N, K, block_m=128, block_n=128, block_k=64, num_sms=148, threshold=0.05) -> int:
    return _lib.gemm_splitk_auto(M, N, K, block_m, block_n, block_k, num_sms, threshold)


def gemm_int4_prepack_bytes(N: int, K: int, group_size: int = 128) -> int:
    """Bytes of the pre-packed int4 weight buffer (0: shape not taken)."""
    return _lib.gemm_int4_prepack_bytes(N, K, group_size)


def gemm_int4_prepack(B: int, ldb: int, scales: int, N: int, K: int, group_size: int, out: int,
                      stream: int = 0) -> int:
    """Raw entry point: device addresses of the plain int4 weights, their fp16
    scales and the output buffer; returns the status."""
    return _lib.gemm_int4_prepack(B or None, ldb, scales or None, N, K, group_size, out or None, stream or None)


def gemm_perm_fwd(index, count, block, stride) -> int:
    return _lib.gemm_perm_fwd(index, count, block, stride)


def gemm_perm_inv(index, count, block, stride) -> int:
    return _lib.gemm_perm_inv(index, count, block, stride)


def gemm_perm_device(in_ptr, n, count, block, stride, inverse, out_ptr, stream=0) -> int:
    """Raw entry point: device addresses of uint32 arrays; returns the status."""
    return _lib.gemm_perm_device(in_ptr or None, n, count, block, stride, int(inverse), out_ptr or None,
                                 stream or None)


def gemm_magic_divmod_host(n_array, divisor):
    """n_array: numpy uint32 array (C-contiguous).  Returns (q, r) arrays."""
    import numpy as np
    n = np.ascontiguousarray(n_array, dtype=np.uint32)
    q = np.empty_like(n)
    r = np.empty_like(n)
    _check(_lib.gemm_magic_divmod_host(n.ctypes.data, n.size, divisor, q.ctypes.data, r.ctypes.data),
           "gemm_magic_divmod_host")
    return q, r


def gemm_magic_divmod_device(n_ptr, count, divisor, q_ptr, r_ptr, stream=0) -> int:
    return _lib.gemm_magic_divmod_device(n_ptr, count, divisor, q_ptr, r_ptr, stream or None)


def reduce_rows_workspace_size(rows: int, cols: int, num_sms: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(_lib.reduce_rows_workspace_size(rows, cols, num_sms, ctypes.byref(n)), "reduce_rows_workspace_size")
    return n.value


def reduce_rows_f32(x: int, rows: int, cols: int, ldx: int, out: int, workspace: int = 0, workspace_bytes: int = 0,
                    stream: int = 0) -> int:
    """Raw entry point: integer device addresses; returns the status code."""
    return _lib.reduce_rows_f32(x or None, rows, cols, ldx, out or None, workspace or None, workspace_bytes,
                                stream or None)


def _require_device(what, **tensors):
    """Every given tensor must live in CUDA device memory: a host address
    handed to a kernel (or encoded into a tensor map) would fault the GPU
    instead of returning an error."""
    for name, t in tensors.items():
        if t is not None and not getattr(t, "is_cuda", False):
            raise ValueError(f"{what}: {name} must be a CUDA tensor")


class RowReduce:
    """out[r] = sum of row r of an fp32 matrix, with its (zero-filled) device
    workspace.  Marshalling only: passes device addresses and the current
    torch stream to reduce_rows_f32."""

    def __init__(self, rows: int, cols: int, device=None):
        import torch
        self.rows, self.cols = rows, cols
        self.ws_bytes = reduce_rows_workspace_size(rows, cols, 0)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.workspace = torch.zeros(max(self.ws_bytes, 1), dtype=torch.uint8, device=dev)

    def run(self, x, out, ldx: int = 0, stream=None):
        import torch
        _require_device("RowReduce.run", x=x, out=out)
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        st = reduce_rows_f32(x.data_ptr(), self.rows, self.cols, ldx, out.data_ptr(),
                             self.workspace.data_ptr() if self.ws_bytes else 0, self.ws_bytes, s)
        _check(st, "reduce_rows_f32")


def make_desc(M, N, K, a_layout=GEMM_K_CONTIG, b_layout=GEMM_K_CONTIG, a_dtype=GEMM_BF16, b_dtype=None,
              c_dtype=None, lda=0, ldb=0, ldc=0, split_k=1, group_size=0, num_sms=0, flags=0) -> gemm_desc_t:
    b_dtype = a_dtype if b_dtype is None else b_dtype
    c_dtype = a_dtype if c_dtype is None else c_dtype
    return gemm_desc_t(M, N, K, a_layout, b_layout, lda, ldb, ldc, a_dtype, b_dtype, c_dtype, split_k,
                       group_size, num_sms, flags)


class Gemm:
    """A plan plus its (zero-filled) device workspace, run on torch tensors.

    Marshalling only: passes the tensors' device addresses and the current
    torch stream to gemm_run."""

    def __init__(self, desc: gemm_desc_t, device=None):
        import torch
        self.desc = desc
        self.plan = gemm_create(desc)
        self.info = gemm_query(self.plan)
        self.ws_bytes = gemm_workspace_size(self.plan)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.workspace = torch.zeros(max(self.ws_bytes, 1), dtype=torch.uint8, device=dev)

    def run(self, A, B, C, scales=None, zeros=None, stream=None, workspace=None, workspace_bytes=None):
        import torch
        ws = self.workspace if workspace is None else workspace
        wsb = self.ws_bytes if workspace_bytes is None else workspace_bytes
        _require_device("Gemm.run", A=A, B=B, C=C, scales=scales, zeros=zeros, workspace=ws if wsb else None)
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        st = gemm_run(self.plan, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                      scales.data_ptr() if scales is not None else 0,
                      zeros.data_ptr() if zeros is not None else 0,
                      ws.data_ptr() if wsb else 0, wsb, s)
        _check(st, "gemm_run")

    def sync_status(self, stream=None) -> int:
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        return gemm_sync_status(self.plan, s)

    def close(self):
        if self.plan:
            gemm_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def int4_prepack(B, scales, N, K, group_size=128, ldb=0, stream=None):
    """Pre-pack int4 weights (device uint8 tensor, N rows of ldb bytes) and
    their fp16 scales for GEMM_FLAG_INT4_PREPACKED; returns the packed device
    uint8 tensor."""
    import torch
    _require_device("int4_prepack", B=B, scales=scales)
    nbytes = gemm_int4_prepack_bytes(N, K, group_size)
    if nbytes == 0:
        raise GemmError(GEMM_ERR_INVALID_ARG, "gemm_int4_prepack_bytes")
    out = torch.empty(nbytes, dtype=torch.uint8, device=B.device)
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    _check(gemm_int4_prepack(B.data_ptr(), ldb, scales.data_ptr(), N, K, group_size, out.data_ptr(), s),
           "gemm_int4_prepack")
    return out


def attn_create_status(desc: attn_desc_t):
    """attn_create returning (status, handle or None) without raising."""
    h = ctypes.c_void_p()
    st = _lib.attn_create(ctypes.byref(desc), ctypes.byref(h))
    return st, h.value


def attn_run(plan: int, Q: int, K: int, V: int, O: int, stream: int = 0) -> int:
    """Raw entry point: integer device addresses; returns the status code."""
    return _lib.attn_run(plan, Q or None, K or None, V or None, O or None, stream or None)


class Attention:
    """A fused-attention plan run on torch tensors laid out [head][row][d]
    (marshalling only: the tensors' device addresses and the current torch
    stream go to attn_run)."""

    def __init__(self, heads, seq_q, seq_k, head_dim, dtype=GEMM_BF16, scale=0.0):
        self.desc = attn_desc_t(heads, seq_q, seq_k, head_dim, dtype, scale)
        st, h = attn_create_status(self.desc)
        _check(st, "attn_create")
        self.plan = h

    def run(self, Q, K, V, O, stream=None):
        import torch
        _require_device("Attention.run", Q=Q, K=K, V=V, O=O)
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        _check(attn_run(self.plan, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), s), "attn_run")

    def sync_status(self, stream=None) -> int:
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        return _lib.attn_sync_status(self.plan, s or None)

    def close(self):
        if self.plan:
            _lib.attn_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
