"""GPU check of the perpendicular-dimension stride permutation (hipBLASLt DTL
page, "Add support for permuting perpDim"): the device routine the loaders
use, run through gemm_perm_device, against the oracle's forward and inverse
maps, bit for bit, for every block size B <= 256 and every stride S dividing
B, over index ranges that end in a partial block (which maps to itself)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import lib

pytestmark = pytest.mark.gpu


def _cases():
    for B in range(1, 257):
        for S in range(1, B + 1):
            if B % S == 0:
                yield B, S


def test_perm_device_matches_oracle_exhaustive():
    m = lib()
    stream = torch.cuda.current_stream().cuda_stream
    cases = list(_cases())
    counts = [3 * B + B // 2 for B, _ in cases]  # three full blocks and a partial tail
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    total = int(offs[-1])
    idx = torch.from_numpy(np.concatenate([np.arange(c, dtype=np.uint32) for c in counts]).view(np.int32)).cuda()
    fwd = torch.empty_like(idx)
    inv = torch.empty_like(idx)
    back = torch.empty_like(idx)
    esz = idx.element_size()
    for (B, S), c, o in zip(cases, counts, offs[:-1]):
        o = int(o)
        src = idx.data_ptr() + o * esz
        assert m.gemm_perm_device(src, c, c, B, S, 0, fwd.data_ptr() + o * esz, stream) == m.GEMM_OK
        assert m.gemm_perm_device(src, c, c, B, S, 1, inv.data_ptr() + o * esz, stream) == m.GEMM_OK
        # inverse of the forward map, in place on a copy
        assert m.gemm_perm_device(fwd.data_ptr() + o * esz, c, c, B, S, 1, back.data_ptr() + o * esz,
                                  stream) == m.GEMM_OK
    torch.cuda.synchronize()
    fwd_h = fwd.cpu().numpy().view(np.uint32)
    inv_h = inv.cpu().numpy().view(np.uint32)
    back_h = back.cpu().numpy().view(np.uint32)
    for (B, S), c, o in zip(cases, counts, offs[:-1]):
        o = int(o)
        full = (c // B) * B
        want_fwd = oracle.perm_apply(c, B, S)
        want_inv = [oracle.perm_inverse(i, B, S) if i < full else i for i in range(c)]
        assert fwd_h[o:o + c].tolist() == want_fwd, (B, S)
        assert inv_h[o:o + c].tolist() == want_inv, (B, S)
        assert back_h[o:o + c].tolist() == list(range(c)), (B, S)
    assert total == fwd_h.size


def test_perm_device_invalid_stride_is_identity_and_null_rejected():
    m = lib()
    stream = torch.cuda.current_stream().cuda_stream
    idx = torch.arange(40, dtype=torch.int32, device="cuda")
    out = torch.empty_like(idx)
    for B, S in ((8, 3), (0, 1), (8, 0)):
        assert m.gemm_perm_device(idx.data_ptr(), 40, 40, B, S, 0, out.data_ptr(), stream) == m.GEMM_OK
        torch.cuda.synchronize()
        assert out.cpu().tolist() == list(range(40))
    assert m.gemm_perm_device(0, 4, 4, 8, 2, 0, out.data_ptr(), stream) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_perm_device(idx.data_ptr(), 0, 0, 8, 2, 0, out.data_ptr(), stream) == m.GEMM_OK
