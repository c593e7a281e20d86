"""Runs one GEMM through the C-ABI on the GPU with guard bands around every
buffer, and returns what the library wrote.

Each stored array lives inside a larger device buffer: `GUARD` sentinel
elements before and after it, and the same sentinel in every leading-
dimension gap.  After the call the harness checks, bit for bit, that no
sentinel changed (A and B entirely unchanged; C changed only inside its
M x N window), so an out-of-bounds write or a write into the ld gap fails the
test.  An element offset can misalign a base pointer on purpose.
"""
from __future__ import annotations

import numpy as np

import dense_fp32_gemm_05_gb300 as sg

GUARD = 64
SENTINEL = np.float32(-7.75e30)


def _embed(arr2d: np.ndarray | None, rows: int, ld: int, offset: int):
    """Flat fp32 host buffer: guard, `offset` extra, rows x ld (gaps sentinel), guard."""
    n = GUARD + offset + rows * ld + GUARD
    buf = np.full(max(n, 1), SENTINEL, dtype=np.float32)
    if arr2d is not None and rows > 0:
        view = buf[GUARD + offset: GUARD + offset + rows * ld].reshape(rows, ld)
        view[:, : arr2d.shape[1]] = arr2d
    return buf, GUARD + offset


def run(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, path=sg.PATH_FFMA,
        split=0, offsets=(0, 0, 0), c_fill=None, device="cuda", check_guards=True, stream=None):
    """Returns (status, C_out) with C_out the M x N result as numpy float32.

    A, B: stored arrays (rows x cols) or None.  C: initial M x N values or
    None (then c_fill, default NaN, is written into C's window).
    """
    import torch

    a_rows = (M if transA.upper() == "N" else K)
    b_rows = (K if transB.upper() == "N" else N)
    hA, oa = _embed(A, a_rows if A is not None else 0, lda, offsets[0])
    hB, ob = _embed(B, b_rows if B is not None else 0, ldb, offsets[1])
    if C is None:
        C = np.full((M, N), np.nan if c_fill is None else c_fill, dtype=np.float32)
    hC, oc = _embed(C, M, ldc, offsets[2])
    dA = torch.from_numpy(hA).to(device)
    dB = torch.from_numpy(hB).to(device)
    dC = torch.from_numpy(hC).to(device)
    pa = dA.data_ptr() + 4 * oa
    pb = dB.data_ptr() + 4 * ob
    pc = dC.data_ptr() + 4 * oc
    if stream is None:
        stream = torch.cuda.current_stream()
    st = sg.sgemm_ex(transA, transB, M, N, K, alpha, pa if A is not None else 0, lda,
                     pb if B is not None else 0, ldb, beta, pc, ldc, stream, path, split)
    torch.cuda.synchronize()
    outC = dC.cpu().numpy()
    if check_guards:
        assert np.array_equal(dA.cpu().numpy().view(np.uint32), hA.view(np.uint32)), "A modified"
        assert np.array_equal(dB.cpu().numpy().view(np.uint32), hB.view(np.uint32)), "B modified"
        mask = np.ones(outC.shape, dtype=bool)
        if M > 0:
            win = mask[oc: oc + M * ldc].reshape(M, ldc)
            win[:, :N] = False
        bad = (outC.view(np.uint32) != hC.view(np.uint32)) & mask
        assert not bad.any(), f"{int(bad.sum())} elements outside C's window changed"
    res = outC[oc: oc + M * ldc].reshape(M, ldc)[:, :N].copy() if M > 0 else np.zeros((0, N), np.float32)
    return st, res
