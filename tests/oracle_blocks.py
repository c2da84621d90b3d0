"""The oracle's full GEMM over large shapes, in blocks run side by side.

Each output element C[m, n] is the oracle's own sum over k for row m of A and
row n of B, so computing C as a grid of (row block of A) x (row block of B)
calls to the unmodified oracle gives exactly the same values as one call.  The
oracle is a C library reached through ctypes, which releases the GIL during a
call, so the blocks run in parallel threads.  Test infrastructure only."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def gemm_full(oracle_mod, aq: np.ndarray, as_: np.ndarray, bq: np.ndarray, bs: np.ndarray,
              threads: int | None = None) -> np.ndarray:
    """fp64 C [M, N] = the oracle's gemm(aq, as_, bq, bs), computed block-wise."""
    M, N = aq.shape[0], bq.shape[0]
    threads = threads or max(1, min(32, os.cpu_count() or 1))
    # about 2 blocks per thread, split along whichever side is longer
    parts = 2 * threads
    mb = max(1, -(-M // parts)) if M >= N else M
    nb = max(1, -(-N // parts)) if N > M else N
    if M >= N and M < parts:
        nb = max(1, -(-N // max(1, parts // M)))
    blocks = [(m0, min(M, m0 + mb), n0, min(N, n0 + nb)) for m0 in range(0, M, mb) for n0 in range(0, N, nb)]
    out = np.empty((M, N), np.float64)

    def run(b):
        m0, m1, n0, n1 = b
        c64, _ = oracle_mod.gemm(aq[m0:m1], as_[m0:m1], bq[n0:n1], bs[n0:n1])
        out[m0:m1, n0:n1] = c64

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(run, blocks))
    return out
