"""The weight layouts the pages' harness hands out, restated in numpy for the
tests (forward direction: natural -> shuffled)."""
from __future__ import annotations

import numpy as np


def shuffle_codes(q: np.ndarray) -> np.ndarray:
    """Natural codes [N, Kh] -> the preshuffled byte array (16 x 16-byte
    subtiles): byte (n, kb) at ((n/16 * Kh/32 + kb/32) * 2 + (kb%32)/16) * 256
    + (n%16) * 16 + kb%16."""
    N, kh = q.shape
    n = np.arange(N)[:, None]
    kb = np.arange(kh)[None, :]
    idx = ((n // 16 * (kh // 32) + kb // 32) * 2 + (kb % 32) // 16) * 256 + (n % 16) * 16 + kb % 16
    out = np.zeros(N * kh, np.uint8)
    out[idx.ravel()] = q.ravel()
    return out


def shuffle_scales(s: np.ndarray, pad_rows_to: int = 256) -> np.ndarray:
    """Natural scales [N, G] -> the e8m0 shuffle: scale (n, g) at (n/32) * 32 *
    Gp + (g/8) * 256 + (g%4) * 64 + (n%16) * 4 + ((g%8)/4) * 2 + (n%32)/16,
    Gp = G rounded up to 8; rows padded to `pad_rows_to` (padding bytes 0)."""
    N, G = s.shape
    gp = -(-G // 8) * 8
    m_pad = -(-N // pad_rows_to) * pad_rows_to
    n = np.arange(N)[:, None]
    g = np.arange(G)[None, :]
    idx = (n // 32) * 32 * gp + (g // 8) * 256 + (g % 4) * 64 + (n % 16) * 4 + ((g % 8) // 4) * 2 + (n % 32) // 16
    out = np.zeros(m_pad * gp, np.uint8)
    out[idx.ravel()] = s.ravel()
    return out
