"""The pages' shuffled weight layouts, and the library's ingest of them.

CPU: the numpy restatement of each forward layout (from the shuffled-scale
store of submission 755056 and the subtile layout) is inverted exactly by the
pages' own inverse -- the reshape/permute of `materialize_linear_weight_layout`
and `materialize_linear_scale_layout` (submission 748756).
GPU: mxfp4_pack_weights_shuffled gives byte-for-byte the buffer
mxfp4_pack_weights gives from the natural layout."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from shuffled_layouts import shuffle_codes, shuffle_scales


def unshuffle_codes_pages(flat: np.ndarray, N: int, kh: int) -> np.ndarray:
    # materialize_linear_weight_layout, without its final transpose
    t = torch.from_numpy(flat.copy()).reshape(1, N // 16, kh // 32, 2, 16, 16)
    return t.permute(0, 1, 4, 2, 3, 5).reshape(N, kh).numpy()


def unshuffle_scales_pages(flat: np.ndarray, N: int, G: int) -> np.ndarray:
    # materialize_linear_scale_layout
    m_pad = -(-N // 256) * 256
    k_pad = -(-G // 8) * 8
    t = torch.from_numpy(flat.copy()).reshape(m_pad // 32, k_pad // 8, 4, 16, 2, 2, 1)
    return t.permute(0, 5, 3, 1, 4, 2, 6).reshape(m_pad, k_pad)[:N, :G].numpy()


@pytest.mark.parametrize("N,K", [(16, 64), (48, 192), (2112, 7168), (2880, 512), (272, 1088)])
def test_shuffles_invert_with_the_pages_functions(N, K):
    rng = np.random.default_rng(N + K)
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    s = rng.integers(0, 255, (N, K // 32), dtype=np.uint8)
    assert np.array_equal(unshuffle_codes_pages(shuffle_codes(q), N, K // 2), q)
    assert np.array_equal(unshuffle_scales_pages(shuffle_scales(s), N, K // 32), s)


@pytest.mark.gpu
@pytest.mark.parametrize("N,K", [(16, 64), (48, 192), (2112, 7168), (2880, 512), (272, 1088)])
def test_pack_from_shuffled_equals_pack_from_natural(N, K):
    import block_scaled_mxfp4_activation_gb300 as mx

    assert torch.cuda.is_available()
    rng = np.random.default_rng(7 * N + K)
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    s = rng.integers(0, 255, (N, K // 32), dtype=np.uint8)
    natural = mx.pack_weights(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    W = mx.pack_weights_shuffled(torch.from_numpy(shuffle_codes(q)).cuda(), torch.from_numpy(shuffle_scales(s)).cuda(),
                                 N, K)
    torch.cuda.synchronize()
    assert torch.equal(W.data, natural)
    q2, s2 = mx.unpack_weights(W.data, N, K)
    assert np.array_equal(q2.cpu().numpy(), q) and np.array_equal(s2.cpu().numpy(), s)


@pytest.mark.gpu
def test_custom_kernel_runs_the_pages_tuple(oracle_mod):
    """The harness tuple (A, B, B_q, B_shuffle, B_scale_sh), B quantized with the
    pages' rule (the oracle), through the pages' entry point name."""
    import block_scaled_mxfp4_activation_gb300 as mx
    import workloads

    M, N, K = 32, 2880, 512
    A, B = workloads.make_random(M, N, K, seed=12)
    bq, bs = oracle_mod.quantize(B)
    data = (A.cuda(), B.cuda(), torch.from_numpy(bq).cuda(), torch.from_numpy(shuffle_codes(bq)).cuda(),
            torch.from_numpy(shuffle_scales(bs)).cuda())
    C = mx.custom_kernel(data)
    C2 = mx.custom_kernel(data)  # the cached packed weight
    _, _, c64, _ = oracle_mod.quant_gemm(A, bq, bs)
    got = C.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(c64 ** 2)))
    assert np.all(np.abs(got - c64) <= 8e-3 * np.abs(c64) + 1e-2 * rms)
    assert torch.equal(C, C2)

