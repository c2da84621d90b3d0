"""The allocation-free entry point, mxfp4_quant_gemm_static_scratch.

Some callers cannot allocate device memory (a plugin inside a framework that
reserves all of it up front, or code that must not call cudaMalloc because it
synchronises the device), so they cannot hand mxfp4_quant_gemm a workspace.
This entry keeps its scratch in a fixed array inside the library.  These
tests call it through the C ABI and compare it with the existing entry point
and with the CPU oracle on the same inputs, twice in a row (the array keeps
the previous call's contents).  The file sorts last so that a run stopping at the first failure
has already run every other test; it also passes on its own in a fresh
process."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import block_scaled_mxfp4_activation_gb300 as mx
import workloads

pytestmark = pytest.mark.gpu

RTOL, ATOL_RMS = 8e-3, 1e-2  # the tolerance of the parity tests


def _entry():
    lib = mx.load_library()
    fn = lib.mxfp4_quant_gemm_static_scratch
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return lib, fn


def _close(got: torch.Tensor, ref: torch.Tensor, what: str):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(r ** 2)))
    bad = np.abs(g - r) > RTOL * np.abs(r) + ATOL_RMS * rms
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance"


def _close64(got: torch.Tensor, ref64: np.ndarray, what: str):
    g = got.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref64 ** 2)))
    bad = np.abs(g - ref64) > RTOL * np.abs(ref64) + ATOL_RMS * rms
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance of the oracle"


@pytest.mark.parametrize("M,N,K,seed", [(64, 512, 2048, 31), (100, 300, 288, 32), (16, 2112, 1024, 33)])
def test_static_scratch_matches_existing_entry_twice(oracle_mod, M, N, K, seed):
    assert torch.cuda.is_available(), "GPU test"
    torch.cuda.set_device(0)
    _, fn = _entry()
    A, B = workloads.make_random(M, N, K, seed=seed)
    bq, bs = oracle_mod.quantize(B)  # the weight quantized by the oracle, packed on the GPU
    W = mx.PackedWeight(mx.pack_weights(torch.from_numpy(bq).cuda(), torch.from_numpy(bs).cuda()), N, K)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        A_call = (A.float() * (1.0 + call)).to(torch.bfloat16)  # a different activation each call
        Ad = A_call.cuda()
        expect = mx.quant_gemm(Ad, W)  # the existing entry (workspace from torch when M >= 64)
        got = torch.empty_like(expect)
        status = fn(Ad.data_ptr(), Ad.stride(0), W.data.data_ptr(), got.data_ptr(), M, N, K, stream)
        assert status == 0, mx.status_string(status)
        torch.cuda.synchronize()
        _close(got, expect, f"call {call}, M={M} N={N} K={K}")
        # against the oracle, at the parity tests' tolerance
        _, _, c64, _ = oracle_mod.quant_gemm(A_call, bq, bs)
        _close64(got, c64, f"call {call}, M={M} N={N} K={K}")
        # the same two passes (quantize, then the GEMM on codes) as the explicit two-call path
        Aq, As = mx.quantize(Ad)
        assert torch.equal(got, mx.gemm(Aq, As, W))
    assert mx.device_error(reset=True) == 0


def test_static_scratch_rejects_sizes_beyond_its_limit():
    torch.cuda.set_device(0)
    lib, fn = _entry()
    lib.mxfp4_last_error_string.restype = ctypes.c_char_p
    M, K = 4096, 8192  # codes + scales = 17 MiB > 4 MiB
    fake = ctypes.c_void_p(1 << 20)  # never touched: the size check comes first
    status = fn(fake, K, fake, fake, M, 128, K, None)
    assert status == 2  # MXFP4_ERR_UNSUPPORTED_SHAPE, nothing launched
    assert b"4 MiB" in lib.mxfp4_last_error_string()
