"""Host-only checks of the C ABI: the library builds and loads, exports every
function include/mxfp4.h declares, and rejects bad arguments with the
documented status before touching a GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import block_scaled_mxfp4_activation_gb300 as mx

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mxfp4.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WS_SMALL, CUDA, TIMEOUT, DEVICE = range(8)


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return mx.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mxfp4_quantize", "mxfp4_pack_weights", "mxfp4_gemm", "mxfp4_quant_gemm",
                     "mxfp4_packed_weight_bytes", "mxfp4_workspace_bytes", "mxfp4_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for s in range(8):
        assert lib.mxfp4_status_string(s)
    assert lib.mxfp4_status_string(99) == b"unknown status"


def test_packed_weight_bytes_layout(lib):
    # codes [roundup(N,128), K/2] then scales at a 1 KB boundary:
    # one 1 KB block per 128-row x 256-column tile
    for N, K in ((2880, 512), (2112, 7168), (7168, 2048), (3072, 1536), (1, 32), (129, 288)):
        n_pad = -(-N // 128) * 128
        data = n_pad * K // 2
        sf_off = -(-data // 1024) * 1024
        expect = sf_off + (n_pad // 128) * (-(-K // 256)) * 1024
        assert lib.mxfp4_packed_weight_bytes(N, K) == expect
    assert lib.mxfp4_packed_weight_bytes(16, 48) == 0  # K % 32 != 0
    assert lib.mxfp4_packed_weight_bytes(0, 64) == 0
    assert lib.mxfp4_workspace_bytes(16, 2112, 7168) == 0  # single fused kernel
    # from M = 64 on: room for the codes and scales of A, each rounded to 256 bytes
    assert lib.mxfp4_workspace_bytes(64, 7168, 2048) == 64 * 1024 + 64 * 64
    assert lib.mxfp4_workspace_bytes(200, 128, 96) == 9728 + 768
    assert lib.mxfp4_workspace_bytes(64, 128, 40) == 0
    # ... except while M <= 128 and the single kernel's bf16 re-reads,
    # 2*M*K per 128-row N tile, stay within 5 MiB
    mib5 = 5 << 20
    for M, N, K in ((100, 128, 96), (128, 4096, 512), (65, 3072, 1536), (128, 2560, 1024), (64, 7168, 2048),
                    (128, 2688, 1024), (129, 128, 96), (96, 7168, 7168)):
        reread = 2 * M * K * (-(-N // 128))
        two = M > 128 or reread > mib5
        assert (lib.mxfp4_workspace_bytes(M, N, K) > 0) == two, (M, N, K, reread)
    # a shape whose tuned plan is the single fused kernel at M = 64
    assert lib.mxfp4_workspace_bytes(64, 3072, 1536) == 0


def test_argument_checks_launch_nothing(lib):
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x10001)
    assert lib.mxfp4_quantize(None, 4, 64, 64, fake, fake, None) == INVALID
    assert lib.mxfp4_quantize(fake, 4, 48, 48, fake, fake, None) == INVALID  # K % 32
    assert lib.mxfp4_quantize(fake, 4, 64, 32, fake, fake, None) == INVALID  # lda < K
    assert lib.mxfp4_quantize(fake, 0, 64, 64, fake, fake, None) == INVALID
    assert lib.mxfp4_quantize(odd, 4, 64, 64, fake, fake, None) == MISALIGNED
    assert lib.mxfp4_quantize(fake, 4, 64, 68, fake, fake, None) == MISALIGNED  # lda % 8
    assert lib.mxfp4_pack_weights(fake, None, 128, 64, fake, None) == INVALID
    assert lib.mxfp4_pack_weights(fake, fake, 128, 80, fake, None) == INVALID
    assert lib.mxfp4_pack_weights(odd, fake, 128, 64, fake, None) == MISALIGNED
    assert lib.mxfp4_gemm(fake, None, fake, fake, 4, 128, 64, None, 0, None) == INVALID
    assert lib.mxfp4_gemm(fake, fake, fake, fake, 4, 128, 40, None, 0, None) == INVALID
    assert lib.mxfp4_gemm(fake, fake, odd, fake, 4, 128, 64, None, 0, None) == MISALIGNED
    assert lib.mxfp4_quant_gemm(fake, 64, fake, None, 4, 128, 64, None, 0, None) == INVALID
    assert lib.mxfp4_quant_gemm(fake, 60, fake, fake, 4, 128, 64, None, 0, None) == INVALID  # lda < K
    assert lib.mxfp4_quant_gemm(fake, 68, fake, fake, 4, 128, 64, None, 0, None) == MISALIGNED  # lda % 8
    assert lib.mxfp4_quant_gemm(fake, 64, fake, fake, 4, 0, 64, None, 0, None) == INVALID
    assert lib.mxfp4_quant_gemm(fake, 1 << 40, fake, fake, 1 << 31, 128, 1 << 31, None, 0, None) == UNSUPPORTED
    # sizes past the library's limits (32-bit in-kernel indices), on every compute entry
    assert lib.mxfp4_quantize(fake, 1 << 40, 64, 64, fake, fake, None) == UNSUPPORTED
    assert lib.mxfp4_gemm(fake, fake, fake, fake, 4, 1 << 40, 64, None, 0, None) == UNSUPPORTED
    assert lib.mxfp4_gemm(fake, fake, fake, fake, 1 << 20, 1 << 20, 64, None, 0, None) == UNSUPPORTED  # M*N > 2^31
    assert lib.mxfp4_quant_gemm_host(fake, 64, fake, 64, fake, fake, fake, 4, 1 << 40, 64, None, 0, None) == UNSUPPORTED
    assert lib.mxfp4_quant_gemm_host(None, 64, fake, 64, fake, fake, fake, 4, 128, 64, None, 0, None) == INVALID
    assert lib.mxfp4_quant_gemm_host(fake, 64, fake, 68, fake, fake, fake, 4, 128, 64, None, 0, None) == MISALIGNED
    assert lib.mxfp4_quant_gemm_host(fake, 64, odd, 64, fake, fake, fake, 4, 128, 64, None, 0, None) == MISALIGNED
    assert lib.mxfp4_pack_weights_shuffled(fake, fake, 24, 128, fake, None) == INVALID  # N % 16
    assert lib.mxfp4_pack_weights_shuffled(fake, fake, 32, 96, fake, None) == INVALID  # K % 64
    assert lib.mxfp4_pack_weights_shuffled(fake, fake, 32, 128, odd, None) == MISALIGNED
    assert lib.mxfp4_gemm_plan(4, 128, 64, 1, None) == INVALID
    assert lib.mxfp4_device_error(None, 0, None) == INVALID
    # the fused entry's workspace: offered but too small for the two-pass route
    # (here M > 128), offered as a null pointer, or misaligned
    assert lib.mxfp4_quant_gemm(fake, 64, fake, fake, 200, 128, 64, fake, 16, None) == WS_SMALL
    assert lib.mxfp4_quant_gemm(fake, 64, fake, fake, 200, 128, 64, None, 1 << 20, None) == INVALID
    assert lib.mxfp4_quant_gemm(fake, 64, fake, fake, 200, 128, 64, odd, 1 << 20, None) == MISALIGNED
    assert lib.mxfp4_quant_gemm_host(fake, 64, fake, 64, fake, fake, fake, 200, 128, 64, fake, 16, None) == WS_SMALL


def test_static_scratch_entry_checks_launch_nothing(lib):
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x10001)
    fn = lib.mxfp4_quant_gemm_static_scratch
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    lib.mxfp4_last_error_string.restype = ctypes.c_char_p
    assert fn(fake, 64, fake, None, 4, 128, 64, None) == INVALID  # null C
    assert fn(None, 64, fake, fake, 4, 128, 64, None) == INVALID  # null A
    assert fn(fake, 32, fake, fake, 4, 128, 64, None) == INVALID  # lda < K
    assert fn(fake, 48, fake, fake, 4, 128, 48, None) == INVALID  # K % 32
    assert fn(fake, 64, fake, fake, 0, 128, 64, None) == INVALID
    assert fn(odd, 64, fake, fake, 4, 128, 64, None) == MISALIGNED
    assert fn(fake, 64, odd, fake, 4, 128, 64, None) == MISALIGNED
    assert fn(fake, 64, fake, odd, 4, 128, 64, None) == MISALIGNED
    assert fn(fake, 68, fake, fake, 4, 128, 64, None) == MISALIGNED  # lda % 8
    # the kernels' index limits, with an activation that fits the 4 MiB scratch
    assert fn(fake, 64, fake, fake, 1 << 11, 1 << 21, 64, None) == UNSUPPORTED  # M * N > 2^31
    assert fn(fake, 1 << 22, fake, fake, 1, 1 << 20, 1 << 22, None) == UNSUPPORTED  # K/2 * N > 2^40
    # the scratch limit itself, named by the error string
    assert fn(fake, 8192, fake, fake, 4096, 128, 8192, None) == UNSUPPORTED
    assert b"4 MiB" in lib.mxfp4_last_error_string()


def test_python_binding_refuses_cpu_tensors():
    import torch

    with pytest.raises(TypeError):
        mx.quantize(torch.zeros(4, 64, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        mx.quant_gemm(torch.zeros(4, 64, dtype=torch.bfloat16), mx.PackedWeight(torch.zeros(8, dtype=torch.uint8), 128, 64))


def test_prepared_calls_check_their_arguments_once():
    import torch

    W = mx.PackedWeight(torch.zeros(8, dtype=torch.uint8), 128, 64)
    cpu = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        mx.prepare_quant_gemm(cpu, W)
    with pytest.raises(TypeError):  # A_dev on the host
        mx.prepare_quant_gemm_host(cpu, W, cpu, cpu, torch.zeros(4, 128, dtype=torch.bfloat16))



def chain_workspace_expected(M: int, K: int, Ns: list[int]) -> int:
    """The multi-layer workspace, restated: per layer codes, scale chunks and
    split-K partials (for up to min(8, K tiles) splits), then the counters."""
    a256 = lambda x: -(-x // 256) * 256
    bm = 16 if M <= 32 else 64
    mt = -(-M // bm)
    total, counters, k = 0, 0, K
    for n in Ns:
        kt, nt = -(-k // 256), -(-n // 128)
        smax = min(8, kt)
        total += a256(M * k // 2) + a256(mt * kt * 1024)
        if smax > 1:
            total += a256(nt * mt * smax * bm * 128 * 4)
        counters += mt * kt + nt * mt
        k = n
    return total + a256((counters + 1) * 4)


def test_chain_workspace_bytes(lib):
    fn = lib.mxfp4_chain_workspace_bytes
    fn.restype = ctypes.c_size_t
    for M, K, Ns in ((32, 512, [4096, 512]), (5, 96, [160, 64, 33]), (256, 1536, [3072, 1536]), (1, 32, [32]),
                     (100, 288, [256, 96, 200])):
        arr = (ctypes.c_int64 * len(Ns))(*Ns)
        assert fn(M, K, len(Ns), arr) == chain_workspace_expected(M, K, Ns), (M, K, Ns)
    arr = (ctypes.c_int64 * 2)(100, 64)
    assert fn(4, 512, 2, arr) == 0  # layer 1's K = 100 is not a multiple of 32
    assert fn(4, 512, 0, arr) == 0
    assert fn(4, 512, 17, (ctypes.c_int64 * 17)(*([512] * 17))) == 0


def test_chain_argument_checks_launch_nothing(lib):
    fake = 0x10000
    fn = lib.mxfp4_quant_gemm_chain
    P = ctypes.c_void_p

    def call(A=fake, lda=512, M=32, K=512, Ns=(4096, 512), B=None, C=None, ws=fake, ws_bytes=1 << 30,
             L=None):
        L = len(Ns) if L is None else L
        n = (ctypes.c_int64 * max(1, len(Ns)))(*Ns)
        b = (P * max(1, len(Ns)))(*([fake] * len(Ns) if B is None else B))
        c = (P * max(1, len(Ns)))(*([fake] * len(Ns) if C is None else C))
        return fn(A, lda, M, K, L, b, n, c, ws, ws_bytes, None)

    assert call(L=0) == INVALID
    assert call(L=17, Ns=[512] * 17) == INVALID
    assert call(A=None) == INVALID
    assert call(lda=256) == INVALID  # lda < K
    assert call(K=48) == INVALID
    assert call(Ns=(100, 512)) == INVALID  # layer 1's K = N_0 not a multiple of 32
    assert call(B=[fake, None]) == INVALID
    assert call(C=[None, fake]) == INVALID
    assert call(ws=None) == INVALID
    assert call(ws_bytes=1024) == WS_SMALL
    assert call(ws=fake + 16) == MISALIGNED  # the workspace must be 256-byte aligned
    assert call(A=fake + 8) == MISALIGNED
    assert call(lda=516) == MISALIGNED
    assert call(C=[fake, fake + 8]) == MISALIGNED
    assert call(M=1 << 20, Ns=(1 << 12, 512)) == UNSUPPORTED  # M * N > 2^31
