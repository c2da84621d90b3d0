"""The checked build (libmxfp4_checked.so, compiled with -DMXFP4_CHECKED)
beside the normal library.

In the checked build every computed-index access the kernels make outside a
TMA copy (activation loads, scale loads, code and scale stores, C stores on
each path, split-K partial sums in shared memory, cluster pushes, the
multi-layer kernel's workspace traffic) is tested against its buffer first; a
miss skips the access and sets bit 8 of the device error word.  Running every
entry point on ragged shapes through both libraries must give bit-identical
results (the guards change no arithmetic) and leave the checked library's
error word at zero (no access of the normal build falls outside its buffer)."""
from __future__ import annotations

import pytest
import torch

import block_scaled_mxfp4_activation_gb300 as mx
import workloads

pytestmark = pytest.mark.gpu

BOUNDS_BIT = 1 << 8


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mx.load_library()
    torch.cuda.set_device(0)
    mx.set_programmatic_launch(3)
    assert mx.device_error(reset=True) == 0
    yield
    assert mx.device_error(reset=True) == 0


def run_both(fn):
    """fn() under the normal library, then under the checked one; returns both
    results (lists of tensors) and the checked library's error word."""
    normal = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    assert mx.device_error(reset=True) == 0
    with mx.checked_library():
        mx.set_programmatic_launch(3)
        assert mx.device_error(reset=True) == 0
        checked = [t.clone() for t in fn()]
        torch.cuda.synchronize()
        code = mx.device_error(reset=True)
    return normal, checked, code


def assert_same(fn, what: str):
    normal, checked, code = run_both(fn)
    assert code == 0, f"{what}: checked build reported {code:#x} (bounds bit {bool(code & BOUNDS_BIT)})"
    assert len(normal) == len(checked)
    for i, (a, b) in enumerate(zip(normal, checked)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{what}: output {i} differs"


def weight(M: int, N: int, K: int, seed: int) -> mx.PackedWeight:
    return mx.quantize_weights(workloads.make_random(M, N, K, seed=seed)[1].cuda())


@pytest.mark.parametrize("M,K,pad", [(1, 32, 0), (37, 96, 32), (300, 2080, 8), (16, 7168, 0)])
def test_quantize(M, K, pad):
    A = torch.zeros((M, K + pad), dtype=torch.bfloat16, device="cuda")
    A[:, :K] = workloads.make_activation(M, K, seed=M + K).cuda()
    assert_same(lambda: list(mx.quantize(A[:, :K])), f"quantize {M}x{K} lda={K + pad}")


def test_every_plan_on_a_ragged_shape():
    # ragged M, N (not a multiple of 128 or of 8) and K (last K tile of 3 steps)
    M, N, K = 40, 131, 2048 - 64
    A = workloads.make_random(M, N, K, seed=5)[0].cuda()
    W = weight(M, N, K, seed=5)
    Aq, As = mx.quantize(A)
    plans = [{"block_m": bm, "splits": s, "stages": 2} for bm in (16, 32, 64, 128, 256) for s in (1, 2, 4, 8)]

    def run():
        outs = []
        for plan in plans:
            for fused in (True, False):
                try:
                    outs.append(mx.gemm_with_plan(A if fused else Aq, None if fused else As, W, plan, fused))
                except mx.MXFP4Error as e:
                    assert e.status == 1  # does not fit: rejected by both libraries alike
        return outs

    assert_same(run, f"every plan {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,share", [(16, 384, 1536, 2), (30, 264, 1024, 4), (5, 131, 512, 2)])
def test_shared_quantization(M, N, K, share):
    A = workloads.make_random(M, N, K, seed=M)[0].cuda()
    W = weight(M, N, K, seed=M)

    def run():
        outs = []
        for bm, splits in ((16, 1), (16, 3), (32, 2)):
            try:
                outs.append(mx.gemm_with_plan(A, None, W, {"block_m": bm, "splits": splits, "share": share}, True))
            except mx.MXFP4Error as e:
                assert e.status == 1
        return outs

    assert_same(run, f"share={share} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(32, 4096, 512), (4, 2880, 512), (16, 2112, 7168), (64, 7168, 2048),
                                   (100, 131, 288), (256, 264, 1536)])
def test_default_entries(M, N, K):
    """The default plans, the two-pass route (M >= 64 with a workspace) and the
    unfused GEMM entry."""
    A = workloads.make_random(M, N, K, seed=N)[0].cuda()
    W = weight(M, N, K, seed=N)
    ws = torch.empty(max(mx.workspace_bytes(M, N, K), 1), dtype=torch.uint8, device="cuda")

    def run():
        Aq, As = mx.quantize(A)
        return [mx.quant_gemm(A, W), mx.quant_gemm(A, W, workspace=ws), mx.gemm(Aq, As, W)]

    assert_same(run, f"default entries {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,lda", [(5, 264, 512, 520), (32, 512, 512, 512), (7, 131, 4096, 4096)])
def test_host_buffer_entry(M, N, K, lda):
    A = workloads.make_random(M, N, K, seed=K)[0]
    W = weight(M, N, K, seed=K)
    Ah = torch.zeros((M, lda), dtype=torch.bfloat16)
    Ah[:, :K] = A
    Ah = Ah.pin_memory()
    Ad = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def run():
        Ch = torch.full((M, N), float("nan"), dtype=torch.bfloat16).pin_memory()
        mx.quant_gemm_host(Ah[:, :K], W, Ad, Cd, Ch)
        torch.cuda.synchronize()
        return [Ch.cuda(), Cd]

    assert_same(run, f"host entry {M}x{N}x{K} lda={lda}")


@pytest.mark.parametrize("M,K,Ns", [(5, 96, [160, 64, 33]), (100, 288, [256, 96, 200]), (32, 512, [4096, 512]),
                                    (16, 7168, [2112, 7168]), (256, 1536, [3072, 1536])])
def test_multi_layer_entry(M, K, Ns):
    A = workloads.make_activation(M, K, seed=M).cuda()
    Ws, k = [], K
    for l, n in enumerate(Ns):
        Ws.append(weight(M, n, k, seed=10 * l + n))
        k = n
    ws = torch.zeros(mx.chain_workspace_bytes(M, K, Ns), dtype=torch.uint8, device="cuda")
    assert_same(lambda: mx.quant_gemm_chain(A, Ws, workspace=ws), f"multi-layer {M}x{K} {Ns}")
