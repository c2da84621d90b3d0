"""Several dependent layers in one launch (mxfp4_quant_gemm_chain), through
the C ABI, against the CPU oracle.

Each layer l is checked against the oracle's quant_gemm of the input that
layer actually received (A for the first layer, the kernel's own bf16 C_{l-1}
after that), at the parity tests' tolerance.  Identity layers check both
quantization points bit for bit: the first layer's shared quantization of A,
and a later layer's quantization of the previous layer's output, which the
kernel performs in the producing layer's epilogue."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_scaled_mxfp4_activation_gb300 as mx
import workloads
from test_gpu_parity import check_close, grid_activation, quantized_weight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mx.load_library()
    torch.cuda.set_device(0)
    mx.set_programmatic_launch(3)
    assert mx.device_error(reset=True) == 0
    yield
    assert mx.device_error(reset=True) == 0, "a device-side wait timed out during the tests"


def random_weight(oracle_mod, N: int, K: int, seed: int):
    g = np.random.default_rng(seed)
    B = torch.from_numpy((g.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)).to(torch.bfloat16)
    return quantized_weight(oracle_mod, B)


CHAINS = [
    # (M, K, [N_0, N_1, ...]): up/down pairs at the leaderboard's shapes, long K,
    # ragged M, N and K (K % 256 and K % 64 != 0, N % 128 != 0, a ragged last N)
    (32, 512, [4096, 512, 2880, 512]),
    (4, 512, [2880, 512]),
    (16, 7168, [2112, 7168]),
    (64, 2048, [7168, 2048]),
    (5, 96, [160, 64, 33]),
    (100, 288, [256, 96, 200]),
    (1, 32, [32]),
    (256, 1536, [3072, 1536]),
]


@pytest.mark.parametrize("M,K,Ns", CHAINS)
def test_chain_every_layer_against_oracle(oracle_mod, M, K, Ns):
    A = workloads.make_activation(M, K, seed=M + K)
    qs, Ws = [], []
    k = K
    for l, n in enumerate(Ns):
        bq, bs, W = random_weight(oracle_mod, n, k, seed=1000 * l + n + k)
        qs.append((bq, bs))
        Ws.append(W)
        k = n
    outs = mx.quant_gemm_chain(A.cuda(), Ws)
    torch.cuda.synchronize()
    assert mx.device_error(reset=True) == 0
    x = A
    for l, (C, (bq, bs)) in enumerate(zip(outs, qs)):
        _, _, c64, _ = oracle_mod.quant_gemm(x, bq, bs)
        check_close(C, c64, f"chain M={M} K={K} Ns={Ns}, layer {l}")
        x = C.cpu()  # the next layer's input is exactly what this layer wrote


@pytest.mark.parametrize("M", [16, 37, 64])
def test_chain_quantization_bitexact_through_identity_layers(oracle_mod, M):
    """Layer 0 = I: C_0 is the dequantized first-layer quantization of A, exactly.
    Layer 1 random.  Layer 2 = I: C_2 is the dequantized quantization of C_1 as
    the epilogue of layer 1 produced it, exactly.  Inputs sit on E2M1 rounding
    ties, signed zeros, tiny values and all-zero blocks."""
    K, N1 = 512, 768
    A = grid_activation(M, K, seed=M + 7)
    _, _, I0 = quantized_weight(oracle_mod, torch.eye(K, dtype=torch.float32).to(torch.bfloat16))
    bq1, bs1, W1 = random_weight(oracle_mod, N1, K, seed=M)
    _, _, I2 = quantized_weight(oracle_mod, torch.eye(N1, dtype=torch.float32).to(torch.bfloat16))
    C0, C1, C2 = mx.quant_gemm_chain(A.cuda(), [I0, W1, I2])
    torch.cuda.synchronize()
    aq, as_ = oracle_mod.quantize(A)
    expect0 = oracle_mod.dequantize(aq, as_)
    got0 = C0.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got0, expect0), f"first-layer quantization: {int((got0 != expect0).sum())} differ"
    _, _, c64, _ = oracle_mod.quant_gemm(C0.cpu(), bq1, bs1)
    check_close(C1, c64, f"identity chain M={M}, layer 1")
    q1, s1 = oracle_mod.quantize(C1.cpu())
    expect2 = oracle_mod.dequantize(q1, s1)
    got2 = C2.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got2, expect2), f"epilogue quantization: {int((got2 != expect2).sum())} differ"


def test_chain_repeated_and_graph_replayed_calls_agree(oracle_mod):
    """The workspace's counters return to zero after every call: repeated calls on
    one workspace, eager and graph-replayed, give identical results."""
    M, K, Ns = 32, 512, [4096, 512, 4096, 512]
    A = workloads.make_activation(M, K, seed=3).cuda()
    Ws = []
    k = K
    for l, n in enumerate(Ns):
        Ws.append(random_weight(oracle_mod, n, k, seed=50 + l)[2])
        k = n
    ws = torch.zeros(mx.chain_workspace_bytes(M, K, Ns), dtype=torch.uint8, device="cuda")
    first = [o.clone() for o in mx.quant_gemm_chain(A, Ws, workspace=ws)]
    for _ in range(3):
        again = mx.quant_gemm_chain(A, Ws, workspace=ws)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    outs = [torch.empty_like(o) for o in first]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        mx.quant_gemm_chain(A, Ws, outs=outs, workspace=ws)
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(first, outs):
            assert torch.equal(a, b)
    assert mx.device_error(reset=True) == 0
    # the per-layer entry on the same inputs agrees within the tolerance
    x = A
    for W, C in zip(Ws, first):
        ref = mx.quant_gemm(x, W)
        rms = float(ref.float().pow(2).mean().sqrt())
        assert float((ref.float() - C.float()).abs().max()) <= 8e-3 * float(ref.float().abs().max()) + 1e-2 * rms
        x = C


def test_chain_unzeroed_workspace_reports_a_timeout(oracle_mod):
    """A workspace whose counters were never zeroed: the layer hand-off waits
    (which wait for exact counts) run out and report through the device error
    word, the kernel finishes, and the context stays usable; a zeroed workspace
    then gives the right result."""
    M, K, Ns = 16, 256, [256, 128]
    A = workloads.make_activation(M, K, seed=11).cuda()
    Ws = [random_weight(oracle_mod, Ns[0], K, seed=1)[2], random_weight(oracle_mod, Ns[1], Ns[0], seed=2)[2]]
    ws = torch.full((mx.chain_workspace_bytes(M, K, Ns),), 1, dtype=torch.uint8, device="cuda")
    assert mx.device_error(reset=True) == 0
    mx.set_wait_timeout_ns(20_000_000)  # 20 ms
    try:
        mx.quant_gemm_chain(A, Ws, workspace=ws)
        code = mx.device_error(reset=True)
    finally:
        mx.set_wait_timeout_ns(0)
    assert code & (1 << 7), f"expected the hand-off wait to report, got {code:#x}"
    ws.zero_()
    outs = mx.quant_gemm_chain(A, Ws, workspace=ws)
    torch.cuda.synchronize()
    assert mx.device_error(reset=True) == 0
    ref0 = mx.quant_gemm(A, Ws[0])
    ref1 = mx.quant_gemm(outs[0], Ws[1])
    for C, ref in ((outs[0], ref0), (outs[1], ref1)):
        rms = float(ref.float().pow(2).mean().sqrt())
        assert float((ref.float() - C.float()).abs().max()) <= 8e-3 * float(ref.float().abs().max()) + 1e-2 * rms
