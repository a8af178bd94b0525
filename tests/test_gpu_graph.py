"""Products captured in a CUDA graph and replayed.

Every kernel of the library is launched with programmatic dependent launch
(it may start while the previous kernel in the stream finishes, and waits
for that kernel before touching memory); in a captured graph those launches
become programmatic dependency edges. Each test captures a sequence of
products on a side stream with torch.cuda.graph, then replays the graph
several times with new operands copied into the captured input buffers,
checking every replay bit for bit against the oracle (integer data).
"""
import pytest
import torch

import oracle
from tests.parity import assert_bit_exact
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu


def draw(M, N, K, dtype, seed):
    g = inputs.generator(seed)
    return inputs.draw(M, K, "int4", g).to(dtype), inputs.draw(K, N, "int4", g).to(dtype)


def capture(fn):
    """Warm the calls up once (first-call set-up happens outside capture),
    then capture them in a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def test_chain_of_products_replays(tgemm):
    """FP32 (one whole wave), TF32 and BF16 products that need no scratch,
    the second reading the first's result: dependent launches in sequence."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 128 * (sms // 8), 256 * 8, 256          # FP32: one wave of 128 x 256 tiles
    A = torch.empty(M, K, device="cuda")
    B = torch.empty(K, N, device="cuda")
    B2 = torch.empty(N, 64, device="cuda")
    Ab = torch.empty(M, K, device="cuda", dtype=torch.bfloat16)
    Bb = torch.empty(K, N, device="cuda", dtype=torch.bfloat16)
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(M, 64, device="cuda")
    C3 = torch.empty(M, N, device="cuda")
    assert tgemm.binding.scratch_bytes(A, B, "f32") == 0
    assert tgemm.binding.set_tc_streamk(0) == 0          # no stream-K tail: no scratch
    try:
        def products():
            tgemm.gemm_f32(A, B, out=C1)
            tgemm.gemm_tc(C1, B2, "tf32", out=C2)      # reads the FP32 product
            tgemm.gemm_tc(Ab, Bb, "bf16", out=C3)
        graph = capture(products)
        for replay in range(3):
            a, b = draw(M, N, K, torch.float32, 100 + replay)
            _, b2 = draw(1, 64, N, torch.float32, 200 + replay)
            b2 = (b2 / 4).round()                          # keeps C1 @ B2 exact in TF32 and FP32
            ab, bb = draw(M, N, K, torch.bfloat16, 300 + replay)
            A.copy_(a); B.copy_(b); B2.copy_(b2); Ab.copy_(ab); Bb.copy_(bb)
            graph.replay()
            torch.cuda.synchronize()
            assert tgemm.device_status() == 0
            c1 = oracle.gemm(a, b)[0]
            assert_bit_exact(C1, c1, f"replay {replay}: f32")
            assert_bit_exact(C2, oracle.gemm(torch.from_numpy(c1).float(), b2)[0], f"replay {replay}: tf32")
            assert_bit_exact(C3, oracle.gemm(ab, bb)[0], f"replay {replay}: bf16")
    finally:
        tgemm.binding.set_tc_streamk(-1)


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
def test_tensor_products_with_scratch_replay(tgemm, kind):
    """Rows off 16 bytes (repack pre-passes) and a split last round (the
    reduction kernel): four dependent launches per product, the scratch
    drawn from the library's pool inside the graph."""
    M, N, K = 700, 1001, 517
    dtype = torch.float32 if kind == "tf32" else torch.bfloat16
    A = torch.empty(M, K, device="cuda", dtype=dtype)
    B = torch.empty(K, N, device="cuda", dtype=dtype)
    C = torch.empty(M, N, device="cuda")
    graph = capture(lambda: tgemm.gemm_tc(A, B, kind, out=C))
    name = tgemm.binding.last_kernel()
    assert "repack_ab+" in name, name
    for replay in range(3):
        a, b = draw(M, N, K, dtype, 400 + replay)
        A.copy_(a); B.copy_(b)
        graph.replay()
        torch.cuda.synchronize()
        assert tgemm.device_status() == 0
        assert_bit_exact(C, oracle.gemm(a, b)[0], f"{kind} replay {replay}")
