"""Calls from several host threads at once, each on its own stream: the
library's per-device state (scratch pool, copy streams, tensor-map encoder,
kernel attributes) and its per-thread last-kernel record must hold up. Every
result is checked against the oracle bit for bit (integer data)."""
import threading

import pytest
import torch

import oracle
from tests.parity import assert_bit_exact
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [("f32", (300, 520, 200)), ("tf32", (513, 1000, 136)), ("bf16", (640, 768, 256)),
         ("tf32x3", (256, 512, 264)), ("f32", (16, 4000, 300)), ("bf16", (1024, 1536, 1024))]
DTYPE = {"f32": torch.float32, "tf32": torch.float32, "bf16": torch.bfloat16,
         "tf32x3": torch.float32}


def test_concurrent_host_threads(tgemm):
    data = []
    for i, (path, (M, N, K)) in enumerate(CASES):
        g = inputs.generator(8100 + i)
        A = inputs.draw(M, K, "int4", g).to(DTYPE[path])
        B = inputs.draw(K, N, "int4", g).to(DTYPE[path])
        data.append((path, A, B, oracle.gemm(A, B)[0]))
    errors = []
    results = {}

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for rep in range(4):
                    for i, (path, A, B, _) in enumerate(data):
                        if (i + t + rep) % 2:
                            continue
                        Ad, Bd = A.cuda(), B.cuda()
                        if path == "f32":
                            C = tgemm.gemm_f32(Ad, Bd)
                        else:
                            C = tgemm.gemm_tc(Ad, Bd, path)
                        name = tgemm.binding.last_kernel()
                        stream.synchronize()
                        results[(t, rep, i)] = (C.cpu(), name)
        except Exception as e:                      # reported below, in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert tgemm.device_status() == 0
    assert len(results) == 4 * 4 * len(data) // 2
    for (t, rep, i), (C, name) in results.items():
        path = data[i][0]
        # the last-kernel record is per thread: it names this thread's call
        expect = {"f32": "f32_", "tf32": "tc_tf32_", "bf16": "tc_bf16_", "tf32x3": "tc_tf32x3_"}[path]
        assert expect in name, (path, name)
        assert_bit_exact(C, data[i][3], f"thread {t} rep {rep} {path}")
