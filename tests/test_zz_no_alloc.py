"""spec_gemm_q4k_noalloc: the GEMM for callers that may not allocate device memory.

Some hosts cannot call the CUDA allocator at the point where they run a
projection (for example a decode loop that must never block on the allocator,
or a process whose device memory was reserved up front by another runtime).
The allocation-free entry point takes its scratch from a fixed array inside
the library.  This test calls it through the C ABI twice in a row and checks
both results against the ordinary spec_gemm_q4k (which uses a spec_ctx
workspace), within the tolerance the other GEMM tests use.  It lives in its
own file, collected last, and builds everything it needs, so it runs the same
alone in a fresh process or after the rest of the suite.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import assert_close  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    import __graft_entry__
    __graft_entry__.build()
    cfg = runtime.ModelConfig(**synth.FULL)
    c = runtime.Context(cfg, max_ctx=2112)
    yield c
    c.close()


@pytest.mark.parametrize("M,N,K", [(16, 6656, 6656), (5, 2048, 17920)])
def test_noalloc_gemm_matches_ctx_gemm_twice(ctx, M, N, K):
    W = synth.q4k_matrix(N, K, 21, N + K)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    x = torch.from_numpy(synth.normal((M, K), 21, M)).cuda()
    y_ref = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, Wt.data_ptr(), N, K, x.data_ptr(), M,
                                                 y_ref.data_ptr()))
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        abi.check("spec_gemm_q4k_noalloc",
                  abi.spec_gemm_q4k_noalloc(Wt.data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), stream))
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy())
    ref = y_ref.cpu().numpy()
    for y in outs:
        assert np.all(np.isfinite(y))
        assert_close(y, ref, what="no-alloc GEMM vs ctx GEMM")
    assert_close(outs[1], outs[0], what="second no-alloc call vs first")


def test_noalloc_gemm_rejects_oversized_requests(ctx):
    # the LM-head shape needs more partial-sum scratch than the fixed array holds
    N, K = 131072, 6656
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((16, K), dtype=torch.float32, device="cuda")
    y = torch.zeros((16, N), dtype=torch.float32, device="cuda")
    rc = abi.spec_gemm_q4k_noalloc(W.data_ptr(), N, K, x.data_ptr(), 16, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == abi.SPEC_ECAPACITY
