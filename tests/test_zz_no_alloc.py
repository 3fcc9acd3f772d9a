"""spec_gemm_q4k_noalloc: the GEMM for callers that may not allocate device memory.

Some hosts cannot call the CUDA allocator at the point where they run a
projection (for example a decode loop that must never block on the allocator,
or a process whose device memory was reserved up front by another runtime).
The allocation-free entry point takes its scratch from a fixed array inside
the library.  It runs the same quantiser, GEMM and ordered piece-sum kernels
under the same work plan as spec_gemm_q4k (which uses a spec_ctx workspace),
so its output must be bit-identical to that entry point's, call after call.
The tests here call it through the C ABI twice in a row, read its status word
back after each call, and run it once in a fresh process before any spec_ctx
exists (its own first-call set-up is then the only one).  The file is
collected last and builds everything it needs, so it runs the same alone in a
fresh process or after the rest of the suite.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
        assert abi.spec_gemm_q4k_noalloc_status(stream) == 0
        outs.append(y.cpu().numpy())
    ref = y_ref.cpu().numpy()
    for y in outs:
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), "no-alloc GEMM differs from ctx GEMM"


def test_noalloc_gemm_reports_nonfinite_input(ctx):
    N, K, M = 256, 512, 3
    W = synth.q4k_matrix(N, K, 22, 1)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    x = synth.normal((M, K), 22, 2)
    x[1, 300] = np.inf
    xd = torch.from_numpy(x).cuda()
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    abi.check("spec_gemm_q4k_noalloc",
              abi.spec_gemm_q4k_noalloc(Wt.data_ptr(), N, K, xd.data_ptr(), M, y.data_ptr(), stream))
    assert abi.spec_gemm_q4k_noalloc_status(stream) & abi.ST_NONFINITE
    # the next call starts from a clear word
    xd.copy_(torch.from_numpy(synth.normal((M, K), 22, 3)))
    abi.check("spec_gemm_q4k_noalloc",
              abi.spec_gemm_q4k_noalloc(Wt.data_ptr(), N, K, xd.data_ptr(), M, y.data_ptr(), stream))
    assert abi.spec_gemm_q4k_noalloc_status(stream) == 0


def test_noalloc_gemm_rejects_oversized_requests(ctx):
    # the LM-head shape needs more partial-sum scratch than the fixed array holds
    N, K = 131072, 6656
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((16, K), dtype=torch.float32, device="cuda")
    y = torch.zeros((16, N), dtype=torch.float32, device="cuda")
    rc = abi.spec_gemm_q4k_noalloc(W.data_ptr(), N, K, x.data_ptr(), 16, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == abi.SPEC_ECAPACITY


_FRESH = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    from speculative_decoding_exact_gb300 import abi, runtime, synth

    N, K, M = 2048, 6656, 16
    W = synth.q4k_matrix(N, K, 23, 1)
    # the tiled layout of include/spec_verify.h, built here without a ctx:
    # per 128-column tile T, superblock b, column c at (128*T*nb + b*cols + c)*144
    nb = K // 256
    sb = W.reshape(N, nb, 144)
    tiled = np.concatenate([sb[t:t + 128].transpose(1, 0, 2).reshape(-1) for t in range(0, N, 128)])
    Wt = torch.from_numpy(tiled).cuda()
    x = torch.from_numpy(synth.normal((M, K), 23, 2)).cuda()
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # first: the allocation-free call, before any spec_ctx exists in this process
    abi.check("noalloc", abi.spec_gemm_q4k_noalloc(Wt.data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), stream))
    assert abi.spec_gemm_q4k_noalloc_status(stream) == 0
    first = y.cpu().numpy()
    # then the ordinary entry point on the same tiled weights
    ctx = runtime.Context(runtime.ModelConfig(**synth.FULL), max_ctx=2112)
    y2 = torch.zeros_like(y)
    abi.check("gemm", abi.spec_gemm_q4k(ctx.h, Wt.data_ptr(), N, K, x.data_ptr(), M, y2.data_ptr()))
    torch.cuda.synchronize()
    assert np.array_equal(first.view(np.uint32), y2.cpu().numpy().view(np.uint32))
    ctx.close()
    print("fresh-process no-alloc call ok")
""")


def test_noalloc_gemm_first_call_in_a_fresh_process():
    import __graft_entry__
    __graft_entry__.build()
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=ROOT)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process no-alloc call ok" in r.stdout
