"""Hidden-state capture for the draft's front projection (Ch. 8: the draft
reads the target's hidden states at pinned layers, concatenated, through fc).

Bit-exact: the captured rows equal the step's residual taps of the same
layers (block outputs), in the order the layer ids were given, for the
graph-replayed step and the directly enqueued one alike.  Tolerance: the fc
projection of the captured rows (Q4_K, K = n*H) against the oracle.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import assert_close  # noqa: E402
from tests.model_util import build_model, fill_context, ocfg_of  # noqa: E402

SMALL = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=26, n_kv_heads=2, head_dim=128,
                            ffn=8960, vocab=4096)


@pytest.fixture(scope="module")
def model():
    import __graft_entry__
    __graft_entry__.build()
    ctx = runtime.Context(SMALL, max_ctx=24 * 16)
    ow, dw = build_model(ctx, SMALL, seed=3)
    yield ctx, ow, dw
    ctx.close()


def step(ctx, dw, hidden, draft, taps=None):
    cfg, k = SMALL, len(draft)
    dkv = runtime.DeviceKV(cfg, 24, 24)
    dkv.reset(ctx)
    dkv.extend(ctx, 40)
    okv = oracle.KV(ocfg_of(cfg), 24, 24)
    okv.extend(40)
    fill_context(cfg, dkv, okv, 40, seed=11)
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    h = torch.from_numpy(hidden).cuda()
    d = torch.from_numpy(draft).cuda()
    if taps is None:
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(),
                                                           d.data_ptr(), k, res.data_ptr()))
    else:
        abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(),
                                                                 d.data_ptr(), k, res.data_ptr(), taps))
    torch.cuda.synchronize()
    assert res.cpu().numpy()[2] == 0


def test_capture_equals_residual_taps_and_feeds_fc(model):
    ctx, ow, dw = model
    cfg, H, k = SMALL, SMALL.hidden, 15
    M = k + 1
    ids = np.array([1, 0], dtype=np.int32)            # concatenation order = the given order
    n = len(ids)
    rows = torch.full((16, n * H), -7.0, dtype=torch.float32, device="cuda")
    abi.check("spec_set_capture", abi.spec_set_capture(ctx.h, ids.ctypes.data, n, rows.data_ptr()))
    hidden = synth.normal((M, H), 3, 901)
    draft = synth.tokens(k, cfg.vocab, 3, 902)
    resid = torch.zeros((cfg.n_layers + 1, M, H), dtype=torch.float32, device="cuda")
    step(ctx, dw, hidden, draft, abi.spec_taps(resid.data_ptr(), None, None))
    cap_taps = rows.cpu().numpy().copy()
    r = resid.cpu().numpy()
    for j, l in enumerate(ids):
        assert np.array_equal(cap_taps[:M, j * H:(j + 1) * H].view(np.uint32), r[l + 1].view(np.uint32)), l
    assert np.all(cap_taps[M:] == -7.0)               # rows >= M untouched
    # the graph-replayed step (no taps) captures the same rows
    rows.fill_(0.0)
    step(ctx, dw, hidden, draft)
    step(ctx, dw, hidden, draft)                     # second call replays the recorded graph
    assert np.array_equal(rows.cpu().numpy()[:M].view(np.uint32), cap_taps[:M].view(np.uint32))
    # the front projection of the captured rows: Q4_K, K = n*H -> H
    K = n * H
    Wfc = synth.q4k_matrix(H, K, 9, 77)
    Wt = runtime.upload_tiled(ctx, Wfc, H, K)
    y = torch.zeros((M, H), dtype=torch.float32, device="cuda")
    abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, Wt.data_ptr(), H, K, rows.data_ptr(), M, y.data_ptr()))
    torch.cuda.synchronize()
    oy = oracle.linear(Wfc, H, K, np.ascontiguousarray(cap_taps[:M]))
    assert_close(y.cpu().numpy(), oy, what="fc of the captured rows")
    # off again: nothing written
    abi.check("spec_set_capture", abi.spec_set_capture(ctx.h, None, 0, None))
    rows.fill_(3.0)
    step(ctx, dw, hidden, draft)
    assert np.all(rows.cpu().numpy() == 3.0)


def test_capture_argument_checks(model):
    ctx = model[0]
    rows = torch.zeros((16, 8 * SMALL.hidden), dtype=torch.float32, device="cuda")
    bad = [(np.array([0, 0], dtype=np.int32), 2), (np.array([2], dtype=np.int32), 1),
           (np.array([-1], dtype=np.int32), 1), (np.zeros(9, dtype=np.int32), 9)]
    for ids, n in bad:
        assert abi.spec_set_capture(ctx.h, ids.ctypes.data, n, rows.data_ptr()) == abi.SPEC_EINVAL
    assert abi.spec_set_capture(ctx.h, np.array([1], dtype=np.int32).ctypes.data, 1, None) == abi.SPEC_ENULL
    assert abi.spec_set_capture(ctx.h, None, 0, None) == 0
