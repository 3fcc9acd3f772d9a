"""Split submit (Ch. 33 §33.2, the Mirror-SD route before Figure 33.1, and
Figure 33.1): the verify step records an event after a capture layer; a
second stream waits on it and runs the draft's front projection on the
captured rows while the step's suffix runs.

Bit-exact: the step's result, argmax and logits with the split on equal
those of the same step without it; the front projection computed on the
second stream after the event equals the same projection computed after the
whole step (the captured rows it read were complete).  Ordering: the event
fires before the step's end.  Tolerance: the projection against the oracle.
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
N_PAST = 40


@pytest.fixture(scope="module")
def model():
    import __graft_entry__
    __graft_entry__.build()
    sa = torch.cuda.Stream()
    ctx = runtime.Context(SMALL, max_ctx=24 * 16, stream=sa)
    ow, dw = build_model(ctx, SMALL, seed=3)
    torch.cuda.synchronize()
    yield ctx, ow, dw, sa
    ctx.close()


def fresh_kv(ctx):
    dkv = runtime.DeviceKV(SMALL, 24, 24)
    dkv.reset(ctx)
    dkv.extend(ctx, N_PAST)
    fill_context(SMALL, dkv, None, N_PAST, seed=11)
    torch.cuda.synchronize()
    return dkv


@pytest.mark.parametrize("graph", [False, True])
def test_split_event_overlaps_the_suffix_and_changes_nothing(model, graph):
    """graph: the step without taps is recorded as a CUDA graph and launched,
    the event being an external event record node of that graph; with taps
    the step is enqueued launch by launch."""
    ctx, ow, dw, sa = model
    cfg, H, k = SMALL, SMALL.hidden, 15
    M = k + 1
    hidden = torch.from_numpy(synth.normal((M, H), 3, 900)).cuda()
    draft = torch.from_numpy(synth.tokens(k, cfg.vocab, 3, 901)).cuda()
    cap = torch.zeros((16, H), dtype=torch.float32, device="cuda")
    ids = np.array([0], dtype=np.int32)
    abi.check("spec_set_capture", abi.spec_set_capture(ctx.h, ids.ctypes.data, 1, cap.data_ptr()))

    def run(split_ev=None, fc=None):
        dkv = fresh_kv(ctx)
        res = torch.zeros(4, dtype=torch.int32, device="cuda")
        am = torch.zeros(M, dtype=torch.int32, device="cuda")
        lg = torch.zeros((M, cfg.vocab), dtype=torch.float32, device="cuda")
        end = torch.cuda.Event(enable_timing=True)
        taps = None if graph else abi.spec_taps(None, am.data_ptr(), lg.data_ptr())
        abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(),
                                                                 hidden.data_ptr(), draft.data_ptr(), k,
                                                                 res.data_ptr(), taps))
        end.record(sa)
        if fc is not None:
            fc(split_ev)
        torch.cuda.synchronize()
        return res.cpu().numpy(), am.cpu().numpy(), lg.cpu().numpy(), end

    base = run()

    # the draft side: its own spec_ctx on its own stream
    sb = torch.cuda.Stream()
    ctx_b = runtime.Context(SMALL, max_ctx=24 * 16, stream=sb)
    try:
        N_fc = 1024
        W = synth.q4k_matrix(N_fc, H, 3, 902)
        Wt = runtime.upload_tiled(ctx_b, W, N_fc, H)
        y = torch.zeros((M, N_fc), dtype=torch.float32, device="cuda")

        def fc(ev):
            sb.wait_event(ev)
            abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx_b.h, Wt.data_ptr(), N_fc, H, cap.data_ptr(), M,
                                                         y.data_ptr()))

        ev = torch.cuda.Event(enable_timing=True)
        ev.record(sa)                                # creates the event
        torch.cuda.synchronize()
        abi.check("spec_set_split", abi.spec_set_split(ctx.h, 0, ev.cuda_event))
        split = run(ev, fc)
        y_overlap = y.cpu().numpy()
        # the event fired inside the step: after it, the last block and the head ran
        assert ev.elapsed_time(split[3]) > 0.0
        # nothing about the step changed
        assert np.array_equal(split[0], base[0])
        assert np.array_equal(split[1], base[1])
        assert np.array_equal(split[2].view(np.uint32), base[2].view(np.uint32))
        # the projection read complete rows: the same call after the whole step agrees
        y.zero_()
        abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx_b.h, Wt.data_ptr(), N_fc, H, cap.data_ptr(), M,
                                                     y.data_ptr()))
        torch.cuda.synchronize()
        assert np.array_equal(y_overlap.view(np.uint32), y.cpu().numpy().view(np.uint32))
        assert_close(y_overlap, oracle.linear(W, N_fc, H, cap.cpu().numpy()), what="front projection")
        # and off again
        abi.check("spec_set_split", abi.spec_set_split(ctx.h, -1, None))
        again = run()
        assert np.array_equal(again[0], base[0])
    finally:
        abi.check("spec_set_split", abi.spec_set_split(ctx.h, -1, None))
        abi.check("spec_set_capture", abi.spec_set_capture(ctx.h, None, 0, None))
        ctx_b.close()


def test_split_rejects_bad_arguments(model):
    ctx = model[0]
    assert abi.spec_set_split(ctx.h, SMALL.n_layers, None) == abi.SPEC_EINVAL
    assert abi.spec_set_split(ctx.h, -2, None) == abi.SPEC_EINVAL
    assert abi.spec_set_split(ctx.h, 0, None) == abi.SPEC_ENULL
    assert abi.spec_set_split(ctx.h, -1, None) == abi.SPEC_OK
