"""The whole verify step on the GPU against the oracle (small model with the full
model's 13:1 query/KV grouping), through spec_verify_step_ex / _host.

Bit-exact: accepted length, next token, status, committed KV metadata, every
row's argmax.  An argmax is only comparable where the oracle's top-2 gap
exceeds 1e-2; every test counts the rows below it and requires that count to
be 0 for its inputs.  Tolerance: logits and the per-layer residual stream,
teacher-forced per layer (the oracle block runs on the GPU's own input to that
layer).
"""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import assert_close, require_clear_rows  # noqa: E402
from tests.model_util import add_qk_norm, build_model, fill_context, ocfg_of  # noqa: E402

SMALL = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=26, n_kv_heads=2, head_dim=128,
                            ffn=8960, vocab=4096)
N_PAST = 71          # the 16-row block straddles a page boundary
PAGES = 24


@pytest.fixture(scope="module")
def model():
    import __graft_entry__
    __graft_entry__.build()
    ctx = runtime.Context(SMALL, max_ctx=PAGES * 16)
    ow, dw = build_model(ctx, SMALL, seed=3)
    yield ctx, ow, dw
    ctx.close()


def fresh_kv(ctx, n_past=N_PAST):
    cfg = SMALL
    dkv = runtime.DeviceKV(cfg, PAGES, PAGES)
    dkv.reset(ctx)
    dkv.extend(ctx, n_past)
    okv = oracle.KV(ocfg_of(cfg), PAGES, PAGES)
    okv.extend(n_past)
    fill_context(cfg, dkv, okv, n_past, seed=11)
    return dkv, okv


def gpu_step(ctx, dw, dkv, hidden, draft, taps=True):
    k = len(draft)
    M = k + 1
    h_d = torch.from_numpy(np.ascontiguousarray(hidden)).cuda()
    d_d = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).cuda()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = {}
    t = None
    if taps:
        out["resid"] = torch.zeros((SMALL.n_layers + 1, M, SMALL.hidden), dtype=torch.float32, device="cuda")
        out["argmax"] = torch.zeros(M, dtype=torch.int32, device="cuda")
        out["logits"] = torch.zeros((M, SMALL.vocab), dtype=torch.float32, device="cuda")
        t = abi.spec_taps(out["resid"].data_ptr(), out["argmax"].data_ptr(), out["logits"].data_ptr())
    rc = abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(), h_d.data_ptr(), d_d.data_ptr(),
                                 k, res.data_ptr(), t)
    abi.check("spec_verify_step_ex", rc)
    torch.cuda.synchronize()
    return res.cpu().numpy(), {k_: v.cpu().numpy() for k_, v in out.items()}


def test_step_matches_oracle_and_is_teacher_forced_per_layer(model):
    ctx, ow, dw = model
    cfg, ocfg = SMALL, ocfg_of(SMALL)
    k = 15
    hidden = synth.normal((k + 1, cfg.hidden), 3, 500)
    dkv, okv = fresh_kv(ctx)
    # target argmax of every row (oracle), then plant drafts
    oidx, olog, ores_resid, st = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True, resid=True)
    assert st == 0
    _, gap = oracle.argmax(olog)
    require_clear_rows(gap, "step rows")
    for L_t in (0, 6, 15):
        dkv, okv = fresh_kv(ctx)
        draft = synth.plant_draft(oidx, L_t, cfg.vocab, 3, 600 + L_t)
        ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        res, taps = gpu_step(ctx, dw, dkv, hidden, draft)
        assert_close(taps["logits"], olog2, what="logits")
        assert np.array_equal(taps["argmax"], oidx2)
        assert list(res) == list(ores), (list(res), list(ores))
        # committed KV metadata
        s = dkv.state()
        oc = okv.committed()
        assert s[0] == oc[0] and np.array_equal(s[1], oc[1]) and np.all(s[2] == -1)
        assert np.array_equal(s[3], oc[3])
        # retained rows of the block (positions n_past .. seq_len-1), every layer
        pool = dkv.pool.view(torch.int16).cpu().numpy().view(np.uint16)
        diff = 0
        total = 0
        for pos in range(N_PAST, oc[0]):
            gp, op_ = s[1][pos // 16], oc[1][pos // 16]
            a = pool[gp, :, :, :, pos % 16].astype(np.int32)
            b = okv.pool[op_, :, :, :, pos % 16].astype(np.int32)
            diff += int(np.sum(a != b))
            total += a.size
            assert np.max(np.abs(a - b)) <= 1, "K/V row differs by more than one bf16 ulp"
        assert diff <= max(1, total // 1000), f"{diff} of {total} K/V values differ by one ulp"
    # teacher-forced per layer: oracle block on the GPU's own layer input
    dkv, okv = fresh_kv(ctx)
    draft = synth.plant_draft(oidx, 15, cfg.vocab, 3, 700)
    res, taps = gpu_step(ctx, dw, dkv, hidden, draft)
    assert_close(taps["resid"][0], hidden, tol=0, what="layer-0 input")
    okv.reserve(N_PAST + k + 1)
    for l in range(cfg.n_layers):
        x_out, st = oracle.block(ocfg, ow, okv, l, taps["resid"][l], N_PAST)
        assert st == 0
        assert_close(taps["resid"][l + 1], x_out, what=f"layer {l} output")


def test_step_long_context_plan_matches_oracle(model):
    """The same step under a long-context work plan (max_ctx 8192: chunks of
    512 keys in sub-chunks of 128, more than the K/V ring holds, so the
    attention reads the KV metadata after its dependency wait) matches the
    oracle as the short plan (sub-chunks of 64) does."""
    _, ow, dw = model
    cfg, ocfg = SMALL, ocfg_of(SMALL)
    k = 15
    hidden = synth.normal((k + 1, cfg.hidden), 3, 510)
    okv0 = fresh_kv(model[0])[1]
    oidx, olog, _, st = oracle.forward(ocfg, ow, okv0.copy(), hidden, logits=True)
    assert st == 0
    _, gap = oracle.argmax(olog)
    require_clear_rows(gap, "long-plan rows")
    ctx_long = runtime.Context(SMALL, max_ctx=8192)
    try:
        for L_t in (3, 15):
            dkv, okv = fresh_kv(ctx_long)
            draft = synth.plant_draft(oidx, L_t, cfg.vocab, 3, 800 + L_t)
            ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
            res, taps = gpu_step(ctx_long, dw, dkv, hidden, draft)
            assert_close(taps["logits"], olog2, what="logits (long plan)")
            assert np.array_equal(taps["argmax"], oidx2)
            assert list(res) == list(ores), (list(res), list(ores))
            s = dkv.state()
            oc = okv.committed()
            assert s[0] == oc[0] and np.array_equal(s[1], oc[1])
    finally:
        ctx_long.close()


@pytest.mark.parametrize("n_past", [0, 120, 250])
def test_step_block_positions_match_oracle(model, n_past):
    """The block at other depths of the short plan (64-key chunks): at the
    start of the cache (no earlier rows to copy before the dependency wait),
    straddling the chunk boundary at 128, and deep in the cache."""
    ctx, ow, dw = model
    cfg, ocfg = SMALL, ocfg_of(SMALL)
    k = 15
    hidden = synth.normal((k + 1, cfg.hidden), 3, 520 + n_past)
    okv0 = fresh_kv(ctx, n_past)[1]
    oidx, olog, _, st = oracle.forward(ocfg, ow, okv0.copy(), hidden, logits=True)
    assert st == 0
    _, gap = oracle.argmax(olog)
    require_clear_rows(gap, f"rows at n_past {n_past}")
    dkv, okv = fresh_kv(ctx, n_past)
    draft = synth.plant_draft(oidx, 9, cfg.vocab, 3, 830 + n_past)
    ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
    res, taps = gpu_step(ctx, dw, dkv, hidden, draft)
    assert_close(taps["logits"], olog2, what=f"logits at n_past {n_past}")
    assert np.array_equal(taps["argmax"], oidx2)
    assert list(res) == list(ores), (list(res), list(ores))
    s = dkv.state()
    oc = okv.committed()
    assert s[0] == oc[0] and np.array_equal(s[1], oc[1])


def test_step_batch_height_invariance(model):
    """Rows 0..3 of a k=15 step and of a k=3 step over the same first rows give
    bit-identical logits ("The Two-Fifteen That Wasn't": exact speculation needs
    batch-height-invariant kernels)."""
    ctx, ow, dw = model
    hidden = synth.normal((16, SMALL.hidden), 3, 800)
    d15 = synth.tokens(15, SMALL.vocab, 3, 801)
    dkv, _ = fresh_kv(ctx)
    _, t15 = gpu_step(ctx, dw, dkv, hidden, d15)
    dkv, _ = fresh_kv(ctx)
    _, t3 = gpu_step(ctx, dw, dkv, hidden[:4], d15[:3])
    assert np.array_equal(t3["logits"].view(np.uint32), t15["logits"][:4].view(np.uint32))
    assert np.array_equal(t3["argmax"], t15["argmax"][:4])
    assert np.array_equal(t3["resid"].view(np.uint32), t15["resid"][:, :4].view(np.uint32))


def test_step_device_errors_leave_kv_committed_state(model):
    ctx, ow, dw = model
    hidden = synth.normal((8, SMALL.hidden), 3, 900)
    draft = synth.tokens(7, SMALL.vocab, 3, 901)
    # token out of range: rejected before any work
    dkv, _ = fresh_kv(ctx)
    before = dkv.state()
    bad = draft.copy()
    bad[3] = SMALL.vocab + 5
    res, _ = gpu_step(ctx, dw, dkv, hidden, bad, taps=False)
    assert res[2] == abi.ST_TOKEN_RANGE and res[1] == -1 and res[3] == N_PAST
    after = dkv.state()
    assert after[0] == before[0] and all(np.array_equal(a, b) for a, b in zip(after[1:], before[1:]))
    # non-finite hidden: computed, then rolled back entirely
    h_nan = hidden.copy()
    h_nan[5, 17] = np.inf
    res, _ = gpu_step(ctx, dw, dkv, h_nan, draft, taps=False)
    assert res[2] & abi.ST_NONFINITE and res[3] == N_PAST
    after = dkv.state()
    assert after[0] == before[0] and all(np.array_equal(a, b) for a, b in zip(after[1:], before[1:]))
    # page pool exhausted
    small = runtime.DeviceKV(SMALL, 5, PAGES)
    small.reset(ctx)
    small.extend(ctx, 80)             # 5 pages used, 0 free; the block needs a 6th
    res, _ = gpu_step(ctx, dw, small, hidden, draft, taps=False)
    assert res[2] == abi.ST_POOL_EMPTY and res[3] == 80
    assert small.state()[0] == 80
    # invalid verify length: host error, nothing enqueued
    h_d = torch.from_numpy(hidden[:6]).cuda()
    d_d = torch.from_numpy(draft[:5]).cuda()
    r = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert abi.spec_verify_step(ctx.h, dw.struct(), dkv.struct(), h_d.data_ptr(), d_d.data_ptr(), 5,
                                r.data_ptr()) == abi.SPEC_EVERIFYLEN


def test_step_host_buffers_and_consecutive_rounds(model):
    """Three consecutive rounds through the host-buffer entry point; the oracle
    runs the same rounds; results and KV state agree each round."""
    ctx, ow, dw = model
    cfg, ocfg = SMALL, ocfg_of(SMALL)
    dkv, okv = fresh_kv(ctx)
    for rnd in range(3):
        hidden = synth.normal((8, cfg.hidden), 4, 1000 + rnd)
        oidx, olog, _, _ = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
        _, gap = oracle.argmax(olog)
        require_clear_rows(gap, f"round {rnd} rows")
        draft = synth.plant_draft(oidx, [2, 7, 0][rnd], cfg.vocab, 4, 1100 + rnd)
        ores, _, _, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        res = abi.spec_result()
        hp = torch.from_numpy(hidden).pin_memory()
        dp = torch.from_numpy(draft).pin_memory()
        abi.check("spec_verify_step_host", abi.spec_verify_step_host(ctx.h, dw.struct(), dkv.struct(),
                                                                     hp.data_ptr(), dp.data_ptr(), 7, res))
        assert [res.accepted_len, res.next_token, res.status, res.seq_len] == list(ores)
        s, oc = dkv.state(), okv.committed()
        assert s[0] == oc[0] and np.array_equal(s[1], oc[1]) and np.array_equal(s[3], oc[3])


def test_step_with_attention_narrower_than_hidden():
    """A block whose attention width differs from the hidden width (24 query
    heads of 128 over 4 KV heads at H = 3328, group 6), the geometry of the
    draft's k/v 6,656 -> 1,024 projections: the step against the oracle."""
    import __graft_entry__
    __graft_entry__.build()
    cfg = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=24, n_kv_heads=4, head_dim=128, ffn=8960,
                              vocab=4096)
    ocfg = ocfg_of(cfg)
    ctx = runtime.Context(cfg, max_ctx=PAGES * 16)
    try:
        ow, dw = build_model(ctx, cfg, seed=8)
        dkv = runtime.DeviceKV(cfg, PAGES, PAGES)
        dkv.reset(ctx)
        dkv.extend(ctx, N_PAST)
        okv = oracle.KV(ocfg, PAGES, PAGES)
        okv.extend(N_PAST)
        fill_context(cfg, dkv, okv, N_PAST, seed=12)
        k = 15
        hidden = synth.normal((k + 1, cfg.hidden), 8, 40)
        oidx, olog, _, st = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
        assert st == 0
        _, gap = oracle.argmax(olog)
        require_clear_rows(gap, "narrow-attention rows")
        draft = synth.plant_draft(oidx, 8, cfg.vocab, 8, 41)
        ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        h_d = torch.from_numpy(hidden).cuda()
        d_d = torch.from_numpy(draft).cuda()
        res = torch.zeros(4, dtype=torch.int32, device="cuda")
        am = torch.zeros(k + 1, dtype=torch.int32, device="cuda")
        lg = torch.zeros((k + 1, cfg.vocab), dtype=torch.float32, device="cuda")
        abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(), h_d.data_ptr(),
                                                                 d_d.data_ptr(), k, res.data_ptr(),
                                                                 abi.spec_taps(None, am.data_ptr(), lg.data_ptr())))
        torch.cuda.synchronize()
        assert_close(lg.cpu().numpy(), olog2, what="logits")
        assert np.array_equal(am.cpu().numpy(), oidx2)
        assert list(res.cpu().numpy()) == list(ores)
        s, oc = dkv.state(), okv.committed()
        assert s[0] == oc[0] and np.array_equal(s[1], oc[1])
    finally:
        ctx.close()


@pytest.mark.parametrize("n_past", [N_PAST, 329])
def test_step_with_qk_norm_and_rope(n_past):
    """The draft's attention variant (Ch. 8 §8.2 lists QK-norms and RoPE):
    every q and k head RMS-normed with its own gains, then rotated at its
    row's position (theta 1e6), 24 query heads over 4 KV heads.  The step
    against the oracle, at two context lengths; the same inputs without the
    transforms give other logits (the transforms are live)."""
    import __graft_entry__
    __graft_entry__.build()
    cfg = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=24, n_kv_heads=4, head_dim=128, ffn=8960,
                              vocab=4096, rope_theta=1.0e6)
    ocfg = ocfg_of(cfg)
    ctx = runtime.Context(cfg, max_ctx=PAGES * 16)
    try:
        ow, dw = build_model(ctx, cfg, seed=9)
        add_qk_norm(cfg, ow, dw, seed=9)
        dkv = runtime.DeviceKV(cfg, PAGES, PAGES)
        dkv.reset(ctx)
        dkv.extend(ctx, n_past)
        okv = oracle.KV(ocfg, PAGES, PAGES)
        okv.extend(n_past)
        fill_context(cfg, dkv, okv, n_past, seed=13)
        k = 15
        hidden = synth.normal((k + 1, cfg.hidden), 9, 40 + n_past)
        oidx, olog, _, st = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
        assert st == 0
        _, gap = oracle.argmax(olog)
        require_clear_rows(gap, "qk-norm/rope rows")
        plain = dataclasses.replace(ocfg, rope_theta=0.0)
        _, olog_plain, _, _ = oracle.forward(plain, ow, okv.copy(), hidden, logits=True)
        assert np.max(np.abs(olog_plain - olog)) > 1e-2
        draft = synth.plant_draft(oidx, 6, cfg.vocab, 9, 41)
        ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        h_d = torch.from_numpy(hidden).cuda()
        d_d = torch.from_numpy(draft).cuda()
        res = torch.zeros(4, dtype=torch.int32, device="cuda")
        am = torch.zeros(k + 1, dtype=torch.int32, device="cuda")
        lg = torch.zeros((k + 1, cfg.vocab), dtype=torch.float32, device="cuda")
        abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(), h_d.data_ptr(),
                                                                 d_d.data_ptr(), k, res.data_ptr(),
                                                                 abi.spec_taps(None, am.data_ptr(), lg.data_ptr())))
        torch.cuda.synchronize()
        assert_close(lg.cpu().numpy(), olog2, what="logits")
        assert np.array_equal(am.cpu().numpy(), oidx2)
        assert list(res.cpu().numpy()) == list(ores)
        s_, oc = dkv.state(), okv.committed()
        assert s_[0] == oc[0] and np.array_equal(s_[1], oc[1])
        # a token tree is refused under a rotary configuration
        tok = torch.zeros(4, dtype=torch.int32, device="cuda")
        par = torch.tensor([-1, 0, 0, 1], dtype=torch.int32, device="cuda")
        path = torch.zeros(64, dtype=torch.int32, device="cuda")
        rc = abi.spec_verify_tree(ctx.h, dw.struct(), dkv.struct(), h_d.data_ptr(), tok.data_ptr(), par.data_ptr(),
                                  4, res.data_ptr(), path.data_ptr(), None)
        assert rc == abi.SPEC_EINVAL
    finally:
        ctx.close()
