"""Sliding-window layers and their rings (Ch. 8 §8.6 item 4: the target's KV
checkpoint rewinds the paged planes' metadata only, while the sliding-window
rings keep the at most 16 rows a block may overwrite; here the ring has 16
spare slots, so those rows are never overwritten).

A 2-layer model whose layer 1 is a sliding-window layer, with the block well
past W (the ring has wrapped): W = 64 (a multiple of 16), W = 40 (rounded up
in the ring) and W = 2048 at a context of 2,400 (several attention chunks).
Against the oracle (plain definition: a windowed causal mask over the full
history):
  * tolerance: logits and the per-layer residual stream (teacher-forced);
  * bit-exact: argmax, accepted length, next token, status, KV metadata;
  * the ring after the step holds, for the last W positions, the oracle's
    rows (context rows bit-exact, the block's own rows within one bf16 ulp);
  * the step leaves the ring rows of the W positions before the block
    untouched (bit-exact), so a rollback to the block's start needs no copy;
    a rollback below it is refused;
  * two consecutive rounds agree with the oracle run over the same rounds.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import assert_close, require_clear_rows  # noqa: E402
from tests.model_util import add_qk_norm, build_model, fill_context, ocfg_of  # noqa: E402

W = 64
CFG = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=26, n_kv_heads=2, head_dim=128, ffn=8960,
                          vocab=4096, swa_window=W, swa_period=2)
N_PAST = 150
PAGES = 24


@pytest.fixture(scope="module")
def model():
    import __graft_entry__
    __graft_entry__.build()
    ctx = runtime.Context(CFG, max_ctx=PAGES * 16)
    ow, dw = build_model(ctx, CFG, seed=5)
    yield ctx, ow, dw
    ctx.close()


def fresh_kv(ctx, n_past=N_PAST, cfg=CFG, pages=PAGES):
    dkv = runtime.DeviceKV(cfg, pages, pages)
    dkv.reset(ctx)
    dkv.extend(ctx, n_past)
    okv = oracle.KV(ocfg_of(cfg), pages, pages)
    okv.extend(n_past)
    fill_context(cfg, dkv, okv, n_past, seed=13)
    torch.cuda.synchronize()
    return dkv, okv


def step(ctx, dw, dkv, hidden, draft, cfg=CFG):
    k, M = len(draft), len(draft) + 1
    h = torch.from_numpy(np.ascontiguousarray(hidden)).cuda()
    d = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).cuda()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    resid = torch.zeros((cfg.n_layers + 1, M, cfg.hidden), dtype=torch.float32, device="cuda")
    am = torch.zeros(M, dtype=torch.int32, device="cuda")
    lg = torch.zeros((M, cfg.vocab), dtype=torch.float32, device="cuda")
    taps = abi.spec_taps(resid.data_ptr(), am.data_ptr(), lg.data_ptr())
    abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(),
                                                             d.data_ptr(), k, res.data_ptr(), taps))
    torch.cuda.synchronize()
    return res.cpu().numpy(), resid.cpu().numpy(), am.cpu().numpy(), lg.cpu().numpy()


def ring_vs_oracle(dkv, okv, upto, block_from, what, w=W):
    """Ring slots of positions [upto - W, upto) against the oracle's rows: the
    context rows bit-exact, rows the GPU computed (>= block_from) within one ulp."""
    pos = np.arange(max(0, upto - w), upto)
    ring = dkv.ring_rows(1, pos).astype(np.int32)                   # [2][nkv][n][dh]
    ref = np.stack([okv.pool[okv.page_table[p // 16], 1, :, :, p % 16] for p in pos], axis=2).astype(np.int32)
    ctx_part = pos < block_from
    assert np.array_equal(ring[:, :, ctx_part], ref[:, :, ctx_part]), f"{what}: context rows differ"
    assert np.max(np.abs(ring - ref)) <= 1, f"{what}: block rows differ by more than one bf16 ulp"


def check_window_step(ctx, ow, dw, cfg, n_past, pages, seed):
    w = cfg.swa_window
    ocfg, k = ocfg_of(cfg), 15
    hidden = synth.normal((k + 1, cfg.hidden), seed, 300)
    dkv, okv = fresh_kv(ctx, n_past, cfg, pages)
    ring_before = dkv.ring_rows(1, np.arange(n_past - w, n_past)).copy()
    oidx, olog, _, st = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
    assert st == 0
    _, gap = oracle.argmax(olog)
    require_clear_rows(gap, f"sliding-window (W {w}) step rows")
    for L_t in (4, 15, 0):
        dkv, okv = fresh_kv(ctx, n_past, cfg, pages)
        draft = synth.plant_draft(oidx, L_t, cfg.vocab, seed, 310 + L_t)
        ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        res, resid, am, lg = step(ctx, dw, dkv, hidden, draft, cfg)
        assert_close(lg, olog2, what="logits")
        assert np.array_equal(am, oidx2)
        assert list(res) == list(ores), (list(res), list(ores))
        s, oc = dkv.state(), okv.committed()
        assert s[0] == oc[0] and np.array_equal(s[1], oc[1]) and np.array_equal(s[3], oc[3])
        ring_vs_oracle(dkv, okv, int(res[3]), n_past, f"ring after accepting {L_t}", w)
        # the block wrote only spare slots: the W rows before it are untouched
        after = dkv.ring_rows(1, np.arange(n_past - w, n_past))
        assert np.array_equal(after, ring_before), "the step overwrote a ring row of the window"
        # back to the block's start: metadata only
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, dkv.struct(), n_past))
        assert abi.spec_last_status(ctx.h) == 0
        assert dkv.state()[0] == n_past
        # below the block: refused, nothing changes
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, dkv.struct(), n_past - 1))
        assert abi.spec_last_status(ctx.h) & abi.ST_ROLLBACK
        assert dkv.state()[0] == n_past
    # teacher-forced per layer on the last step's taps (block at n_past)
    okv_t = fresh_kv(ctx, n_past, cfg, pages)[1]
    okv_t.reserve(n_past + k + 1)
    for l in range(cfg.n_layers):
        x_out, st = oracle.block(ocfg, ow, okv_t, l, resid[l], n_past)
        assert st == 0
        assert_close(resid[l + 1], x_out, what=f"layer {l} output (window {cfg.swa_index(l) >= 0})")


def test_swa_step_matches_oracle_and_ring_keeps_the_window(model):
    ctx, ow, dw = model
    check_window_step(ctx, ow, dw, CFG, N_PAST, PAGES, 5)


@pytest.mark.parametrize("w,n_past,pages", [(40, 150, 24), (2048, 2400, 152), (8192, 8400, 530)])
def test_swa_other_windows(w, n_past, pages):
    """A window that is not a multiple of 16 (the ring rounds it up), a
    2,048-position window at a context of 2,400 (the window spans several
    attention chunks and starts inside a page), and an 8,192-position window
    at 8,400 (the window's plan takes 128-key sub-chunks)."""
    cfg = runtime.ModelConfig(**{**CFG.__dict__, "swa_window": w})
    ctx = runtime.Context(cfg, max_ctx=pages * 16)
    try:
        ow, dw = build_model(ctx, cfg, seed=5)
        check_window_step(ctx, ow, dw, cfg, n_past, pages, 7)
    finally:
        ctx.close()


def test_swa_consecutive_rounds_match_oracle(model):
    ctx, ow, dw = model
    ocfg = ocfg_of(CFG)
    dkv, okv = fresh_kv(ctx)
    for rnd, L_t in enumerate((6, 15, 2)):
        hidden = synth.normal((16, CFG.hidden), 6, 400 + rnd)
        oidx, olog, _, _ = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
        _, gap = oracle.argmax(olog)
        require_clear_rows(gap, f"round {rnd} rows")
        draft = synth.plant_draft(oidx, L_t, CFG.vocab, 6, 500 + rnd)
        ores, _, _, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        res, _, am, lg = step(ctx, dw, dkv, hidden, draft)
        assert list(res) == list(ores), (rnd, list(res), list(ores))
        assert np.array_equal(am, oidx)
        ring_vs_oracle(dkv, okv, int(res[3]), N_PAST, f"round {rnd}")


def test_swa_model_refuses_token_trees(model):
    ctx, ow, dw = model
    dkv, _ = fresh_kv(ctx)
    h = torch.zeros((4, CFG.hidden), dtype=torch.float32, device="cuda")
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    p = torch.tensor([-1, 0, 0, 1], dtype=torch.int32, device="cuda")
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert abi.spec_verify_tree(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(), t.data_ptr(), p.data_ptr(), 4,
                                res.data_ptr(), None, None) == abi.SPEC_EINVAL


@pytest.mark.parametrize("n_past,M", [(10, 4), (60, 16), (150, 16), (300, 8)])
def test_window_attention_alone_matches_oracle(model, n_past, M):
    """spec_attention on the window layer (its ring, the window mask and the
    window's chunk plan) against the oracle's windowed attention: a block
    inside the first window, one at the window's edge, one past a wrapped
    ring, one far past it."""
    ctx, _, _ = model
    n = n_past + M
    dkv, okv = fresh_kv(ctx, n)
    # the block's first row looks back W - 1 positions past the last W: lay
    # down the last R positions (the whole ring) from the oracle's rows
    p0 = max(0, n - CFG.swa_ring_rows)
    pos = np.arange(p0, n)
    kb = np.stack([okv.pool[okv.page_table[p // 16], 1, 0, :, p % 16].reshape(-1) for p in pos])
    vb = np.stack([okv.pool[okv.page_table[p // 16], 1, 1, :, p % 16].reshape(-1) for p in pos])
    dkv.write_ring_rows(1, p0, kb, vb)
    torch.cuda.synchronize()
    q = synth.normal((M, CFG.n_q_heads, CFG.head_dim), 9, n_past) * 4.0
    qd = torch.from_numpy(np.ascontiguousarray(q.reshape(M, -1))).cuda()
    out = torch.zeros((M, CFG.n_q_heads * CFG.head_dim), dtype=torch.float32, device="cuda")
    abi.check("spec_attention", abi.spec_attention(ctx.h, dkv.struct(), 1, qd.data_ptr(), M, out.data_ptr()))
    torch.cuda.synchronize()
    ref = okv.attention(1, q.reshape(M, -1), n_past)
    assert_close(out.cpu().numpy(), ref, what=f"window attention at n_past {n_past}, M {M}")


def test_window_layers_with_qk_norm_and_rope():
    """Window layers together with QK-norm and RoPE (the transforms run before
    the K row enters the ring): one step against the oracle, and the ring
    rows of the block against the oracle's (within one bf16 ulp)."""
    cfg = runtime.ModelConfig(**{**CFG.__dict__, "rope_theta": 10000.0})
    ctx = runtime.Context(cfg, max_ctx=PAGES * 16)
    try:
        ow, dw = build_model(ctx, cfg, seed=6)
        add_qk_norm(cfg, ow, dw, seed=6)
        ocfg = ocfg_of(cfg)
        hidden = synth.normal((16, cfg.hidden), 6, 700)
        dkv, okv = fresh_kv(ctx, N_PAST, cfg, PAGES)
        oidx, olog, _, st = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
        assert st == 0
        _, gap = oracle.argmax(olog)
        require_clear_rows(gap, "window + rope rows")
        draft = synth.plant_draft(oidx, 9, cfg.vocab, 6, 701)
        ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        res, _, am, lg = step(ctx, dw, dkv, hidden, draft, cfg)
        assert_close(lg, olog2, what="logits (window + rope)")
        assert np.array_equal(am, oidx2)
        assert list(res) == list(ores)
        ring_vs_oracle(dkv, okv, int(res[3]), N_PAST, "ring (window + rope)")
    finally:
        ctx.close()
