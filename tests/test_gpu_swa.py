"""Sliding-window layers and their ring checkpoint (Ch. 8 §8.6 item 4: the
target's KV checkpoint rewinds the paged planes' metadata only, while the
sliding-window rings keep the at most 16 rows a block may overwrite).

A 2-layer model whose layer 1 is a sliding-window layer of W = 64 positions,
with the block well past W (the ring has wrapped).  Against the oracle (plain
definition: a windowed causal mask over the full history):
  * tolerance: logits and the per-layer residual stream (teacher-forced);
  * bit-exact: argmax, accepted length, next token, status, KV metadata;
  * the ring after the step holds, for the last W positions, the oracle's
    rows (context rows bit-exact, the block's own rows within one bf16 ulp);
  * a rollback to the block's start puts back every ring row the block
    overwrote (bit-exact against the context written before the step), and a
    rollback below it is refused;
  * two consecutive rounds agree with the oracle run over the same rounds.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import assert_close, require_clear_rows  # noqa: E402
from tests.model_util import build_model, fill_context, ocfg_of  # noqa: E402

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


def fresh_kv(ctx, n_past=N_PAST):
    dkv = runtime.DeviceKV(CFG, PAGES, PAGES)
    dkv.reset(ctx)
    dkv.extend(ctx, n_past)
    okv = oracle.KV(ocfg_of(CFG), PAGES, PAGES)
    okv.extend(n_past)
    fill_context(CFG, dkv, okv, n_past, seed=13)
    torch.cuda.synchronize()
    return dkv, okv


def step(ctx, dw, dkv, hidden, draft):
    k, M = len(draft), len(draft) + 1
    h = torch.from_numpy(np.ascontiguousarray(hidden)).cuda()
    d = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).cuda()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    resid = torch.zeros((CFG.n_layers + 1, M, CFG.hidden), dtype=torch.float32, device="cuda")
    am = torch.zeros(M, dtype=torch.int32, device="cuda")
    lg = torch.zeros((M, CFG.vocab), dtype=torch.float32, device="cuda")
    taps = abi.spec_taps(resid.data_ptr(), am.data_ptr(), lg.data_ptr())
    abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(),
                                                             d.data_ptr(), k, res.data_ptr(), taps))
    torch.cuda.synchronize()
    return res.cpu().numpy(), resid.cpu().numpy(), am.cpu().numpy(), lg.cpu().numpy()


def ring_vs_oracle(dkv, okv, upto, block_from, what):
    """Ring slots of positions [upto - W, upto) against the oracle's rows: the
    context rows bit-exact, rows the GPU computed (>= block_from) within one ulp."""
    pos = np.arange(max(0, upto - W), upto)
    ring = dkv.ring_rows(1, pos).astype(np.int32)                   # [2][nkv][n][dh]
    ref = np.stack([okv.pool[okv.page_table[p // 16], 1, :, :, p % 16] for p in pos], axis=2).astype(np.int32)
    ctx_part = pos < block_from
    assert np.array_equal(ring[:, :, ctx_part], ref[:, :, ctx_part]), f"{what}: context rows differ"
    assert np.max(np.abs(ring - ref)) <= 1, f"{what}: block rows differ by more than one bf16 ulp"


def test_swa_step_matches_oracle_and_ring_checkpoint_restores(model):
    ctx, ow, dw = model
    ocfg, k = ocfg_of(CFG), 15
    hidden = synth.normal((k + 1, CFG.hidden), 5, 300)
    dkv, okv = fresh_kv(ctx)
    ring_before = dkv.ring_rows(1, np.arange(N_PAST - W, N_PAST)).copy()
    oidx, olog, _, st = oracle.forward(ocfg, ow, okv.copy(), hidden, logits=True)
    assert st == 0
    _, gap = oracle.argmax(olog)
    require_clear_rows(gap, "sliding-window step rows")
    for L_t in (4, 15, 0):
        dkv, okv = fresh_kv(ctx)
        draft = synth.plant_draft(oidx, L_t, CFG.vocab, 5, 310 + L_t)
        ores, oidx2, olog2, _ = oracle.verify_step(ocfg, ow, okv, hidden, draft)
        res, resid, am, lg = step(ctx, dw, dkv, hidden, draft)
        assert_close(lg, olog2, what="logits")
        assert np.array_equal(am, oidx2)
        assert list(res) == list(ores), (list(res), list(ores))
        s, oc = dkv.state(), okv.committed()
        assert s[0] == oc[0] and np.array_equal(s[1], oc[1]) and np.array_equal(s[3], oc[3])
        ring_vs_oracle(dkv, okv, int(res[3]), N_PAST, f"ring after accepting {L_t}")
        # back to the block's start: the checkpoint puts every overwritten row back
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, dkv.struct(), N_PAST))
        assert abi.spec_last_status(ctx.h) == 0
        after = dkv.ring_rows(1, np.arange(N_PAST - W, N_PAST))
        assert np.array_equal(after, ring_before), "rollback did not restore the ring"
        # below the checkpoint: refused, nothing changes
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, dkv.struct(), N_PAST - 1))
        assert abi.spec_last_status(ctx.h) & abi.ST_ROLLBACK
        assert dkv.state()[0] == N_PAST
    # teacher-forced per layer on the last step's taps (block at N_PAST)
    okv_t = fresh_kv(ctx)[1]
    okv_t.reserve(N_PAST + k + 1)
    for l in range(CFG.n_layers):
        x_out, st = oracle.block(ocfg, ow, okv_t, l, resid[l], N_PAST)
        assert st == 0
        assert_close(resid[l + 1], x_out, what=f"layer {l} output (window {CFG.swa_index(l) >= 0})")


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
