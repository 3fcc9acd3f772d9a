"""Token-tree verification (Ch. 33 §33.7) on the GPU against the oracle,
through spec_verify_tree.

Bit-exact: a chain tree equals the linear verify step (result, argmax, logits,
KV metadata and rows); the tree step's result, accepted path and committed KV
metadata equal the oracle's (every node's top-2 gap must be clear, > 1e-2:
the tests count the nodes below it and require none);
the path's K/V rows after the moves equal the oracle's to one bf16 ulp.
Tolerance: logits.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import assert_close, require_clear_rows  # noqa: E402
from tests.model_util import build_model, fill_context, ocfg_of  # noqa: E402

SMALL = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=26, n_kv_heads=2, head_dim=128,
                            ffn=8960, vocab=4096)
N_PAST = 71
PAGES = 24


@pytest.fixture(scope="module")
def model():
    import __graft_entry__
    __graft_entry__.build()
    ctx = runtime.Context(SMALL, max_ctx=PAGES * 16)
    ow, dw = build_model(ctx, SMALL, seed=3)
    yield ctx, ow, dw
    ctx.close()


def fresh_kv(ctx):
    cfg = SMALL
    dkv = runtime.DeviceKV(cfg, PAGES, PAGES)
    dkv.reset(ctx)
    dkv.extend(ctx, N_PAST)
    okv = oracle.KV(ocfg_of(cfg), PAGES, PAGES)
    okv.extend(N_PAST)
    fill_context(cfg, dkv, okv, N_PAST, seed=11)
    return dkv, okv


def gpu_tree(ctx, dw, dkv, rows, tokens, parent):
    n = len(parent)
    h = torch.from_numpy(np.ascontiguousarray(rows, dtype=np.float32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).cuda()
    p = torch.from_numpy(np.ascontiguousarray(parent, dtype=np.int32)).cuda()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    path = torch.zeros(max(16, n), dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    lg = torch.zeros((n, SMALL.vocab), dtype=torch.float32, device="cuda")
    taps = abi.spec_taps(None, am.data_ptr(), lg.data_ptr())
    abi.check("spec_verify_tree", abi.spec_verify_tree(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(), t.data_ptr(),
                                                       p.data_ptr(), n, res.data_ptr(), path.data_ptr(), taps))
    torch.cuda.synchronize()
    return res.cpu().numpy(), path.cpu().numpy(), am.cpu().numpy(), lg.cpu().numpy()


def kv_rows_equal(dkv, okv, upto, ulp=1):
    s = dkv.state()
    oc = okv.committed()
    assert s[0] == oc[0] == upto and np.array_equal(s[1], oc[1]) and np.array_equal(s[3], oc[3])
    pool = dkv.pool.view(torch.int16).cpu().numpy().view(np.uint16)
    for pos in range(N_PAST, upto):
        a = pool[s[1][pos // 16], :, :, :, pos % 16].astype(np.int32)
        b = okv.pool[oc[1][pos // 16], :, :, :, pos % 16].astype(np.int32)
        assert np.max(np.abs(a - b)) <= ulp, f"K/V row {pos} differs by more than {ulp} bf16 ulp"


def test_chain_tree_equals_linear_step(model):
    ctx, ow, dw = model
    cfg, k = SMALL, 15
    hidden = synth.normal((k + 1, cfg.hidden), 3, 500)
    draft = synth.tokens(k, cfg.vocab, 3, 600)
    # linear step
    dkv_l, _ = fresh_kv(ctx)
    res_l = torch.zeros(4, dtype=torch.int32, device="cuda")
    am_l = torch.zeros(k + 1, dtype=torch.int32, device="cuda")
    lg_l = torch.zeros((k + 1, cfg.vocab), dtype=torch.float32, device="cuda")
    h_d = torch.from_numpy(hidden).cuda()         # kept alive until the step has run
    d_d = torch.from_numpy(draft).cuda()
    abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(
        ctx.h, dw.struct(), dkv_l.struct(), h_d.data_ptr(), d_d.data_ptr(), k, res_l.data_ptr(),
        abi.spec_taps(None, am_l.data_ptr(), lg_l.data_ptr())))
    torch.cuda.synchronize()
    # the same rows as a chain tree
    dkv_t, _ = fresh_kv(ctx)
    parent = np.arange(-1, k, dtype=np.int32)
    tokens = np.concatenate([[0], draft]).astype(np.int32)
    res_t, path, am_t, lg_t = gpu_tree(ctx, dw, dkv_t, hidden, tokens, parent)
    assert np.array_equal(res_t, res_l.cpu().numpy())
    assert np.array_equal(path[: res_t[0] + 1], np.arange(res_t[0] + 1)) and np.all(path[res_t[0] + 1:] == -1)
    assert np.array_equal(am_t, am_l.cpu().numpy())
    assert np.array_equal(lg_t.view(np.uint32), lg_l.cpu().numpy().view(np.uint32))
    a, b = dkv_t.state(), dkv_l.state()
    assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[3], b[3])
    assert torch.equal(dkv_t.pool, dkv_l.pool)


def planted_tree(cfg, ow, okv0, seed, n_max):
    # a true branch that follows the oracle's own greedy decode, decoys off it
    rng = np.random.default_rng(seed)
    depth_max = int(rng.integers(2, 8))
    hidden = synth.normal((depth_max + 1, cfg.hidden), 5, 700 + seed)
    serial, _ = oracle.serial_greedy(ocfg_of(cfg), ow, okv0.copy(), hidden, depth_max)
    L_t = int(rng.integers(0, depth_max + 1))
    rows, tokens, parent, true_node = [hidden[0]], [0], [-1], [0]
    for depth in range(depth_max):
        for _ in range(int(rng.integers(0, 3))):
            if len(rows) >= n_max - 1:
                break
            rows.append(synth.normal((cfg.hidden,), 5, 2000 + 31 * seed + len(rows)))
            tokens.append((serial[depth] + 1 + int(rng.integers(0, cfg.vocab - 1))) % cfg.vocab)
            parent.append(int(rng.choice(true_node)))
        if len(rows) >= n_max:
            break
        rows.append(hidden[depth + 1])
        tokens.append(serial[depth] if depth < L_t else (serial[depth] + 5) % cfg.vocab)
        parent.append(true_node[-1])
        true_node.append(len(rows) - 1)
    return (np.stack(rows).astype(np.float32), np.array(tokens, dtype=np.int32),
            np.array(parent, dtype=np.int32))


def test_tree_step_long_plan_matches_oracle(model):
    """A tree step under a long-context work plan (max_ctx 8192: the
    attention's tree instance with 128-key sub-chunks, 64 score columns per
    row thread and 64-bit visibility masks) against the oracle."""
    _, ow, dw = model
    cfg = SMALL
    ctx_long = runtime.Context(SMALL, max_ctx=8192)
    try:
        for seed in (7, 8):
            dkv, okv = fresh_kv(ctx_long)
            rows, tokens, parent = planted_tree(cfg, ow, okv, seed, 16)
            ores, opath, oidx, olg = oracle.verify_tree(ocfg_of(cfg), ow, okv, rows, tokens, parent)
            assert ores[2] == 0
            res, path, am, lg = gpu_tree(ctx_long, dw, dkv, rows, tokens, parent)
            assert_close(lg, olg, what="logits (long plan)")
            _, gap = oracle.argmax(olg)
            require_clear_rows(gap, f"long-plan tree {seed} nodes")
            assert np.array_equal(am, oidx)
            assert list(res) == list(ores)
            assert np.array_equal(path[: res[0] + 1], opath)
            kv_rows_equal(dkv, okv, int(ores[3]))
    finally:
        ctx_long.close()


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5, 6])
def test_tree_step_matches_oracle(model, seed):
    ctx, ow, dw = model
    cfg = SMALL
    dkv, okv = fresh_kv(ctx)
    rows, tokens, parent = planted_tree(cfg, ow, okv, seed, 16)
    ores, opath, oidx, olg = oracle.verify_tree(ocfg_of(cfg), ow, okv, rows, tokens, parent)
    assert ores[2] == 0
    res, path, am, lg = gpu_tree(ctx, dw, dkv, rows, tokens, parent)
    assert res[2] == 0
    assert_close(lg, olg, what="logits")
    _, gap = oracle.argmax(olg)
    require_clear_rows(gap, f"tree {seed} nodes")
    assert np.array_equal(am, oidx)
    assert list(res) == list(ores)
    assert np.array_equal(path[: res[0] + 1], opath) and np.all(path[res[0] + 1:] == -1)
    kv_rows_equal(dkv, okv, int(ores[3]))


def test_tree_graph_replay_and_bad_tree(model):
    ctx, ow, dw = model
    cfg = SMALL
    dkv0, okv0 = fresh_kv(ctx)
    rows, tokens, parent = planted_tree(cfg, ow, okv0, 9, 12)
    out = []
    for _ in range(2):                                 # direct (taps) then recorded graph (no taps)
        dkv, _ = fresh_kv(ctx)
        out.append(gpu_tree(ctx, dw, dkv, rows, tokens, parent)[:2])
    dkv, _ = fresh_kv(ctx)
    n = len(parent)
    h = torch.from_numpy(rows).cuda()
    t = torch.from_numpy(tokens).cuda()
    p = torch.from_numpy(parent).cuda()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    path = torch.zeros(16, dtype=torch.int32, device="cuda")
    for _ in range(2):
        dkv, _ = fresh_kv(ctx)
        abi.check("spec_verify_tree", abi.spec_verify_tree(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(),
                                                           t.data_ptr(), p.data_ptr(), n, res.data_ptr(),
                                                           path.data_ptr(), None))
        torch.cuda.synchronize()
        assert np.array_equal(res.cpu().numpy(), out[0][0]) and np.array_equal(path.cpu().numpy(), out[0][1])
    # a parent list that is not a tree: nothing reserved, KV as before
    dkv, _ = fresh_kv(ctx)
    before = dkv.state()
    bad = parent.copy()
    bad[3] = 3
    p_bad = torch.from_numpy(bad).cuda()
    abi.check("spec_verify_tree", abi.spec_verify_tree(ctx.h, dw.struct(), dkv.struct(), h.data_ptr(),
                                                       t.data_ptr(), p_bad.data_ptr(), n, res.data_ptr(),
                                                       path.data_ptr(), None))
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    assert r[2] & abi.ST_BAD_TREE and r[1] == -1 and r[3] == N_PAST
    after = dkv.state()
    assert after[0] == before[0] and all(np.array_equal(x, y) for x, y in zip(after[1:], before[1:]))
    assert np.all(path.cpu().numpy() == -1)


def planted_big_tree(cfg, ow, okv0, seed, depth_max, decoys):
    """A true branch of depth depth_max following the oracle's greedy decode,
    with decoys (wrong tokens, other rows) hanging off random true nodes."""
    rng = np.random.default_rng(seed)
    hidden = synth.normal((depth_max + 1, cfg.hidden), 7, 900 + seed)
    serial, _ = oracle.serial_greedy(ocfg_of(cfg), ow, okv0.copy(), hidden, depth_max)
    L_t = int(rng.integers(depth_max // 2, depth_max + 1))
    rows, tokens, parent, true_node = [hidden[0]], [0], [-1], [0]
    for depth in range(depth_max):
        for _ in range(int(rng.integers(decoys[0], decoys[1] + 1))):
            rows.append(synth.normal((cfg.hidden,), 7, 5000 + 97 * seed + len(rows)))
            tokens.append((serial[depth] + 1 + int(rng.integers(0, cfg.vocab - 1))) % cfg.vocab)
            parent.append(int(rng.choice(true_node)))
        rows.append(hidden[depth + 1])
        tokens.append(serial[depth] if depth < L_t else (serial[depth] + 5) % cfg.vocab)
        parent.append(true_node[-1])
        true_node.append(len(rows) - 1)
    return (np.stack(rows).astype(np.float32), np.array(tokens, dtype=np.int32),
            np.array(parent, dtype=np.int32), L_t)


@pytest.mark.parametrize("seed,depth_max,decoys", [(1, 7, (2, 3)), (2, 10, (2, 4)), (3, 12, (3, 4))])
def test_large_tree_step_matches_oracle(model, seed, depth_max, decoys):
    """Trees of 24 to 64 nodes (Ch. 33 §33.7), verified in passes of 16 rows."""
    ctx, ow, dw = model
    cfg = SMALL
    dkv, okv = fresh_kv(ctx)
    rows, tokens, parent, L_t = planted_big_tree(cfg, ow, okv, seed, depth_max, decoys)
    n = len(parent)
    assert 17 <= n <= 64, n
    ores, opath, oidx, olg = oracle.verify_tree(ocfg_of(cfg), ow, okv, rows, tokens, parent)
    assert ores[2] == 0 and ores[0] == L_t
    res, path, am, lg = gpu_tree(ctx, dw, dkv, rows, tokens, parent)
    assert res[2] == 0
    assert_close(lg, olg, what=f"logits of {n} nodes")
    _, gap = oracle.argmax(olg)
    require_clear_rows(gap, f"large tree {seed} ({n} nodes)")
    assert np.array_equal(am, oidx)
    assert list(res) == list(ores)
    assert np.array_equal(path[: res[0] + 1], opath) and np.all(path[res[0] + 1:] == -1)
    kv_rows_equal(dkv, okv, int(ores[3]))


def test_large_chain_tree_and_64_nodes(model):
    """A chain of 40 nodes accepts down to its first wrong token; a 64-node
    tree (the largest) matches the oracle and its graph replay."""
    ctx, ow, dw = model
    cfg = SMALL
    dkv, okv = fresh_kv(ctx)
    rows, tokens, parent, _ = planted_big_tree(cfg, ow, okv, 9, 16, (3, 3))
    rows, tokens, parent = rows[:64], tokens[:64], parent[:64]
    assert len(parent) == 64
    ores, opath, oidx, olg = oracle.verify_tree(ocfg_of(cfg), ow, okv, rows, tokens, parent)
    _, gap = oracle.argmax(olg)
    require_clear_rows(gap, "64-node tree")
    res, path, am, _ = gpu_tree(ctx, dw, dkv, rows, tokens, parent)
    assert list(res) == list(ores) and np.array_equal(am, oidx)
    assert np.array_equal(path[: res[0] + 1], opath)
    kv_rows_equal(dkv, okv, int(ores[3]))
    # the same tree through the recorded graph (no taps), twice
    h = torch.from_numpy(rows).cuda()
    t = torch.from_numpy(tokens).cuda()
    p = torch.from_numpy(parent).cuda()
    r = torch.zeros(4, dtype=torch.int32, device="cuda")
    pth = torch.zeros(64, dtype=torch.int32, device="cuda")
    for _ in range(2):
        dkv2, _ = fresh_kv(ctx)
        abi.check("spec_verify_tree", abi.spec_verify_tree(ctx.h, dw.struct(), dkv2.struct(), h.data_ptr(),
                                                           t.data_ptr(), p.data_ptr(), 64, r.data_ptr(),
                                                           pth.data_ptr(), None))
        torch.cuda.synchronize()
        assert list(r.cpu().numpy()) == list(ores)
        assert np.array_equal(pth.cpu().numpy()[: res[0] + 1], opath)
    # 65 nodes: refused before any work
    assert abi.spec_verify_tree(ctx.h, dw.struct(), dkv2.struct(), h.data_ptr(), t.data_ptr(), p.data_ptr(), 65,
                                r.data_ptr(), pth.data_ptr(), None) == abi.SPEC_EVERIFYLEN
