"""GPU parity of the stochastic exact acceptance (Ch. 33 §33.2) against the
oracle, through the C ABI.

Bit-exact: the MT19937 state after every call (the device draws exactly the
oracle's uniforms, regenerations included).  Decisions (accepted length, drawn
token): equal to the oracle's on the same logits, q, drafts and stream
whenever no uniform lies within 1e-5 of the threshold it is compared with
(the two sides compute p with different exp implementations, and the
residual's total in different summation orders); every test counts the
trials it skips and bounds that count.  Distribution: the first emitted token
follows the target's p_0 (chi-square against p_0 in closed form).
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.model_util import build_model, fill_context, ocfg_of  # noqa: E402

SMALL = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=26, n_kv_heads=2, head_dim=128,
                            ffn=8960, vocab=4096)
FULL = runtime.ModelConfig(**synth.FULL)
MARGIN = 1e-5


@pytest.fixture(scope="module")
def small_ctx():
    import __graft_entry__
    __graft_entry__.build()
    c = runtime.Context(SMALL, max_ctx=24 * 16)
    yield c
    c.close()


@pytest.fixture(scope="module")
def full_ctx():
    import __graft_entry__
    __graft_entry__.build()
    c = runtime.Context(FULL, max_ctx=2112)
    yield c
    c.close()


def mt_device(seed, advance=0):
    st = oracle.mt_seed(seed)
    if advance:
        oracle.mt_next(st, advance)
    return st, torch.from_numpy(st.view(np.int32).copy()).cuda()


def gpu_sample(ctx, logits, q, draft, mt_d, kv=None):
    k = len(draft)
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    qd = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    dd = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).cuda()
    abi.check("spec_sample_accept", abi.spec_sample_accept(ctx.h, lg.data_ptr(), qd.data_ptr(), dd.data_ptr(),
                                                           k, mt_d.data_ptr(), kv, res.data_ptr()))
    torch.cuda.synchronize()
    return res.cpu().numpy()


def random_case(rng, k, V, scale):
    logits = (rng.normal(0, scale, (k + 1, V))).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.3, size=k).astype(np.float32)
    # drafts from q (inverse cdf), sometimes the target's argmax
    draft = np.array([int(min(np.searchsorted(np.cumsum(q[i].astype(np.float64)), rng.random(), side="right"),
                              V - 1)) for i in range(k)], dtype=np.int32)
    hot = rng.random(k) < 0.5
    draft[hot] = np.argmax(logits[:k][hot], axis=1)
    return logits, q, draft


def test_mt_seed_matches_oracle():
    for seed in (0, 5489, 2**32 - 1):
        st = np.zeros(abi.MT_WORDS, dtype=np.uint32)
        abi.check("spec_mt_seed", abi.spec_mt_seed(st.ctypes.data, seed))
        assert np.array_equal(st, oracle.mt_seed(seed))


@pytest.mark.parametrize("k", [3, 7, 15])
def test_sample_accept_matches_oracle(small_ctx, k):
    ctx, V = small_ctx, SMALL.vocab
    rng = np.random.default_rng(100 + k)
    skipped = 0
    trials = 48
    for t in range(trials):
        # start some streams just before a regeneration of the 624 words
        ost, dst = mt_device(7 * t + k, advance=(620 if t % 4 == 0 else 0))
        logits, q, draft = random_case(rng, k, V, scale=(1.0, 3.0, 8.0)[t % 3])
        res = gpu_sample(ctx, logits, q, draft, dst)
        L, nxt, rc, margin = oracle.sample_accept(logits, q, draft, ost)
        assert rc == 0 and res[2] == 0
        assert np.array_equal(dst.cpu().numpy().view(np.uint32), ost), "MT state differs"
        if margin <= MARGIN:
            skipped += 1
            continue
        assert (res[0], res[1]) == (L, nxt), (t, res, L, nxt, margin)
    print(f"k={k}: {skipped} of {trials} trials skipped (a uniform within {MARGIN} of its threshold)")
    assert skipped <= 2, f"{skipped} of {trials} trials had a uniform within {MARGIN} of its threshold"


def test_sample_accept_full_vocab(full_ctx):
    ctx, V, k = full_ctx, FULL.vocab, 15
    rng = np.random.default_rng(5)
    skipped, trials = 0, 8
    for t in range(trials):
        ost, dst = mt_device(900 + t)
        logits, q, draft = random_case(rng, k, V, scale=4.0)
        res = gpu_sample(ctx, logits, q, draft, dst)
        L, nxt, rc, margin = oracle.sample_accept(logits, q, draft, ost)
        assert rc == 0 and res[2] == 0
        assert np.array_equal(dst.cpu().numpy().view(np.uint32), ost)
        if margin <= MARGIN:
            skipped += 1
            continue
        assert (res[0], res[1]) == (L, nxt), (t, res, L, nxt)
    print(f"full vocabulary: {skipped} of {trials} trials skipped (a uniform within {MARGIN} of its threshold)")
    assert skipped <= 1


def test_sample_accept_one_hot_is_greedy(small_ctx):
    ctx, V, k = small_ctx, SMALL.vocab, 7
    rng = np.random.default_rng(9)
    for t in range(10):
        idx = rng.integers(0, V, k + 1).astype(np.int32)
        L_t = int(rng.integers(0, k + 1))
        draft = idx[:k].copy()
        if L_t < k:
            draft[L_t] = (idx[L_t] + 3) % V
        logits = np.full((k + 1, V), -1.0e4, dtype=np.float32)
        logits[np.arange(k + 1), idx] = 0.0
        q = np.zeros((k, V), dtype=np.float32)
        q[np.arange(k), draft] = 1.0
        ost, dst = mt_device(40 + t)
        res = gpu_sample(ctx, logits, q, draft, dst)
        _, _, _, margin = oracle.sample_accept(logits, q, draft, ost)
        # margin 0: a uniform of exactly 0 accepts a draft of p = 0 (u <= a)
        assert margin > 0, "a uniform of exactly 0 in this stream; pick another seed"
        assert (res[0], res[1]) == (L_t, idx[L_t])


def test_sample_accept_device_errors_draw_nothing(small_ctx):
    ctx, V, k = small_ctx, SMALL.vocab, 3
    logits = np.zeros((k + 1, V), dtype=np.float32)
    q = np.full((k, V), 1.0 / V, dtype=np.float32)
    ost, dst = mt_device(1)
    res = gpu_sample(ctx, logits, q, np.array([0, V, 1], dtype=np.int32), dst)
    assert res[2] & abi.ST_TOKEN_RANGE and res[1] == -1
    assert np.array_equal(dst.cpu().numpy().view(np.uint32), ost)
    logits[2, 5] = np.nan
    res = gpu_sample(ctx, logits, q, np.array([0, 2, 1], dtype=np.int32), dst)
    assert res[2] & abi.ST_NONFINITE
    assert np.array_equal(dst.cpu().numpy().view(np.uint32), ost)


def test_sample_accept_first_token_follows_target(small_ctx):
    # 16 live tokens (the others have p = 0 exactly) with logits ln(w): p_0 =
    # w / sum(w) in closed form; draft x0 ~ q0 per trial
    ctx, V = small_ctx, SMALL.vocab
    rng = np.random.default_rng(21)
    live = np.sort(rng.choice(V, 16, replace=False))
    w = np.arange(1, 17, dtype=np.float64)
    logits = np.full((2, V), -1.0e4, dtype=np.float32)
    logits[0, live] = np.log(w).astype(np.float32)
    logits[1, live] = rng.normal(0, 1.2, 16).astype(np.float32)
    p0 = w / w.sum()
    q = np.zeros((1, V), dtype=np.float32)
    q[0, live] = rng.dirichlet(np.ones(16)).astype(np.float32)
    cq = np.cumsum(q[0, live].astype(np.float64))
    _, dst = mt_device(31337)
    lg = torch.from_numpy(logits).cuda()
    qd = torch.from_numpy(q).cuda()
    dd = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    N = 6000
    draws = rng.random(N)
    x0s = live[np.minimum(np.searchsorted(cq, draws * cq[-1], side="right"), 15)]
    out = torch.zeros((N, 4), dtype=torch.int32, device="cuda")
    x0d = torch.from_numpy(x0s.astype(np.int32)).cuda()
    for i in range(N):
        dd.copy_(x0d[i:i + 1])
        abi.check("spec_sample_accept", abi.spec_sample_accept(ctx.h, lg.data_ptr(), qd.data_ptr(), dd.data_ptr(),
                                                               1, dst.data_ptr(), None, res.data_ptr()))
        out[i].copy_(res)
    o = out.cpu().numpy()
    assert np.all(o[:, 2] == 0)
    first = np.where(o[:, 0] == 1, x0s, o[:, 1])
    counts = np.array([np.sum(first == t) for t in live], dtype=np.float64)
    assert counts.sum() == N
    expect = N * p0 / p0.sum()
    chi2 = float(np.sum((counts - expect) ** 2 / expect))
    assert chi2 < 40.0, (chi2, counts, expect)       # 15 dof: P(chi2 > 40) < 5e-4
    a = float(np.minimum(p0, q[0, live]).sum())
    acc = o[:, 0].mean()
    assert abs(acc - a) < 5 * math.sqrt(a * (1 - a) / N)


def test_sampled_step_matches_oracle_on_its_logits():
    import __graft_entry__
    __graft_entry__.build()
    cfg = SMALL
    ctx = runtime.Context(cfg, max_ctx=24 * 16)
    try:
        ow, dw = build_model(ctx, cfg, seed=3)
        k, n_past = 15, 71
        rng = np.random.default_rng(8)
        skipped = 0
        for t in range(3):
            dkv = runtime.DeviceKV(cfg, 24, 24)
            dkv.reset(ctx)
            dkv.extend(ctx, n_past)
            okv = oracle.KV(ocfg_of(cfg), 24, 24)
            okv.extend(n_past)
            fill_context(cfg, dkv, okv, n_past, seed=11)
            hidden = synth.normal((k + 1, cfg.hidden), 3, 500 + t)
            q = rng.dirichlet(np.ones(cfg.vocab) * 0.2, size=k).astype(np.float32)
            draft = rng.integers(0, cfg.vocab, k).astype(np.int32)
            ost, dst = mt_device(77 + t)
            h_d = torch.from_numpy(hidden).cuda()
            d_d = torch.from_numpy(draft).cuda()
            q_d = torch.from_numpy(q).cuda()
            res = torch.zeros(4, dtype=torch.int32, device="cuda")
            lg = torch.zeros((k + 1, cfg.vocab), dtype=torch.float32, device="cuda")
            am = torch.zeros(k + 1, dtype=torch.int32, device="cuda")
            taps = abi.spec_taps(None, am.data_ptr(), lg.data_ptr())
            abi.check("spec_verify_step_sampled",
                      abi.spec_verify_step_sampled(ctx.h, dw.struct(), dkv.struct(), h_d.data_ptr(), d_d.data_ptr(),
                                                   q_d.data_ptr(), k, dst.data_ptr(), res.data_ptr(), taps))
            torch.cuda.synchronize()
            r = res.cpu().numpy()
            logits = lg.cpu().numpy()
            # the step's logits agree with the oracle forward, and its argmax tap with them
            _, olog, _, st = oracle.forward(ocfg_of(cfg), ow, okv.copy(), hidden, logits=True, resid=True)
            assert st == 0
            from tests.gpu_util import assert_close
            assert_close(logits, olog, what="logits")
            assert np.array_equal(am.cpu().numpy(), np.argmax(logits, axis=1))
            # the decision on the step's own logits
            L, nxt, rc, margin = oracle.sample_accept(logits, q, draft, ost)
            assert rc == 0 and r[2] == 0
            assert np.array_equal(dst.cpu().numpy().view(np.uint32), ost)
            if margin <= MARGIN:
                skipped += 1
            else:
                assert (r[0], r[1]) == (L, nxt)
            # the KV keeps the frontier and the accepted drafts
            assert r[3] == n_past + r[0] + 1 == dkv.state()[0]
        print(f"sampled step: {skipped} of 3 decisions skipped (a uniform within {MARGIN} of its threshold)")
        assert skipped <= 1
    finally:
        ctx.close()
