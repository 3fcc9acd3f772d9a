"""GPU parity of the individual kernels against the CPU oracle, through the C ABI.

Bit-exact: quantised codes, d_a, sub-block sums, the integer sums ISc/IMn of
every (row, column, superblock), argmax indices, accepted lengths and the KV
metadata.  Tolerance (max-relative 1e-3, floored by the row rms): fp32 GEMM
outputs, logits and attention outputs.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from speculative_decoding_exact_gb300 import abi, runtime, synth  # noqa: E402
from tests.gpu_util import require_clear_rows, assert_close  # noqa: E402

SMALL = runtime.ModelConfig(hidden=3328, n_layers=2, n_q_heads=26, n_kv_heads=2, head_dim=128,
                            ffn=8960, vocab=4096)
FULL = runtime.ModelConfig(**synth.FULL)


@pytest.fixture(scope="module")
def ctx():
    import __graft_entry__
    __graft_entry__.build()
    c = runtime.Context(FULL, max_ctx=2112)
    yield c
    c.close()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def sync():
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K", [(1, 256), (4, 512), (16, 6656), (7, 17920), (16, 33280)])
def test_quantize_bit_exact(ctx, M, K):
    x = synth.normal((M, K), 3, K + M)
    x[0, :256] = 0.0                         # all-zero block
    if K > 256:
        x[-1, 256:260] = [0.5, -0.5, 1.5, 2.5]
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 256), dtype=torch.float32, device="cuda")
    A = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    xd = dev(x)
    abi.check("spec_quantize_q8", abi.spec_quantize_q8(ctx.h, xd.data_ptr(), M, K, q.data_ptr(),
                                                       da.data_ptr(), A.data_ptr()))
    sync()
    oq, oda, oA, st = oracle.quantize_q8(x)
    assert st == 0 and abi.spec_last_status(ctx.h) == 0
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(da.cpu().numpy().view(np.uint32), oda.view(np.uint32))
    assert np.array_equal(A.cpu().numpy(), oA)


def test_quantize_ties_bit_exact(ctx):
    # quotients x/d_a on or within an ulp of a half-integer: the codes follow
    # the IEEE quotient with round-half-even (d_a = 1 blocks give exact ties)
    rng = np.random.default_rng(17)
    M, K = 4, 2048
    x = np.zeros((M, K), dtype=np.float32)
    for m in range(M):
        for b in range(K // 256):
            amax = np.float32(127.0) if (m + b) % 2 == 0 else np.float32(rng.uniform(0.05, 40.0))
            d = np.float32(amax / np.float32(127.0))
            n = rng.integers(-127, 127, 256).astype(np.float32)
            blk = ((n + np.float32(0.5)) * d).astype(np.float32)
            step = rng.integers(-1, 2, 256)
            blk = np.where(step > 0, np.nextafter(blk, np.float32(np.inf)),
                           np.where(step < 0, np.nextafter(blk, np.float32(-np.inf)), blk)).astype(np.float32)
            blk = np.clip(blk, -amax, amax)
            blk[0] = amax
            x[m, 256 * b:256 * (b + 1)] = blk
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 256), dtype=torch.float32, device="cuda")
    A = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    xd = dev(x)
    abi.check("spec_quantize_q8", abi.spec_quantize_q8(ctx.h, xd.data_ptr(), M, K, q.data_ptr(),
                                                       da.data_ptr(), A.data_ptr()))
    sync()
    oq, oda, oA, st = oracle.quantize_q8(x)
    assert st == 0
    assert np.array_equal(da.cpu().numpy().view(np.uint32), oda.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(A.cpu().numpy(), oA)


def test_quantize_flags_nonfinite(ctx):
    x = synth.normal((2, 512), 0, 5)
    x[1, 300] = np.nan
    q = torch.zeros((2, 512), dtype=torch.int8, device="cuda")
    da = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    A = torch.zeros((2, 16), dtype=torch.int32, device="cuda")
    xd = dev(x)
    abi.spec_quantize_q8(ctx.h, xd.data_ptr(), 2, 512, q.data_ptr(), da.data_ptr(), A.data_ptr())
    assert abi.spec_last_status(ctx.h) & abi.ST_NONFINITE


# ---------------------------------------------------------------------------
# GEMM: exact integer sums, fp32 outputs, batch-height invariance
# ---------------------------------------------------------------------------
def run_gemm(ctx, Wt, N, K, x, sums=False):
    M = x.shape[0]
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    xd = dev(x)
    if sums:
        isc = torch.zeros((M, N, K // 256), dtype=torch.int32, device="cuda")
        imn = torch.zeros_like(isc)
        abi.check("spec_gemm_q4k_sums", abi.spec_gemm_q4k_sums(ctx.h, Wt.data_ptr(), N, K, xd.data_ptr(),
                                                               M, y.data_ptr(), isc.data_ptr(),
                                                               imn.data_ptr()))
        sync()
        return y.cpu().numpy(), isc.cpu().numpy(), imn.cpu().numpy()
    abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, Wt.data_ptr(), N, K, xd.data_ptr(), M,
                                                 y.data_ptr()))
    sync()
    return y.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(4, 2048, 512), (4, 4096, 2048), (1, 16, 256), (16, 272, 768),
                                   (3, 48, 17920), (16, 1024, 6656)])
def test_gemm_integer_sums_bit_exact(ctx, M, N, K):
    W = synth.q4k_matrix(N, K, 4, N + K)
    x = synth.normal((M, K), 4, 7 * M + K)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y, isc, imn = run_gemm(ctx, Wt, N, K, x, sums=True)
    q, da, A, _ = oracle.quantize_q8(x)
    oy, oisc, oimn, _ = oracle.gemm_q4k(W, N, K, q, da, A, sums=True)
    assert np.array_equal(isc, oisc), "ISc differs"
    assert np.array_equal(imn, oimn), "IMn differs"
    assert_close(y, oy, what="y")


@pytest.mark.parametrize("M,N,K", [(16, 6656, 6656), (16, 7680, 6656), (4, 2048, 512), (16, 272, 768),
                                   (7, 400, 256), (1, 4096, 17920), (16, 35840, 6656),
                                   (16, 131072, 6656)])
def test_gemm_output_bit_exact_in_the_fixed_order(ctx, M, N, K):
    """y itself, not only the integer sums, is bit for bit the oracle's: the
    per-superblock values agree exactly, and the oracle adds them in the
    order of the GEMM's work split for this GPU's SM count (G ranges of
    (group, superblock) units; partials in range order)."""
    W = synth.q4k_matrix(N, K, 5, N + K)
    x = synth.normal((M, K), 5, 3 * M + K)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y = run_gemm(ctx, Wt, N, K, x)
    q, da, A, _ = oracle.quantize_q8(x)
    _, _, _, vb = oracle.gemm_q4k(W, N, K, q, da, A, sums=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G = oracle.split_ranges(N, K, sms)
    oy = oracle.sum_split(vb, G)
    assert np.array_equal(y.view(np.uint32), oy.view(np.uint32)), \
        f"{int(np.sum(y.view(np.uint32) != oy.view(np.uint32)))} of {y.size} outputs differ (G {G})"


def _extreme_superblocks(rng, n):
    """n canonical superblocks drawn from three extreme patterns: every code 15
    with sc = m = 63 (the largest sums), codes alternating 0/15 with sc
    alternating 63/0 per sub-block, and random codes in {0, 15} with random
    sc, m in {0, 63}.  d and dmin vary over [1e-3, 1e-2)."""
    from tests.q4k_pack import pack_superblock
    out = np.empty((n, 144), dtype=np.uint8)
    for i in range(n):
        kind = i % 3
        d, dmin = float(rng.uniform(1e-3, 1e-2)), float(rng.uniform(1e-3, 1e-2))
        if kind == 0:
            sc, m, codes = [63] * 8, [63] * 8, [15] * 256
        elif kind == 1:
            sc, m, codes = [63, 0] * 4, [63] * 8, [15 * (e % 2) for e in range(256)]
        else:
            sc = list(63 * rng.integers(0, 2, 8))
            m = list(63 * rng.integers(0, 2, 8))
            codes = list(15 * rng.integers(0, 2, 256))
        out[i] = pack_superblock(d, dmin, sc, m, codes)
    return out


def _extreme_rows(rng, K):
    """16 activation rows whose codes are all +-127 (or 0): constant +1, constant
    -1, sign alternating per element, per sub-block and per superblock, and
    random signs (some rows with zeros); any amax gives codes +-127 here."""
    e = np.arange(K)
    rows = [np.ones(K), -np.ones(K), np.where(e % 2, -1.0, 1.0), np.where((e // 32) % 2, -1.0, 1.0),
            np.where((e // 256) % 2, -1.0, 1.0) * 3.5]
    while len(rows) < 16:
        r = rng.choice([-1.0, 1.0], K)
        if len(rows) % 3 == 0:
            r = r * rng.integers(0, 2, K)           # codes in {-127, 0, 127}
            r[::256] = 1.0                          # keep every block's amax at 1
        rows.append(r * float(rng.uniform(0.01, 100.0)))
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("K", [256, 17920])
def test_gemm_integer_sums_exact_at_extreme_magnitudes(ctx, K):
    """The tensor-core path keeps S_j, ISc and IMn exact at their largest
    magnitudes (|S_j| = 32*15*127 = 60960, |ISc| up to 8*63*60960, IMn up
    to 8*63*32*127): codes 15, scales and mins 63, activation codes +-127, and
    alternating-sign extremes, over one superblock and over 70."""
    rng = np.random.default_rng(K)
    N, nb = 256, K // 256
    W = _extreme_superblocks(rng, N * nb).reshape(-1)
    x = _extreme_rows(rng, K)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y, isc, imn = run_gemm(ctx, Wt, N, K, x, sums=True)
    q, da, A, st = oracle.quantize_q8(x)
    assert st == 0 and np.all(np.isin(q, [-127, 0, 127]))
    oy, oisc, oimn, _ = oracle.gemm_q4k(W, N, K, q, da, A, sums=True)
    assert int(np.max(np.abs(oisc))) == 8 * 63 * 60960      # the extremes are reached
    assert int(np.max(np.abs(oimn))) == 8 * 63 * 32 * 127
    assert np.array_equal(isc, oisc), "ISc differs"
    assert np.array_equal(imn, oimn), "IMn differs"
    assert_close(y, oy, what="y")


@pytest.mark.parametrize("M,N,K", [(16, 1024, 6656), (5, 2048, 17920), (1, 272, 256)])
def test_cudacore_gemm_matches_oracle_and_tensor_core_gemm(ctx, M, N, K):
    """The dp4a comparison kernel computes the same y within rounding."""
    W = synth.q4k_matrix(N, K, 12, N + K)
    x = synth.normal((M, K), 12, 3 * M + K)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    xd = dev(x)
    abi.check("spec_gemm_q4k_cudacore", abi.spec_gemm_q4k_cudacore(ctx.h, Wt.data_ptr(), N, K, xd.data_ptr(), M,
                                                                   y.data_ptr()))
    sync()
    yc = y.cpu().numpy()
    assert_close(yc, oracle.linear(W, N, K, x), what="dp4a GEMM vs oracle")
    assert_close(yc, run_gemm(ctx, Wt, N, K, x), what="dp4a GEMM vs tensor-core GEMM")


def test_bounded_waits_give_up_and_leave_the_context_usable(ctx):
    """Failure detection without a GPU fault: with the GEMM's copy producer
    held back, every consumer wait runs out (about 2 s), the kernel unwinds
    with nothing in flight and reports SPEC_ST_DEVICE_WAIT; the next GEMM on
    the same context is correct and clean."""
    import time
    N, K, M = 1024, 6656, 16
    W = synth.q4k_matrix(N, K, 13, 1)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    sync()
    t0 = time.perf_counter()
    abi.check("spec_gemm_wait_selftest", abi.spec_gemm_wait_selftest(ctx.h, Wt.data_ptr(), N, K))
    st = abi.spec_last_status(ctx.h)                 # synchronises
    dt = time.perf_counter() - t0
    assert st == abi.ST_DEVICE_WAIT, st
    assert 1.0 < dt < 30.0, dt                       # the waits' 2 s limit, not a hang
    x = synth.normal((M, K), 13, 2)
    y = run_gemm(ctx, Wt, N, K, x)
    assert abi.spec_last_status(ctx.h) == 0
    assert_close(y, oracle.linear(W, N, K, x), what="GEMM after the self-test")


@pytest.mark.parametrize("N", [6656, 26624])
def test_gemm_full_width_sampled(ctx, N):
    """Projection sweep shapes (K=6656, M=16): all outputs on the GPU, a sample of
    columns through the oracle (sampled columns are an exact sub-problem)."""
    K, M = 6656, 16
    W = synth.q4k_matrix(N, K, 5, N)
    x = synth.normal((M, K), 5, 99)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y = run_gemm(ctx, Wt, N, K, x)
    rng = np.random.default_rng(N)
    cols = np.sort(np.concatenate([rng.choice(N, 256, replace=False), [0, 255, 256, N - 1]]))
    Wsub = W.reshape(N, -1)[cols].reshape(-1)
    oy = oracle.linear(Wsub, len(cols), K, x)
    assert_close(y[:, cols], oy, what="y sampled")


@pytest.mark.parametrize("M", [2, 5, 13, 16])
def test_gemm_fc_front_projection_sampled(ctx, M):
    """Draft front projection shape (5 concatenated hidden rows: K = 33280,
    N = 6656) at M = accepted + 1 rows and at M = 16: exact integer sums and
    fp32 outputs on a sample of columns (an exact sub-problem of the oracle)."""
    N, K = 6656, 33280
    W = synth.q4k_matrix(N, K, 8, M)
    x = synth.normal((M, K), 8, 17 + M)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y, isc, imn = run_gemm(ctx, Wt, N, K, x, sums=True)
    rng = np.random.default_rng(M)
    cols = np.sort(np.concatenate([rng.choice(N, 96, replace=False), [0, 127, 128, N - 1]]))
    Wsub = W.reshape(N, -1)[cols].reshape(-1)
    q, da, A, _ = oracle.quantize_q8(x)
    oy, oisc, oimn, _ = oracle.gemm_q4k(Wsub, len(cols), K, q, da, A, sums=True)
    assert np.array_equal(isc[:, cols], oisc), "ISc differs"
    assert np.array_equal(imn[:, cols], oimn), "IMn differs"
    assert_close(y[:, cols], oy, what="y sampled")


def test_gemm_batch_height_invariance(ctx):
    N, K = 4096, 6656
    W = synth.q4k_matrix(N, K, 6, 1)
    x = synth.normal((16, K), 6, 2)
    Wt = runtime.upload_tiled(ctx, W, N, K)
    y16 = run_gemm(ctx, Wt, N, K, x)
    for M in (1, 2, 4, 8):
        yM = run_gemm(ctx, Wt, N, K, x[:M])
        assert np.array_equal(yM.view(np.uint32), y16[:M].view(np.uint32)), f"M={M}"
    for i in (3, 11, 15):
        yi = run_gemm(ctx, Wt, N, K, x[i:i + 1])
        assert np.array_equal(yi.view(np.uint32), y16[i:i + 1].view(np.uint32)), f"row {i}"


# ---------------------------------------------------------------------------
# LM head + argmax
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,centred", [(4, False), (16, False), (16, True)])
def test_lm_head_argmax(small_ctx, M, centred):
    """centred: zero-mean weights (dmin = 7.5 d), so the rows' argmaxes differ
    and the cross-CTA reduction decides among many columns."""
    ctx = small_ctx
    V, H = SMALL.vocab, SMALL.hidden
    W = synth.q4k_matrix(V, H, 7, M, dmin_over_d=7.5 if centred else None)
    x = synth.normal((M, H), 7, 3) * 3.0
    gamma = (1.0 + 0.1 * synth.normal((H,), 7, 4)).astype(np.float32)
    Wt = runtime.upload_tiled(ctx, W, V, H)
    idx = torch.zeros(M, dtype=torch.int32, device="cuda")
    lg = torch.zeros((M, V), dtype=torch.float32, device="cuda")
    xd, gd = dev(x), dev(gamma)
    abi.check("spec_lm_head_argmax", abi.spec_lm_head_argmax(ctx.h, Wt.data_ptr(), gd.data_ptr(),
                                                             xd.data_ptr(), M, idx.data_ptr(),
                                                             lg.data_ptr()))
    sync()
    xn = oracle.rmsnorm(x, gamma, 1e-6)
    olg = oracle.linear(W, V, H, xn)
    oidx, gap = oracle.argmax(olg)
    assert_close(lg.cpu().numpy(), olg, what="logits")
    gi = idx.cpu().numpy()
    require_clear_rows(gap, f"head rows (M={M}, centred={centred})")
    assert np.array_equal(gi, oidx), "argmax differs from the oracle"
    if centred:
        assert len(set(oidx.tolist())) >= M // 2, "centred weights should spread the argmax"
    # the fused argmax equals the argmax of the kernel's own logits (lowest index on ties)
    assert np.array_equal(gi, np.argmax(lg.cpu().numpy(), axis=1))


# ---------------------------------------------------------------------------
# accept + KV metadata
# ---------------------------------------------------------------------------
def make_kv(cfg, num_pages=12, max_seq_pages=12):
    return runtime.DeviceKV(cfg, num_pages, max_seq_pages)


def run_accept(ctx, idx, draft, kv=None):
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    i_d, d_d = dev(idx.astype(np.int32)), dev(draft.astype(np.int32))
    abi.check("spec_accept", abi.spec_accept(ctx.h, i_d.data_ptr(), d_d.data_ptr(), len(draft),
                                             kv.struct() if kv is not None else None,
                                             res.data_ptr()))
    sync()
    return res.cpu().numpy()


@pytest.mark.parametrize("k", [3, 7, 15])
def test_accept_patterns(ctx, k):
    V = FULL.vocab
    rng = np.random.default_rng(k)
    pats = range(1 << k) if k == 3 else rng.integers(0, 1 << k, 64)
    for pattern in pats:
        idx = rng.integers(0, V, k + 1).astype(np.int32)
        draft = np.array([idx[i] if (int(pattern) >> i) & 1 else (idx[i] + 5) % V for i in range(k)],
                         dtype=np.int32)
        L, nxt, st = oracle.accept(idx, draft, V)
        r = run_accept(ctx, idx, draft)
        assert list(r[:3]) == [L, nxt, st]


def test_accept_rollback_matches_oracle_kv(ctx):
    cfg = FULL
    rng = np.random.default_rng(1)
    for n_past, L_t in [(2055, 0), (2055, 7), (2055, 15), (16, 15), (0, 3), (31, 0)]:
        kv = make_kv(cfg, num_pages=140, max_seq_pages=140)
        kv.reset(ctx)
        kv.extend(ctx, n_past + 16)
        idx = rng.integers(0, cfg.vocab, 16).astype(np.int32)
        draft = synth.plant_draft(idx, L_t, cfg.vocab, 0, L_t)
        r = run_accept(ctx, idx, draft, kv)
        assert list(r) == [L_t, idx[L_t], 0, n_past + L_t + 1]
        # host model of the same metadata (oracle KV without a pool)
        m = _MetaKV(140, 140)
        m.extend(n_past + 16)
        m.rollback(n_past + L_t + 1)
        st = kv.state()
        assert st[0] == m.seq_len
        assert np.array_equal(st[1], m.pt[: len(st[1])]) and np.all(st[2] == -1)
        assert np.array_equal(st[3], np.array(m.stack, dtype=np.int32))


class _MetaKV:
    """KV metadata through the oracle's C functions (pool of one token)."""

    def __init__(self, num_pages, max_seq_pages):
        tiny = oracle.Config(hidden=256, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=128,
                             ffn=256, vocab=64)
        self.kv = oracle.KV(tiny, num_pages, max_seq_pages)

    def extend(self, n):
        return self.kv.extend(n)

    def rollback(self, n):
        return self.kv.rollback(n)

    @property
    def seq_len(self):
        return self.kv.seq_len

    @property
    def pt(self):
        return self.kv.page_table

    @property
    def stack(self):
        return self.kv.free_stack[: self.kv.free_top]


def test_kv_metadata_sequences_match_oracle(ctx):
    rng = np.random.default_rng(5)
    kv = make_kv(SMALL, num_pages=9, max_seq_pages=12)
    kv.reset(ctx)
    m = _MetaKV(9, 12)
    for _ in range(60):
        op = rng.integers(0, 3)
        if op == 0:
            n = int(rng.integers(0, 40))
            kv.extend(ctx, n)
            st_o = m.extend(n)
        else:
            n = int(rng.integers(0, m.seq_len + 3))
            kv.rollback(ctx, n)
            st_o = m.rollback(n)
        st_g = abi.spec_last_status(ctx.h)
        assert st_g == st_o, (op, n)
        s = kv.state()
        assert s[0] == m.seq_len
        assert np.array_equal(s[1], m.pt[: len(s[1])]) and np.all(s[2] == -1)
        assert np.array_equal(s[3], m.stack)


def test_positions_past_max_ctx_are_refused():
    """A context sized for max_ctx positions refuses a reservation past it
    (SPEC_ST_CTX_FULL) even when the page table has room, and commits
    nothing; one that ends exactly at max_ctx is served."""
    c = runtime.Context(SMALL, max_ctx=64)
    try:
        kv = make_kv(SMALL, num_pages=24, max_seq_pages=24)
        kv.reset(c)
        kv.extend(c, 60)
        assert abi.spec_last_status(c.h) == 0 and kv.state()[0] == 60
        kv.extend(c, 5)
        assert abi.spec_last_status(c.h) & abi.ST_CTX_FULL
        assert kv.state()[0] == 60
        kv.extend(c, 4)
        assert kv.state()[0] == 64
    finally:
        c.close()


def test_accept_token_range_restores_kv(ctx):
    kv = make_kv(FULL, num_pages=140, max_seq_pages=140)
    kv.reset(ctx)
    kv.extend(ctx, 40 + 16)
    idx = np.arange(16, dtype=np.int32)
    draft = idx[:15].copy()
    draft[9] = FULL.vocab
    r = run_accept(ctx, idx, draft, kv)
    assert r[2] == abi.ST_TOKEN_RANGE and r[1] == -1 and r[3] == 40
    assert kv.state()[0] == 40


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _ocfg(cfg):
    return oracle.Config(hidden=cfg.hidden, n_layers=cfg.n_layers, n_q_heads=cfg.n_q_heads,
                         n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, ffn=cfg.ffn,
                         vocab=cfg.vocab)


@pytest.fixture(scope="module")
def small_ctx():
    import __graft_entry__
    __graft_entry__.build()
    c = runtime.Context(SMALL, max_ctx=1024)
    yield c
    c.close()


def fill_kv_both(ctx, cfg, kv, okv, layer, n, seed):
    kb = synth.bf16_bits(synth.normal((n, cfg.n_kv_heads * cfg.head_dim), seed, 1))
    vb = synth.bf16_bits(synth.normal((n, cfg.n_kv_heads * cfg.head_dim), seed, 2))
    kv.write_rows_bulk(layer, n, kb, vb)
    for p in range(n):
        page, slot = okv.page_table[p // 16], p % 16
        okv.pool[page, layer, 0, :, slot] = kb[p].reshape(cfg.n_kv_heads, cfg.head_dim)
        okv.pool[page, layer, 1, :, slot] = vb[p].reshape(cfg.n_kv_heads, cfg.head_dim)


@pytest.mark.parametrize("n_past,M", [(0, 1), (5, 4), (23, 16), (77, 16), (130, 8), (500, 16)])
def test_attention_parity(small_ctx, n_past, M):
    cfg = SMALL
    kv = make_kv(cfg, num_pages=64, max_seq_pages=64)
    kv.reset(small_ctx)
    kv.extend(small_ctx, n_past + M)
    okv = oracle.KV(_ocfg(cfg), 64, 64)
    okv.extend(n_past + M)
    fill_kv_both(small_ctx, cfg, kv, okv, 1, n_past + M, 40 + n_past)
    q = synth.normal((M, cfg.n_q_heads, 128), 41, M) * 4.0
    qd = dev(q)
    out = torch.zeros((M, cfg.hidden), dtype=torch.float32, device="cuda")
    abi.check("spec_attention", abi.spec_attention(small_ctx.h, kv.struct(), 1, qd.data_ptr(), M,
                                                   out.data_ptr()))
    sync()
    ref = okv.attention(1, q, n_past)
    assert_close(out.cpu().numpy(), ref, what="attention")


@pytest.fixture(scope="module")
def long_ctx():
    import __graft_entry__
    __graft_entry__.build()
    c = runtime.Context(SMALL, max_ctx=16448)
    yield c
    c.close()


@pytest.mark.parametrize("M", [16, 4])
def test_attention_parity_long_context(long_ctx, M):
    # long-context verify (16k keys, the block straddling a page boundary):
    # the long plan's 128-key sub-chunks, chunks merged in chunk order; with
    # M = 4 rows 4..15 of every tile are dead rows
    cfg = SMALL
    n_past = 16384 + 7
    pages = (n_past + M + 15) // 16 + 1
    kv = make_kv(cfg, num_pages=pages, max_seq_pages=pages)
    kv.reset(long_ctx)
    kv.extend(long_ctx, n_past + M)
    okv = oracle.KV(_ocfg(cfg), pages, pages)
    okv.extend(n_past + M)
    fill_kv_both(long_ctx, cfg, kv, okv, 1, n_past + M, 90)
    q = synth.normal((M, cfg.n_q_heads, 128), 91, M) * 4.0
    qd = dev(q)
    out = torch.zeros((M, cfg.hidden), dtype=torch.float32, device="cuda")
    abi.check("spec_attention", abi.spec_attention(long_ctx.h, kv.struct(), 1, qd.data_ptr(), M,
                                                   out.data_ptr()))
    sync()
    ref = okv.attention(1, q, n_past)
    assert_close(out.cpu().numpy(), ref, what="attention at 16k context")


def test_attention_batch_height_invariance_long_plan(long_ctx):
    """Under the long plan (128-key sub-chunks) as under the short one: row i
    of a 16-row block equals the same row computed alone, bit for bit."""
    cfg = SMALL
    n_past, M = 1000, 16
    pages = 66
    kv = make_kv(cfg, num_pages=pages, max_seq_pages=pages)
    kv.reset(long_ctx)
    kv.extend(long_ctx, n_past + M)
    okv = oracle.KV(_ocfg(cfg), pages, pages)
    okv.extend(n_past + M)
    fill_kv_both(long_ctx, cfg, kv, okv, 0, n_past + M, 19)
    q = synth.normal((M, cfg.n_q_heads, 128), 43, 1) * 4.0
    out16 = torch.zeros((M, cfg.hidden), dtype=torch.float32, device="cuda")
    abi.check("spec_attention", abi.spec_attention(long_ctx.h, kv.struct(), 0, dev(q).data_ptr(), M,
                                                   out16.data_ptr()))
    sync()
    o16 = out16.cpu().numpy()
    for i in (0, 5, 15):
        kv.rollback(long_ctx, n_past + i + 1)
        out1 = torch.zeros((1, cfg.hidden), dtype=torch.float32, device="cuda")
        abi.check("spec_attention", abi.spec_attention(long_ctx.h, kv.struct(), 0, dev(q[i:i + 1]).data_ptr(), 1,
                                                       out1.data_ptr()))
        sync()
        assert np.array_equal(out1.cpu().numpy().view(np.uint32), o16[i:i + 1].view(np.uint32)), i
        kv.extend(long_ctx, M - i - 1)


def test_attention_batch_height_invariance(small_ctx):
    cfg = SMALL
    n_past, M = 45, 16
    kv = make_kv(cfg, num_pages=16, max_seq_pages=16)
    kv.reset(small_ctx)
    kv.extend(small_ctx, n_past + M)
    okv = oracle.KV(_ocfg(cfg), 16, 16)
    okv.extend(n_past + M)
    fill_kv_both(small_ctx, cfg, kv, okv, 0, n_past + M, 9)
    q = synth.normal((M, cfg.n_q_heads, 128), 42, 1) * 4.0
    out16 = torch.zeros((M, cfg.hidden), dtype=torch.float32, device="cuda")
    qd = dev(q)
    abi.spec_attention(small_ctx.h, kv.struct(), 0, qd.data_ptr(), M, out16.data_ptr())
    sync()
    o16 = out16.cpu().numpy()
    for i in (0, 1, 7, 15):
        kv.rollback(small_ctx, n_past + i + 1)
        out1 = torch.zeros((1, cfg.hidden), dtype=torch.float32, device="cuda")
        q1 = dev(q[i:i + 1])
        abi.spec_attention(small_ctx.h, kv.struct(), 0, q1.data_ptr(), 1, out1.data_ptr())
        sync()
        assert np.array_equal(out1.cpu().numpy().view(np.uint32), o16[i:i + 1].view(np.uint32)), i
        kv.extend(small_ctx, M - i - 1)
