"""CPU oracle of the exact greedy speculative verify step.

TEST INFRASTRUCTURE ONLY.  This package exists to be compared against: the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; the product library never imports, links or falls
back to it.  It shares no code with the CUDA path.

The arithmetic lives in ``spec_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``); this module only marshals numpy arrays through
ctypes.  Sources, by page title and section:
  * Muser book Ch. 33 "Speculation: the local win and the distributed verdict"
    §33.2 (accept rule), §33.7 (carried frontier);
  * Muser book Ch. 8 "The DFlash draft" §8.6 (verify lengths, KV rewind);
  * Muser book Ch. 32 "Precision across the handoff" §32.7 (integer-dot anchor);
  * sanctum.run "The Two-Fifteen That Wasn't" (temp-0 fidelity gate).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

ST_TOKEN_RANGE, ST_NONFINITE, ST_POOL_EMPTY, ST_ROLLBACK, ST_CTX_FULL = 1, 2, 4, 8, 16


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2 -ffp-contract=off)."""
    os.makedirs(_BUILD, exist_ok=True)
    hdr = os.path.join(_HERE, "spec_oracle.h")
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(hdr))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_layers", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("page_size", C.c_int32), ("rms_eps", C.c_float),
                ("swa_window", C.c_int32), ("swa_period", C.c_int32), ("rope_theta", C.c_float)]


class _Weights(C.Structure):
    _fields_ = [("w_qkv", C.c_void_p), ("w_o", C.c_void_p), ("w_gate_up", C.c_void_p),
                ("w_down", C.c_void_p), ("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p),
                ("final_norm", C.c_void_p), ("w_head", C.c_void_p), ("q_norm", C.c_void_p),
                ("k_norm", C.c_void_p)]


class _KV(C.Structure):
    _fields_ = [("pool", C.c_void_p), ("num_pages", C.c_int32), ("max_seq_pages", C.c_int32),
                ("page_table", C.c_void_p), ("seq_len", C.c_void_p), ("free_stack", C.c_void_p),
                ("free_top", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _lib.orc_half_to_float.restype = C.c_float
        _lib.orc_half_to_float.argtypes = [C.c_uint16]
        _lib.orc_bf16_to_float.restype = C.c_float
        _lib.orc_bf16_to_float.argtypes = [C.c_uint16]
        _lib.orc_float_to_bf16.restype = C.c_uint16
        _lib.orc_float_to_bf16.argtypes = [C.c_float]
        _lib.orc_rmsnorm.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_float, C.c_void_p]
        _lib.orc_mt_next.restype = C.c_uint32
        _lib.orc_mt_next.argtypes = [C.c_void_p]
        _lib.orc_mt_seed.argtypes = [C.c_void_p, C.c_uint32]
        _lib.orc_uniform_f32.restype = C.c_float
        _lib.orc_uniform_f32.argtypes = [C.c_void_p]
        _lib.orc_layer_window.restype = C.c_int
        _lib.orc_layer_window.argtypes = [C.c_void_p, C.c_int]
        _lib.orc_sample_ordered.restype = C.c_int32
        _lib.orc_sample_ordered.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        _lib.orc_sample_accept.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                           C.c_void_p, C.c_void_p, C.c_void_p]
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def half_to_float(h: int) -> float:
    return float(lib().orc_half_to_float(int(h)))


def bf16_to_float(b: int) -> float:
    return float(lib().orc_bf16_to_float(int(b)))


def float_to_bf16(f: float) -> int:
    return int(lib().orc_float_to_bf16(float(f)))


# ---------------------------------------------------------------------------
# Q4_K accessors
# ---------------------------------------------------------------------------
def scale_min(sb: np.ndarray, j: int) -> tuple[int, int]:
    sb = np.ascontiguousarray(sb, dtype=np.uint8)
    sc, m = C.c_int(), C.c_int()
    lib().orc_q4k_scale_min(_p(sb), int(j), C.byref(sc), C.byref(m))
    return sc.value, m.value


def code(sb: np.ndarray, e: int) -> int:
    sb = np.ascontiguousarray(sb, dtype=np.uint8)
    return int(lib().orc_q4k_code(_p(sb), int(e)))


def dequant_f64(W: np.ndarray, N: int, K: int) -> np.ndarray:
    out = np.empty((N, K), dtype=np.float64)
    lib().orc_q4k_dequant_f64(_p(np.ascontiguousarray(W)), N, K, _p(out))
    return out


# ---------------------------------------------------------------------------
# quantiser, GEMM
# ---------------------------------------------------------------------------
def quantize_q8(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.int8)
    d_a = np.empty((M, K // 256), dtype=np.float32)
    A = np.empty((M, K // 32), dtype=np.int32)
    st = lib().orc_quantize_q8(_p(x), M, K, _p(q), _p(d_a), _p(A))
    return q, d_a, A, int(st)


def gemm_q4k(W: np.ndarray, N: int, K: int, q, d_a, A, sums: bool = False):
    M = q.shape[0]
    nb = K // 256
    y = np.empty((M, N), dtype=np.float32)
    isc = np.empty((M, N, nb), dtype=np.int32) if sums else None
    imn = np.empty((M, N, nb), dtype=np.int32) if sums else None
    vb = np.empty((M, N, nb), dtype=np.float32) if sums else None
    lib().orc_gemm_q4k(_p(np.ascontiguousarray(W)), N, K, _p(q), _p(d_a), _p(A), M, _p(y),
                       _p(isc), _p(imn), _p(vb))
    return (y, isc, imn, vb) if sums else y


def split_ranges(N: int, K: int, processors: int) -> int:
    """G of the fixed summation order for a GPU of `processors` SMs."""
    return int(lib().orc_split_ranges(N, K, processors))


def sum_split(vb: np.ndarray, G: int) -> np.ndarray:
    """y[m][n] = sum over superblocks of vb[m][n][b] in the fixed order of G ranges."""
    vb = np.ascontiguousarray(vb, dtype=np.float32)
    M, N, nb = vb.shape
    y = np.empty((M, N), dtype=np.float32)
    lib().orc_sum_split(_p(vb), M, N, nb, int(G), _p(y))
    return y


def linear(W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    q, d_a, A, _ = quantize_q8(x)
    return gemm_q4k(W, N, K, q, d_a, A)


def dense_f64(W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_dense_f64(_p(np.ascontiguousarray(W)), N, K, _p(x), M, _p(y))
    return y


def rmsnorm(x: np.ndarray, gamma: np.ndarray | None, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, H = x.shape
    y = np.empty_like(x)
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
    lib().orc_rmsnorm(_p(x), _p(g), M, H, C.c_float(eps), _p(y))
    return y


def silu_mul(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    up = np.ascontiguousarray(up, dtype=np.float32)
    h = np.empty_like(gate)
    lib().orc_silu_mul(_p(gate), _p(up), gate.size, _p(h))
    return h


def argmax(logits: np.ndarray):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    M, V = logits.shape
    idx = np.empty(M, dtype=np.int32)
    gap = np.empty(M, dtype=np.float32)
    lib().orc_argmax(_p(logits), M, V, _p(idx), _p(gap))
    return idx, gap


def accept(idx: np.ndarray, draft: np.ndarray, vocab: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    L, nxt = C.c_int32(), C.c_int32()
    st = lib().orc_accept(_p(idx), _p(draft), len(draft), int(vocab), C.byref(L), C.byref(nxt))
    return int(L.value), int(nxt.value), int(st)


# ---------------------------------------------------------------------------
# stochastic exact acceptance ([33] §33.2) and its MT19937 stream
# ---------------------------------------------------------------------------
MT_WORDS = 625        # 624 state words + the index of the next word


def mt_seed(seed: int) -> np.ndarray:
    st = np.zeros(MT_WORDS, dtype=np.uint32)
    lib().orc_mt_seed(_p(st), int(seed) & 0xFFFFFFFF)
    return st


def mt_next(st: np.ndarray, n: int) -> np.ndarray:
    """n raw 32-bit draws; st (a 625-word state) is advanced in place."""
    out = np.empty(n, dtype=np.uint32)
    for i in range(n):
        out[i] = lib().orc_mt_next(_p(st))
    return out


def uniform_f32(st: np.ndarray) -> float:
    return float(lib().orc_uniform_f32(_p(st)))


def softmax_row(logits: np.ndarray) -> np.ndarray:
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    p = np.empty_like(logits)
    lib().orc_softmax_row(_p(logits), logits.shape[0], _p(p))
    return p


def sample_ordered(w: np.ndarray, st: np.ndarray):
    """One draw from the distribution w (fp32 [V]): (token, margin); st (625
    words) is advanced in place."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert st.dtype == np.uint32
    margin = C.c_double(0.0)
    tok = lib().orc_sample_ordered(_p(w), w.shape[0], _p(st), C.byref(margin))
    return int(tok), float(margin.value)


def sample_accept(logits: np.ndarray, q: np.ndarray, draft: np.ndarray, st: np.ndarray):
    """(accepted, next, status, margin); st (625 words) is advanced in place.
    logits fp32 [k+1][V], q fp32 [k][V], draft int32 [k]."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    k = len(draft)
    V = logits.shape[1]
    assert logits.shape == (k + 1, V) and q.shape == (k, V) and st.dtype == np.uint32
    res = np.zeros(2, dtype=np.int32)
    margin = C.c_double(0.0)
    rc = lib().orc_sample_accept(_p(logits), _p(q), _p(draft), k, V, _p(st), _p(res), C.byref(margin))
    return int(res[0]), int(res[1]), int(rc), float(margin.value)


# ---------------------------------------------------------------------------
# model geometry, weights and the paged KV model
# ---------------------------------------------------------------------------
@dataclass
class Config:
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    page_size: int = 16
    rms_eps: float = 1e-6
    swa_window: int = 0      # sliding-window layers: every swa_period-th layer (the last of each period)
    swa_period: int = 0
    rope_theta: float = 0.0  # rotary position embedding of q and k (0 = none)

    def c(self) -> _Cfg:
        return _Cfg(self.hidden, self.n_layers, self.n_q_heads, self.n_kv_heads, self.head_dim,
                    self.ffn, self.vocab, self.page_size, self.rms_eps, self.swa_window, self.swa_period,
                    self.rope_theta)

    def layer_window(self, layer: int) -> int:
        return int(lib().orc_layer_window(C.byref(self.c()), int(layer)))

    @property
    def n_qkv(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass
class Weights:
    """Canonical Q4_K byte arrays (uint8) per layer, plus fp32 norm gains."""
    w_qkv: list
    w_o: list
    w_gate_up: list
    w_down: list
    w_head: np.ndarray
    attn_norm: list | None = None
    ffn_norm: list | None = None
    final_norm: np.ndarray | None = None
    q_norm: list | None = None       # per-layer QK-norm gains [head_dim] (None = no QK-norm)
    k_norm: list | None = None
    _keep: list = field(default_factory=list, repr=False)

    def c(self) -> _Weights:
        def arr(lst):
            if lst is None:
                return None
            ptrs = (C.c_void_p * len(lst))(*[None if a is None else a.ctypes.data for a in lst])
            self._keep.append(ptrs)
            return C.cast(ptrs, C.c_void_p)
        return _Weights(arr(self.w_qkv), arr(self.w_o), arr(self.w_gate_up), arr(self.w_down),
                        arr(self.attn_norm), arr(self.ffn_norm),
                        None if self.final_norm is None else self.final_norm.ctypes.data,
                        self.w_head.ctypes.data, arr(self.q_norm), arr(self.k_norm))


class KV:
    """Host paged KV cache: bf16 bits [num_pages][n_layers][2][n_kv][page][dh]."""

    def __init__(self, cfg: Config, num_pages: int, max_seq_pages: int):
        self.cfg = cfg
        self.pool = np.zeros((num_pages, cfg.n_layers, 2, cfg.n_kv_heads, cfg.page_size,
                              cfg.head_dim), dtype=np.uint16)
        self.page_table = np.full(max_seq_pages, -1, dtype=np.int32)
        self.seq_len_arr = np.zeros(1, dtype=np.int32)
        self.free_stack = np.zeros(num_pages, dtype=np.int32)
        self.free_top_arr = np.zeros(1, dtype=np.int32)
        self.num_pages = num_pages
        self.max_seq_pages = max_seq_pages
        self.reset()

    def c(self) -> _KV:
        return _KV(_p(self.pool), self.num_pages, self.max_seq_pages, _p(self.page_table),
                   _p(self.seq_len_arr), _p(self.free_stack), _p(self.free_top_arr))

    @property
    def seq_len(self) -> int:
        return int(self.seq_len_arr[0])

    @property
    def free_top(self) -> int:
        return int(self.free_top_arr[0])

    def reset(self):
        kv = self.c()
        lib().orc_kv_reset(C.byref(kv))

    def reserve(self, upto: int) -> int:
        kv = self.c()
        return int(lib().orc_kv_reserve(C.byref(kv), int(upto)))

    def extend(self, n: int) -> int:
        kv = self.c()
        return int(lib().orc_kv_extend(C.byref(kv), int(n)))

    def rollback(self, new_len: int) -> int:
        kv = self.c()
        return int(lib().orc_kv_rollback(C.byref(kv), int(new_len)))

    def write_row(self, layer: int, pos: int, k_row: np.ndarray, v_row: np.ndarray):
        kv = self.c()
        cfg = self.cfg.c()
        lib().orc_kv_write_row(C.byref(cfg), C.byref(kv), layer, pos,
                               _p(np.ascontiguousarray(k_row, dtype=np.float32)),
                               _p(np.ascontiguousarray(v_row, dtype=np.float32)))

    def attention(self, layer: int, q: np.ndarray, n_past: int) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.float32)
        M = q.shape[0]
        out = np.empty((M, self.cfg.n_q_heads * self.cfg.head_dim), dtype=np.float32)
        kv = self.c()
        cfg = self.cfg.c()
        lib().orc_attention(C.byref(cfg), C.byref(kv), layer, _p(q), M, n_past, _p(out))
        return out

    def committed(self):
        """The committed state: seq_len, mapped page ids, free stack contents."""
        n = self.seq_len
        pages = (n + self.cfg.page_size - 1) // self.cfg.page_size
        return (n, self.page_table[:pages].copy(), self.page_table[pages:].copy(),
                self.free_stack[: self.free_top].copy())

    def copy(self) -> "KV":
        other = KV.__new__(KV)
        other.cfg = self.cfg
        other.pool = self.pool.copy()
        other.page_table = self.page_table.copy()
        other.seq_len_arr = self.seq_len_arr.copy()
        other.free_stack = self.free_stack.copy()
        other.free_top_arr = self.free_top_arr.copy()
        other.num_pages = self.num_pages
        other.max_seq_pages = self.max_seq_pages
        return other


def qk_norm_rope(cfg: Config, w: Weights, layer: int, qkv: np.ndarray, n_past: int) -> np.ndarray:
    """QK-norm (when the layer has gains) and RoPE (when rope_theta > 0) of the
    rows of a QKV projection output [M][(nq + 2 nkv) * dh] at positions n_past.."""
    out = np.ascontiguousarray(qkv, dtype=np.float32).copy()
    lib().orc_qk_norm_rope(C.byref(cfg.c()), C.byref(w.c()), int(layer), _p(out), out.shape[0], int(n_past))
    return out


def block(cfg: Config, w: Weights, kv: KV, layer: int, x: np.ndarray, n_past: int):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    c, cw, ck = cfg.c(), w.c(), kv.c()
    st = lib().orc_block(C.byref(c), C.byref(cw), C.byref(ck), layer, _p(x), x.shape[0],
                         n_past, _p(out))
    return out, int(st)


def forward(cfg: Config, w: Weights, kv: KV, hidden: np.ndarray, logits: bool = True,
            resid: bool = False):
    hidden = np.ascontiguousarray(hidden, dtype=np.float32)
    M = hidden.shape[0]
    idx = np.empty(M, dtype=np.int32)
    lg = np.empty((M, cfg.vocab), dtype=np.float32) if logits else None
    rs = np.empty((cfg.n_layers + 1, M, cfg.hidden), dtype=np.float32) if resid else None
    c, cw, ck = cfg.c(), w.c(), kv.c()
    st = lib().orc_forward(C.byref(c), C.byref(cw), C.byref(ck), _p(hidden), M, _p(idx), _p(lg),
                           _p(rs))
    return idx, lg, rs, int(st)


def verify_step(cfg: Config, w: Weights, kv: KV, hidden: np.ndarray, draft: np.ndarray,
                logits: bool = True, resid: bool = False):
    """Returns (res = [accepted, next, status, seq_len], idx, logits, resid)."""
    hidden = np.ascontiguousarray(hidden, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    k = len(draft)
    res = np.zeros(4, dtype=np.int32)
    idx = np.full(k + 1, -1, dtype=np.int32)
    lg = np.empty((k + 1, cfg.vocab), dtype=np.float32) if logits else None
    rs = np.empty((cfg.n_layers + 1, k + 1, cfg.hidden), dtype=np.float32) if resid else None
    c, cw, ck = cfg.c(), w.c(), kv.c()
    rc = lib().orc_verify_step(C.byref(c), C.byref(cw), C.byref(ck), _p(hidden), _p(draft), k,
                               _p(res), _p(idx), _p(lg), _p(rs))
    if rc != 0:
        raise ValueError(f"verify length {k} not in (3, 7, 15)")
    return res, idx, lg, rs


ST_BAD_TREE = 0x40


TREE_MAX = 64        # nodes of a token tree ([33] §33.7 names trees of 24 to 64 nodes)


def tree_masks(tokens: np.ndarray, parent: np.ndarray, vocab: int):
    """(ancestor-or-self masks uint64 [n], status) of a token tree of up to 64 nodes."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    mask = np.zeros(max(1, len(parent)), dtype=np.uint64)
    st = lib().orc_tree_masks(_p(tokens), _p(parent), len(parent), int(vocab), _p(mask))
    return mask, int(st)


def tree_accept(idx: np.ndarray, tokens: np.ndarray, parent: np.ndarray):
    """(L, next, path[0..L]) of the greedy rule on a token tree."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    L, nxt = C.c_int32(), C.c_int32()
    path = np.zeros(TREE_MAX, dtype=np.int32)
    lib().orc_tree_accept(_p(idx), _p(tokens), _p(parent), len(parent), C.byref(L), C.byref(nxt), _p(path))
    return int(L.value), int(nxt.value), path[: L.value + 1].copy()


def verify_tree(cfg: Config, w: Weights, kv: KV, hidden: np.ndarray, tokens: np.ndarray,
                parent: np.ndarray, logits: bool = True):
    """Returns (res = [accepted, next, status, seq_len], path, idx, logits) of the
    tree verify step; node 0 = the carried frontier, parent[i] < i."""
    hidden = np.ascontiguousarray(hidden, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    n = len(parent)
    res = np.zeros(4, dtype=np.int32)
    path = np.full(TREE_MAX, -1, dtype=np.int32)
    idx = np.full(n, -1, dtype=np.int32)
    lg = np.empty((n, cfg.vocab), dtype=np.float32) if logits else None
    c, cw, ck = cfg.c(), w.c(), kv.c()
    rc = lib().orc_verify_tree(C.byref(c), C.byref(cw), C.byref(ck), _p(hidden), _p(tokens), _p(parent), n,
                               _p(res), _p(path), _p(idx), _p(lg))
    if rc:
        raise ValueError("token trees are not modelled with rotary positions")
    return res, path[: res[0] + 1].copy(), idx, lg


def serial_greedy(cfg: Config, w: Weights, kv: KV, hidden: np.ndarray, k: int):
    hidden = np.ascontiguousarray(hidden, dtype=np.float32)
    tokens = np.empty(k + 1, dtype=np.int32)
    c, cw, ck = cfg.c(), w.c(), kv.c()
    st = lib().orc_serial_greedy(C.byref(c), C.byref(cw), C.byref(ck), _p(hidden), k, _p(tokens))
    return tokens, int(st)
