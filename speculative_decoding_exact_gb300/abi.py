"""ctypes binding of include/spec_verify.h — argument marshalling only.

Every function here has the name of the C entry point it calls; all work runs
in the CUDA library.  There is no fallback: if the library is missing or fails
to load, importing a function raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libspecverify.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "spec_verify.h")

SPEC_OK, SPEC_EINVAL, SPEC_EVERIFYLEN, SPEC_ENULL, SPEC_EALIGN = 0, -1, -2, -3, -4
SPEC_ENOMEM, SPEC_ECAPACITY, SPEC_ECUDA, SPEC_ENODEV = -5, -6, -7, -8
ST_TOKEN_RANGE, ST_NONFINITE, ST_POOL_EMPTY, ST_ROLLBACK, ST_CTX_FULL = 1, 2, 4, 8, 16
ST_DEVICE_WAIT, ST_BAD_TREE = 0x20, 0x40


class spec_config(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_layers", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("max_rows", C.c_int32), ("page_size", C.c_int32),
                ("max_ctx", C.c_int32), ("rms_eps", C.c_float), ("swa_window", C.c_int32),
                ("swa_period", C.c_int32), ("rope_theta", C.c_float)]


class spec_weights(C.Structure):
    _fields_ = [("w_qkv", C.c_void_p), ("w_o", C.c_void_p), ("w_gate_up", C.c_void_p),
                ("w_down", C.c_void_p), ("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p),
                ("final_norm", C.c_void_p), ("w_head", C.c_void_p), ("q_norm", C.c_void_p),
                ("k_norm", C.c_void_p)]


class spec_kv(C.Structure):
    _fields_ = [("pool", C.c_void_p), ("num_pages", C.c_int32), ("max_seq_pages", C.c_int32),
                ("page_table", C.c_void_p), ("seq_len", C.c_void_p), ("free_stack", C.c_void_p),
                ("free_top", C.c_void_p), ("swa_ring", C.c_void_p), ("swa_state", C.c_void_p)]


class spec_result(C.Structure):
    _fields_ = [("accepted_len", C.c_int32), ("next_token", C.c_int32), ("status", C.c_int32),
                ("seq_len", C.c_int32)]


class spec_taps(C.Structure):
    _fields_ = [("resid", C.c_void_p), ("argmax", C.c_void_p), ("logits", C.c_void_p)]


P = C.c_void_p
I = C.c_int
_SIGS = {
    "spec_verify_init": (I, [C.POINTER(spec_config), P, C.POINTER(P)]),
    "spec_verify_destroy": (None, [P]),
    "spec_set_stream": (I, [P, P]),
    "spec_strerror": (C.c_char_p, [I]),
    "spec_verify_step": (I, [P, C.POINTER(spec_weights), C.POINTER(spec_kv), P, P, I, P]),
    "spec_verify_step_ex": (I, [P, C.POINTER(spec_weights), C.POINTER(spec_kv), P, P, I, P,
                                C.POINTER(spec_taps)]),
    "spec_verify_step_host": (I, [P, C.POINTER(spec_weights), C.POINTER(spec_kv), P, P, I,
                                  C.POINTER(spec_result)]),
    "spec_last_step_launches": (I, [P]),
    "spec_kv_reset": (I, [P, C.POINTER(spec_kv)]),
    "spec_kv_extend": (I, [P, C.POINTER(spec_kv), C.c_int32]),
    "spec_kv_rollback": (I, [P, C.POINTER(spec_kv), C.c_int32]),
    "spec_last_status": (I, [P]),
    "spec_weights_repack": (I, [P, P, P, I, I]),
    "spec_quantize_q8": (I, [P, P, I, I, P, P, P]),
    "spec_gemm_q4k": (I, [P, P, I, I, P, I, P]),
    "spec_gemm_ranges": (I, [I, I, I]),
    "spec_gemm_q4k_sums": (I, [P, P, I, I, P, I, P, P, P]),
    "spec_gemm_q4k_cudacore": (I, [P, P, I, I, P, I, P]),
    "spec_gemm_wait_selftest": (I, [P, P, I, I]),
    "spec_lm_head_argmax": (I, [P, P, P, P, I, P, P]),
    "spec_attention": (I, [P, C.POINTER(spec_kv), I, P, I, P]),
    "spec_accept": (I, [P, P, P, I, C.POINTER(spec_kv), P]),
    "spec_profile_gemms": (I, [P, I]),
    "spec_profile_read": (I, [P, C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "spec_gemm_q4k_noalloc": (I, [P, I, I, P, I, P, P]),
    "spec_gemm_q4k_noalloc_status": (I, [P]),
    "spec_mt_seed": (I, [P, C.c_uint32]),
    "spec_set_capture": (I, [P, P, I, P]),
    "spec_set_split": (I, [P, I, P]),
    "spec_verify_tree": (I, [P, C.POINTER(spec_weights), C.POINTER(spec_kv), P, P, P, I, P, P,
                             C.POINTER(spec_taps)]),
    "spec_sample_accept": (I, [P, P, P, P, I, P, C.POINTER(spec_kv), P]),
    "spec_verify_step_sampled": (I, [P, C.POINTER(spec_weights), C.POINTER(spec_kv), P, P, P, I, P, P,
                                     C.POINTER(spec_taps)]),
}

MT_WORDS = 625

_lib = None


def declared_symbols() -> list[str]:
    """Every entry point declared in include/spec_verify.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^SPEC_API\s+[\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)))


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class SpecError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        super().__init__(f"{fn} failed: {rc} ({lib().spec_strerror(rc).decode()})")
        self.rc = rc


def check(fn: str, rc: int) -> int:
    if rc < 0:
        raise SpecError(fn, rc)
    return rc


def _call(name: str, *args) -> int:
    return getattr(lib(), name)(*args)


# thin wrappers with the C names -------------------------------------------------
def spec_verify_init(cfg: spec_config, stream: int | None):
    h = P()
    check("spec_verify_init", _call("spec_verify_init", C.byref(cfg), P(stream or 0), C.byref(h)))
    return h


def spec_verify_destroy(ctx) -> None:
    _call("spec_verify_destroy", ctx)


def spec_set_stream(ctx, stream: int | None) -> int:
    return check("spec_set_stream", _call("spec_set_stream", ctx, P(stream or 0)))


def spec_strerror(code: int) -> str:
    return _call("spec_strerror", code).decode()


def spec_verify_step(ctx, w: spec_weights, kv: spec_kv, hidden, draft, k: int, res) -> int:
    return _call("spec_verify_step", ctx, C.byref(w), C.byref(kv), P(hidden), P(draft), k, P(res))


def spec_verify_step_ex(ctx, w, kv, hidden, draft, k, res, taps: spec_taps | None) -> int:
    return _call("spec_verify_step_ex", ctx, C.byref(w), C.byref(kv), P(hidden), P(draft), k,
                 P(res), C.byref(taps) if taps is not None else None)


def spec_verify_step_host(ctx, w, kv, hidden_host, draft_host, k, res_host: spec_result) -> int:
    return _call("spec_verify_step_host", ctx, C.byref(w), C.byref(kv), P(hidden_host),
                 P(draft_host), k, C.byref(res_host))


def spec_last_step_launches(ctx) -> int:
    return _call("spec_last_step_launches", ctx)


def spec_kv_reset(ctx, kv) -> int:
    return _call("spec_kv_reset", ctx, C.byref(kv))


def spec_kv_extend(ctx, kv, n: int) -> int:
    return _call("spec_kv_extend", ctx, C.byref(kv), n)


def spec_kv_rollback(ctx, kv, new_len: int) -> int:
    return _call("spec_kv_rollback", ctx, C.byref(kv), new_len)


def spec_last_status(ctx) -> int:
    return _call("spec_last_status", ctx)


def spec_weights_repack(ctx, src, dst, N: int, K: int) -> int:
    return _call("spec_weights_repack", ctx, P(src), P(dst), N, K)


def spec_quantize_q8(ctx, x, M, K, q, d_a, A) -> int:
    return _call("spec_quantize_q8", ctx, P(x), M, K, P(q), P(d_a), P(A))


def spec_gemm_q4k(ctx, w, N, K, x, M, y) -> int:
    return _call("spec_gemm_q4k", ctx, P(w), N, K, P(x), M, P(y))


def spec_gemm_ranges(N: int, K: int, num_sms: int) -> int:
    return _call("spec_gemm_ranges", N, K, num_sms)


def spec_gemm_q4k_sums(ctx, w, N, K, x, M, y, isc, imn) -> int:
    return _call("spec_gemm_q4k_sums", ctx, P(w), N, K, P(x), M, P(y), P(isc), P(imn))


def spec_lm_head_argmax(ctx, w_head, final_norm, x, M, idx, logits) -> int:
    return _call("spec_lm_head_argmax", ctx, P(w_head), P(final_norm), P(x), M, P(idx), P(logits))


def spec_attention(ctx, kv, layer, q, M, out) -> int:
    return _call("spec_attention", ctx, C.byref(kv), layer, P(q), M, P(out))


def spec_verify_tree(ctx, w, kv, hidden, tokens, parent, n, res, path_out, taps: spec_taps | None) -> int:
    return _call("spec_verify_tree", ctx, C.byref(w), C.byref(kv), P(hidden), P(tokens), P(parent), n, P(res),
                 P(path_out), C.byref(taps) if taps is not None else None)


def spec_set_capture(ctx, layer_ids_host, n, rows) -> int:
    return _call("spec_set_capture", ctx, P(layer_ids_host), n, P(rows))


def spec_mt_seed(state_host, seed: int) -> int:
    return _call("spec_mt_seed", P(state_host), int(seed) & 0xFFFFFFFF)


def spec_sample_accept(ctx, logits, q, draft, k, mt, kv: spec_kv | None, res) -> int:
    return _call("spec_sample_accept", ctx, P(logits), P(q), P(draft), k, P(mt),
                 C.byref(kv) if kv is not None else None, P(res))


def spec_verify_step_sampled(ctx, w, kv, hidden, draft, q, k, mt, res, taps: spec_taps | None) -> int:
    return _call("spec_verify_step_sampled", ctx, C.byref(w), C.byref(kv), P(hidden), P(draft), P(q), k,
                 P(mt), P(res), C.byref(taps) if taps is not None else None)


def spec_accept(ctx, idx, draft, k, kv: spec_kv | None, res) -> int:
    return _call("spec_accept", ctx, P(idx), P(draft), k, C.byref(kv) if kv is not None else None,
                 P(res))


def spec_profile_gemms(ctx, enable: int) -> int:
    return _call("spec_profile_gemms", ctx, enable)


def spec_profile_read(ctx):
    ms, n = C.c_float(), C.c_int()
    check("spec_profile_read", _call("spec_profile_read", ctx, C.byref(ms), C.byref(n)))
    return ms.value, n.value


def spec_gemm_q4k_noalloc(w, N, K, x, M, y, stream) -> int:
    return _call("spec_gemm_q4k_noalloc", P(w), N, K, P(x), M, P(y), P(stream or 0))


def spec_gemm_q4k_noalloc_status(stream) -> int:
    return _call("spec_gemm_q4k_noalloc_status", P(stream or 0))


def spec_set_split(ctx, layer: int, event) -> int:
    """event: a cudaEvent_t handle (e.g. torch.cuda.Event().cuda_event), or None with layer = -1."""
    return _call("spec_set_split", ctx, int(layer), P(event or 0))


def spec_gemm_q4k_cudacore(ctx, w, N, K, x, M, y) -> int:
    return _call("spec_gemm_q4k_cudacore", ctx, P(w), N, K, P(x), M, P(y))


def spec_gemm_wait_selftest(ctx, w, N, K) -> int:
    return _call("spec_gemm_wait_selftest", ctx, P(w), N, K)
