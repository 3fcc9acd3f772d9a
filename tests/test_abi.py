"""The C-ABI library loads and exports every declared entry point; host-side
validation that needs no GPU.  No compute call runs here."""
import ctypes as C

import pytest

from speculative_decoding_exact_gb300 import abi


def test_library_exports_every_declared_symbol():
    declared = abi.declared_symbols()
    assert len(declared) >= 19
    L = abi.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert set(declared) == set(abi._SIGS), "binding and header disagree"


def test_strerror_texts():
    assert abi.spec_strerror(0) == "ok"
    assert "3, 7 or 15" in abi.spec_strerror(abi.SPEC_EVERIFYLEN)
    assert abi.spec_strerror(-99) == "unknown error"


def _cfg(**kw):
    base = dict(hidden=6656, n_layers=52, n_q_heads=52, n_kv_heads=4, head_dim=128, ffn=17920,
                vocab=131072, max_rows=16, page_size=16, max_ctx=2112, rms_eps=1e-6, swa_window=0,
                swa_period=0, rope_theta=0.0)
    base.update(kw)
    return abi.spec_config(*[base[f] for f, _ in abi.spec_config._fields_])


@pytest.mark.parametrize("bad", [dict(hidden=6600), dict(ffn=100), dict(head_dim=64),
                                 dict(n_kv_heads=3), dict(n_q_heads=56, n_kv_heads=2),
                                 dict(max_rows=17), dict(vocab=131071), dict(page_size=32),
                                 dict(max_ctx=4), dict(n_layers=0), dict(swa_window=-1),
                                 dict(swa_window=8, swa_period=2), dict(swa_window=4096, swa_period=2),
                                 dict(swa_window=256, swa_period=0), dict(swa_window=256, swa_period=53),
                                 dict(rope_theta=-1.0), dict(rope_theta=float("nan")),
                                 dict(rope_theta=float("inf"))])
def test_init_rejects_bad_geometry_before_touching_a_device(bad):
    h = C.c_void_p()
    rc = abi.lib().spec_verify_init(C.byref(_cfg(**bad)), None, C.byref(h))
    assert rc == abi.SPEC_EINVAL and not h.value


def test_null_arguments_are_rejected():
    L = abi.lib()
    assert L.spec_verify_init(None, None, None) == abi.SPEC_ENULL
    assert L.spec_verify_step(None, None, None, None, None, 15, None) == abi.SPEC_ENULL
    assert L.spec_kv_rollback(None, None, 0) == abi.SPEC_ENULL
    assert L.spec_gemm_q4k(None, None, 16, 256, None, 1, None) == abi.SPEC_ENULL
    L.spec_verify_destroy(None)


@pytest.mark.parametrize("sms", [1, 2, 3, 7, 64, 132, 148, 152, 160, 1000])
def test_gemm_summation_ranges_match_the_oracle(sms):
    """The GEMM's fixed fp32 order is fixed by its number of unit ranges G:
    the library's plan (host code, no device) takes the value the oracle's
    restatement of the rule gives, for the model's matrices and ragged or
    single-superblock shapes, on GPUs of any SM count."""
    import oracle
    shapes = [(7680, 6656), (6656, 6656), (35840, 6656), (6656, 17920), (131072, 6656),
              (6656, 33280), (16, 256), (272, 768), (400, 256), (2048, 512), (4096, 17920),
              (1040, 2560), (12800, 25600)]
    for N, K in shapes:
        assert abi.spec_gemm_ranges(N, K, sms) == oracle.split_ranges(N, K, sms), (N, K, sms)


def test_gemm_ranges_rejects_bad_shapes():
    for N, K, sms in [(0, 256, 152), (8, 256, 152), (16, 0, 152), (16, 200, 152), (16, 256, 0)]:
        assert abi.spec_gemm_ranges(N, K, sms) == abi.SPEC_EINVAL
