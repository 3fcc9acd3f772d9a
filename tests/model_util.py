"""Build the same synthetic model for the oracle (canonical Q4_K bytes on the
host) and for the CUDA path (tiled bytes on the device)."""
import numpy as np

import oracle
from speculative_decoding_exact_gb300 import runtime, synth


def ocfg_of(cfg: runtime.ModelConfig) -> oracle.Config:
    return oracle.Config(hidden=cfg.hidden, n_layers=cfg.n_layers, n_q_heads=cfg.n_q_heads,
                         n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, ffn=cfg.ffn,
                         vocab=cfg.vocab, rms_eps=cfg.rms_eps, swa_window=cfg.swa_window,
                         swa_period=cfg.swa_period, rope_theta=cfg.rope_theta)


def build_model(ctx, cfg: runtime.ModelConfig, seed: int = 0, gammas: bool = True,
                keep_layers=None):
    """Returns (oracle.Weights or None-entries for dropped layers, runtime.DeviceWeights).
    keep_layers: host copies kept only for these layers (all when None)."""
    import torch
    H = cfg.hidden
    ow = oracle.Weights(w_qkv=[], w_o=[], w_gate_up=[], w_down=[], w_head=None)
    dw = runtime.DeviceWeights(cfg)
    if gammas:
        ow.attn_norm, ow.ffn_norm = [], []
        dw.attn_norm, dw.ffn_norm = [], []
    for l in range(cfg.n_layers):
        keep = keep_layers is None or l in keep_layers
        for j, (name, N, K) in enumerate(cfg.matrices()):
            W = synth.q4k_matrix(N, K, seed, 1000 * l + j)
            getattr(dw, name).append(runtime.upload_tiled(ctx, W, N, K))
            getattr(ow, name).append(W if keep else None)
        if gammas:
            ga = (1.0 + 0.1 * synth.normal((H,), seed, 1000 * l + 7)).astype(np.float32)
            gf = (1.0 + 0.1 * synth.normal((H,), seed, 1000 * l + 8)).astype(np.float32)
            ow.attn_norm.append(ga)
            ow.ffn_norm.append(gf)
            dw.attn_norm.append(torch.from_numpy(ga).cuda())
            dw.ffn_norm.append(torch.from_numpy(gf).cuda())
    Wh = synth.q4k_matrix(cfg.vocab, H, seed, 999999)
    dw.w_head = runtime.upload_tiled(ctx, Wh, cfg.vocab, H)
    ow.w_head = Wh
    if gammas:
        gfin = (1.0 + 0.1 * synth.normal((H,), seed, 999998)).astype(np.float32)
        ow.final_norm = gfin
        dw.final_norm = torch.from_numpy(gfin).cuda()
    return ow, dw


def add_qk_norm(cfg, ow, dw, seed: int):
    """Per-layer QK-norm gains (head_dim long, around 1) on both sides."""
    import torch
    ow.q_norm, ow.k_norm, dw.q_norm, dw.k_norm = [], [], [], []
    for l in range(cfg.n_layers):
        gq = (1.0 + 0.2 * synth.normal((cfg.head_dim,), seed, 1000 * l + 900)).astype(np.float32)
        gk = (1.0 + 0.2 * synth.normal((cfg.head_dim,), seed, 1000 * l + 901)).astype(np.float32)
        ow.q_norm.append(gq)
        ow.k_norm.append(gk)
        dw.q_norm.append(torch.from_numpy(gq).cuda())
        dw.k_norm.append(torch.from_numpy(gk).cuda())


def fill_context(cfg, dkv, okv, n_past: int, seed: int):
    """Random N(0,1) bf16 K/V rows for positions [0, n_past) of every layer, written
    identically into the device cache and the oracle's host cache (both already
    extended to n_past)."""
    for l in range(cfg.n_layers):
        kb = synth.bf16_bits(synth.normal((n_past, cfg.n_kv_heads * cfg.head_dim), seed, 2 * l + 100))
        vb = synth.bf16_bits(synth.normal((n_past, cfg.n_kv_heads * cfg.head_dim), seed, 2 * l + 101))
        if cfg.swa_index(l) >= 0:
            # a sliding-window layer keeps the last W positions in its ring
            p0 = max(0, n_past - cfg.swa_window)
            dkv.write_ring_rows(l, p0, kb[p0:], vb[p0:])
        else:
            dkv.write_rows_bulk(l, n_past, kb, vb)
        if okv is not None:
            for p in range(n_past):
                page, slot = okv.page_table[p // 16], p % 16
                okv.pool[page, l, 0, :, slot] = kb[p].reshape(cfg.n_kv_heads, cfg.head_dim)
                okv.pool[page, l, 1, :, slot] = vb[p].reshape(cfg.n_kv_heads, cfg.head_dim)
