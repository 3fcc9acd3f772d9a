"""Device-memory plumbing around the C ABI: PyTorch allocates and frees every
buffer (weights, KV cache, inputs, outputs) and provides the stream; the
library only borrows pointers.  No arithmetic of the verify step lives here.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np
import torch

from . import abi


@dataclass
class ModelConfig:
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    page_size: int = 16
    rms_eps: float = 1e-6
    swa_window: int = 0     # sliding-window layers: window W (0 = none) ...
    swa_period: int = 0     # ... at layers l with l % period == period - 1
    rope_theta: float = 0.0  # rotary embedding base of q and k (0 = none)

    def swa_index(self, layer: int) -> int:
        """Index of layer among the sliding-window layers, or -1."""
        if self.swa_window <= 0 or self.swa_period <= 0 or layer % self.swa_period != self.swa_period - 1:
            return -1
        return layer // self.swa_period

    @property
    def swa_ring_rows(self) -> int:
        """Slots of a sliding-window ring: W rounded up to 16, plus 16 spare."""
        return (self.swa_window + 15) // 16 * 16 + 16 if self.swa_window > 0 else 0

    @property
    def n_swa(self) -> int:
        return self.n_layers // self.swa_period if self.swa_window > 0 and self.swa_period > 0 else 0

    @property
    def n_qkv(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def matrices(self):
        """(name, N, K) of every Q4_K matrix of one block, then the head."""
        H, F = self.hidden, self.ffn
        return [("w_qkv", self.n_qkv, H), ("w_o", H, self.n_q_heads * self.head_dim), ("w_gate_up", 2 * F, H),
                ("w_down", H, F)]

    def weight_bytes(self) -> int:
        per_block = sum(N * (K // 256) * 144 for _, N, K in self.matrices())
        return self.n_layers * per_block + self.vocab * (self.hidden // 256) * 144


class Context:
    """A spec_ctx bound to one CUDA stream."""

    def __init__(self, cfg: ModelConfig, max_ctx: int, max_rows: int = 16,
                 stream: torch.cuda.Stream | None = None):
        self.cfg = cfg
        self.stream = stream or torch.cuda.current_stream()
        self.c = abi.spec_config(cfg.hidden, cfg.n_layers, cfg.n_q_heads, cfg.n_kv_heads,
                                 cfg.head_dim, cfg.ffn, cfg.vocab, max_rows, cfg.page_size,
                                 max_ctx, cfg.rms_eps, cfg.swa_window, cfg.swa_period, cfg.rope_theta)
        self.h = abi.spec_verify_init(self.c, self.stream.cuda_stream)
        self.max_ctx = max_ctx

    def close(self):
        if self.h:
            abi.spec_verify_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def upload_tiled(ctx: Context, canonical: np.ndarray, N: int, K: int) -> torch.Tensor:
    """Copy canonical Q4_K bytes to the device and repack them into the tiled layout."""
    src = torch.from_numpy(np.ascontiguousarray(canonical)).to("cuda")
    dst = torch.empty_like(src)
    abi.check("spec_weights_repack", abi.spec_weights_repack(ctx.h, ptr(src), ptr(dst), N, K))
    ctx.stream.synchronize()
    del src
    return dst


class DeviceWeights:
    """Tiled Q4_K matrices and fp32 norm gains on the device."""

    def __init__(self, cfg: ModelConfig):
        self.cfg = cfg
        self.w_qkv, self.w_o, self.w_gate_up, self.w_down = [], [], [], []
        self.attn_norm: list | None = None
        self.ffn_norm: list | None = None
        self.final_norm: torch.Tensor | None = None
        self.w_head: torch.Tensor | None = None
        self.q_norm: list | None = None      # per layer: fp32 [head_dim] QK-norm gains
        self.k_norm: list | None = None
        self._keep = []

    def struct(self) -> abi.spec_weights:
        def arr(lst):
            if lst is None:
                return None
            a = (C.c_void_p * len(lst))(*[None if t is None else t.data_ptr() for t in lst])
            self._keep.append(a)
            return C.cast(a, C.c_void_p)
        return abi.spec_weights(arr(self.w_qkv), arr(self.w_o), arr(self.w_gate_up),
                                arr(self.w_down), arr(self.attn_norm), arr(self.ffn_norm),
                                ptr(self.final_norm), ptr(self.w_head), arr(self.q_norm), arr(self.k_norm))


class DeviceKV:
    """Paged bf16 KV cache and its metadata, all in device memory."""

    def __init__(self, cfg: ModelConfig, num_pages: int, max_seq_pages: int):
        self.cfg = cfg
        self.pool = torch.zeros((num_pages, cfg.n_layers, 2, cfg.n_kv_heads, cfg.page_size,
                                 cfg.head_dim), dtype=torch.bfloat16, device="cuda")
        self.page_table = torch.full((max_seq_pages,), -1, dtype=torch.int32, device="cuda")
        self.seq_len = torch.zeros(4, dtype=torch.int32, device="cuda")
        self.free_stack = torch.zeros(num_pages, dtype=torch.int32, device="cuda")
        self.free_top = torch.zeros(4, dtype=torch.int32, device="cuda")
        self.num_pages = num_pages
        self.max_seq_pages = max_seq_pages
        # sliding-window layers: ring [n_swa][K,V][n_kv][R][dh] (R = W rounded up
        # to 16, plus 16 spare slots) and the last block's state
        self.swa_ring = self.swa_state = None
        if cfg.n_swa > 0:
            self.swa_ring = torch.zeros((cfg.n_swa, 2, cfg.n_kv_heads, cfg.swa_ring_rows, cfg.head_dim),
                                        dtype=torch.bfloat16, device="cuda")
            self.swa_state = torch.full((4,), -1, dtype=torch.int32, device="cuda")

    def struct(self) -> abi.spec_kv:
        return abi.spec_kv(self.pool.data_ptr(), self.num_pages, self.max_seq_pages,
                           self.page_table.data_ptr(), self.seq_len.data_ptr(),
                           self.free_stack.data_ptr(), self.free_top.data_ptr(),
                           ptr(self.swa_ring), ptr(self.swa_state))

    def write_ring_rows(self, layer: int, pos0: int, k_bits: np.ndarray, v_bits: np.ndarray):
        """Write bf16 bit patterns [n][n_kv*dh] of positions pos0.. of a
        sliding-window layer into its ring (slot = position mod R)."""
        s = self.cfg.swa_index(layer)
        assert s >= 0
        n, R, nkv, dh = k_bits.shape[0], self.cfg.swa_ring_rows, self.cfg.n_kv_heads, self.cfg.head_dim
        kb = torch.from_numpy(k_bits.astype(np.int16).reshape(n, nkv, dh)).cuda()
        vb = torch.from_numpy(v_bits.astype(np.int16).reshape(n, nkv, dh)).cuda()
        slots = torch.from_numpy((np.arange(pos0, pos0 + n) % R).astype(np.int64)).cuda()
        ring16 = self.swa_ring.view(torch.int16)
        ring16[s, 0, :, slots, :] = kb.permute(1, 0, 2)
        ring16[s, 1, :, slots, :] = vb.permute(1, 0, 2)

    def ring_rows(self, layer: int, positions) -> np.ndarray:
        """bf16 bits [2][n_kv][len(positions)][dh] of the given positions' ring slots."""
        s = self.cfg.swa_index(layer)
        slots = np.asarray(positions) % self.cfg.swa_ring_rows
        return self.swa_ring.view(torch.int16)[s][:, :, slots, :].cpu().numpy().view(np.uint16)

    def reset(self, ctx: Context):
        abi.check("spec_kv_reset", abi.spec_kv_reset(ctx.h, self.struct()))

    def extend(self, ctx: Context, n: int):
        abi.check("spec_kv_extend", abi.spec_kv_extend(ctx.h, self.struct(), n))

    def rollback(self, ctx: Context, new_len: int):
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, self.struct(), new_len))

    def state(self):
        """(seq_len, mapped page ids, unmapped tail, free stack) read back to the host."""
        n = int(self.seq_len[0].item())
        pt = self.page_table.cpu().numpy()
        top = int(self.free_top[0].item())
        pages = (n + self.cfg.page_size - 1) // self.cfg.page_size
        return n, pt[:pages].copy(), pt[pages:].copy(), self.free_stack[:top].cpu().numpy()

    def write_rows(self, layer: int, pos0: int, k_bits: np.ndarray, v_bits: np.ndarray):
        """Write bf16 bit patterns [n][n_kv*dh] for positions pos0.. of one layer."""
        pt = self.page_table.cpu().numpy()
        n = k_bits.shape[0]
        kb = torch.from_numpy(k_bits.astype(np.int16).reshape(n, self.cfg.n_kv_heads, self.cfg.head_dim))
        vb = torch.from_numpy(v_bits.astype(np.int16).reshape(n, self.cfg.n_kv_heads, self.cfg.head_dim))
        pool16 = self.pool.view(torch.int16)
        for p in range(n):
            pos = pos0 + p
            page = int(pt[pos // self.cfg.page_size])
            slot = pos % self.cfg.page_size
            pool16[page, layer, 0, :, slot, :] = kb[p].cuda()
            pool16[page, layer, 1, :, slot, :] = vb[p].cuda()

    def write_rows_bulk(self, layer: int, n: int, k_bits: np.ndarray, v_bits: np.ndarray):
        """Write positions [0, n) of one layer in page-sized slabs."""
        pt = self.page_table.cpu().numpy()
        ps, nkv, dh = self.cfg.page_size, self.cfg.n_kv_heads, self.cfg.head_dim
        kb = torch.from_numpy(k_bits.astype(np.int16).reshape(n, nkv, dh)).cuda()
        vb = torch.from_numpy(v_bits.astype(np.int16).reshape(n, nkv, dh)).cuda()
        pool16 = self.pool.view(torch.int16)
        for lp in range((n + ps - 1) // ps):
            a, b = lp * ps, min(n, lp * ps + ps)
            page = int(pt[lp])
            pool16[page, layer, 0, :, : b - a, :] = kb[a:b].permute(1, 0, 2)
            pool16[page, layer, 1, :, : b - a, :] = vb[a:b].permute(1, 0, 2)
