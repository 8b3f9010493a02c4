"""Device-memory helpers around the C ABI: allocate packed weights, the KV
cache and the workspace with PyTorch, and fill them through the library's own
entry points.  No arithmetic of the method happens here."""
from __future__ import annotations

import numpy as np
import torch

from . import (FT_F32, FT_W_QKV, FT_W_O, FT_W_GATEUP, FT_W_DOWN, FT_WFMT_E4M3, check, ft_decode_block,
               ft_decode_workspace_bytes, ft_embed_bf16, ft_kv_append_int4, ft_kv_cache_bytes, ft_lm_head_bf16,
               ft_pack_weights_e4m3, ft_pack_weights_int4, ft_packed_weight_bytes)

ROLE_KEYS = {FT_W_QKV: ("wqkv", "gamma_attn"), FT_W_O: ("wo", None), FT_W_GATEUP: ("wgu", "gamma_ffn"),
             FT_W_DOWN: ("wdown", None)}
ROLE_NAMES = {FT_W_QKV: "qkv", FT_W_O: "o", FT_W_GATEUP: "gateup", FT_W_DOWN: "down"}


def _dev(a, dtype=None, device="cuda"):
    t = a.contiguous() if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def pack_layer(cfg, w: dict, device="cuda", stream=None) -> dict:
    """Pack the four projections of one layer from FP32 arrays or tensors (synth layout)."""
    out = {}
    for role, (wk, gk) in ROLE_KEYS.items():
        W = _dev(w[wk], device=device)
        g = _dev(w[gk], device=device) if gk else None
        packed = torch.empty(ft_packed_weight_bytes(cfg, role), dtype=torch.uint8, device=device)
        if cfg.weight_format == FT_WFMT_E4M3:
            check(ft_pack_weights_e4m3(cfg, role, W, g, packed, stream), "ft_pack_weights_e4m3")
        else:
            check(ft_pack_weights_int4(cfg, role, W, g, packed, stream), "ft_pack_weights_int4")
        out[ROLE_NAMES[role]] = packed
        del W, g
    return out


def alloc_cache(cfg, max_batch: int, max_ctx: int, device="cuda") -> torch.Tensor:
    return torch.zeros(ft_kv_cache_bytes(cfg, max_batch, max_ctx), dtype=torch.uint8, device=device)


def alloc_workspace(cfg, B: int, max_ctx: int, device="cuda") -> torch.Tensor:
    return torch.empty(ft_decode_workspace_bytes(cfg, B, max_ctx), dtype=torch.uint8, device=device)


def bits_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 BF16 bit patterns -> int16 device tensor (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)


def fill_history(cfg, cache, max_batch, max_ctx, k_bits: np.ndarray, v_bits: np.ndarray, status=None,
                 stream=None, chunk: int = 4096) -> None:
    """Append a [B, T, n_kv, d] BF16 history at positions 0..T-1 through ft_kv_append_int4."""
    B, T = k_bits.shape[:2]
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        k = bits_tensor(k_bits[:, t0:t1])
        v = bits_tensor(v_bits[:, t0:t1])
        pos = torch.full((B,), t0, dtype=torch.int32, device=k.device)
        check(ft_kv_append_int4(cfg, cache, max_batch, max_ctx, k, v, pos, B, t1 - t0, status, stream),
              "ft_kv_append_int4")


def model_step(cfg, layers, caches, max_batch, max_ctx, emb, lm, gamma_final, tokens, pos, bufs, workspaces,
               status=None, stream=None, save_layer_inputs=None):
    """One full decode step through the C ABI: embedding, every layer's decode
    block with an FP32 residual, final RMSNorm + LM head.  ``bufs`` holds two
    FP32 [B, H] device buffers and the FP32 [B, V] logits; ``save_layer_inputs``
    (optional list) receives a copy of each layer's input."""
    B = tokens.numel()
    V, H = emb.shape
    x, y = bufs["x"], bufs["y"]
    check(ft_embed_bf16(emb, tokens, x, B, V, H, status, stream), "ft_embed_bf16")
    for li, (w, c) in enumerate(zip(layers, caches)):
        if save_layer_inputs is not None:
            save_layer_inputs.append(x.clone())
        check(ft_decode_block(cfg, w, c, max_batch, max_ctx, x, y, FT_F32, pos, B, workspaces[li % len(workspaces)],
                              status, stream), "ft_decode_block")
        x, y = y, x
    check(ft_lm_head_bf16(x, gamma_final, lm, bufs["logits"], B, V, H, cfg.rms_eps, stream), "ft_lm_head_bf16")
    return x
