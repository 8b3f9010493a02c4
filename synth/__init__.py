"""Seeded synthetic inputs for the INT4-weight / rotated-INT4-KV decode block.

This module serves both the CUDA path's tests/benchmark and the CPU oracle.  It
holds none of the method's arithmetic: it only draws random tensors with the
shapes and value distributions of the workloads described on the
"FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
Hopper" pages (Llama-3-8B and Llama-3-70B layer shapes, batch 1-32) and rounds
activations to BF16 with torch's own float->bfloat16 conversion.

Every draw comes from ``numpy.random.Generator(PCG64(SeedSequence([config_id,
layer, tensor_id])))`` so that the same tensor is reproduced on any machine.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

__all__ = [
    "BlockShape", "Workload", "WORKLOADS", "workload", "rng",
    "layer_weights", "activations", "kv_history", "positions",
    "model_tensors", "bf16_bits_to_f32",
    "device_layer_weights", "device_activations", "device_kv_history", "device_model_tensors",
]


@dataclasses.dataclass(frozen=True)
class BlockShape:
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    inter: int
    w_group: int = 128
    had_block: int = 0          # 0 -> head_dim
    kv_group: int = 0           # 0 -> had_block
    rms_eps: float = 1e-5
    rope_base: float = 500000.0

    @property
    def hb(self) -> int:
        return self.had_block or self.head_dim

    @property
    def kvg(self) -> int:
        return self.kv_group or self.hb

    @property
    def n_qkv(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    def replace(self, **kw) -> "BlockShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    shape: BlockShape
    batch: int
    ctx: int
    layers: int = 1
    vocab: int = 0


TINY = BlockShape(hidden=512, n_q=8, n_kv=2, head_dim=64, inter=1408, rope_base=10000.0)
L8B = BlockShape(hidden=4096, n_q=32, n_kv=8, head_dim=128, inter=14336)
L70B = BlockShape(hidden=8192, n_q=64, n_kv=8, head_dim=128, inter=28672)

WORKLOADS = {
    "tiny": Workload("tiny", 1, TINY, batch=1, ctx=128),
    "8b_b1_ctx1024": Workload("8b_b1_ctx1024", 2, L8B, batch=1, ctx=1024),
    "8b_b32_ctx4096": Workload("8b_b32_ctx4096", 3, L8B, batch=32, ctx=4096),
    **{f"70b_b{b}_ctx2048": Workload(f"70b_b{b}_ctx2048", 4, L70B, batch=b, ctx=2048)
       for b in (1, 2, 4, 8, 16, 32)},
    "70b_b1_ctx32768": Workload("70b_b1_ctx32768", 4, L70B, batch=1, ctx=32768),
    "8b_full_b1_ctx4096": Workload("8b_full_b1_ctx4096", 5, L8B, batch=1, ctx=4096,
                                   layers=32, vocab=128256),
}
# The 8B batch sweep at context 1024 (batch 1-32 on the 8B layer shape).
for _b in (2, 4, 8, 16, 32):
    WORKLOADS[f"8b_b{_b}_ctx1024"] = Workload(f"8b_b{_b}_ctx1024", 2, L8B, batch=_b, ctx=1024)


def workload(name: str) -> Workload:
    return WORKLOADS[name]


# tensor ids used in the seed sequence
T_WQKV, T_WO, T_WGATE, T_WUP, T_WDOWN, T_GATTN, T_GFFN = 1, 2, 3, 4, 5, 6, 7
T_X, T_XOUT, T_K, T_V, T_KOUT, T_VOUT, T_POS = 10, 11, 12, 13, 14, 15, 16
T_EMB, T_LM, T_GFINAL, T_TOK = 20, 21, 22, 23


def rng(config_id: int, layer: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([config_id, layer, tensor_id])))


def _to_bf16(a: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round float32 values to bfloat16 with torch; return (uint16 bits, float32 values)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, t.to(torch.float32).numpy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def layer_weights(shape: BlockShape, config_id: int, layer: int = 0,
                  rows: Optional[dict] = None) -> dict:
    """FP32 projection weights N(0, 0.02) and RMSNorm gains U(0.5, 1.5).

    Returned in the logical [N_out, K_in] row-major orientation:
    ``wqkv`` stacks the q, k and v rows; ``wgu`` stacks the gate rows then the
    up rows.
    """
    s = shape
    out = {}
    out["wqkv"] = rng(config_id, layer, T_WQKV).normal(0.0, 0.02, (s.n_qkv, s.hidden)).astype(np.float32)
    out["wo"] = rng(config_id, layer, T_WO).normal(0.0, 0.02, (s.hidden, s.n_q * s.head_dim)).astype(np.float32)
    gate = rng(config_id, layer, T_WGATE).normal(0.0, 0.02, (s.inter, s.hidden)).astype(np.float32)
    up = rng(config_id, layer, T_WUP).normal(0.0, 0.02, (s.inter, s.hidden)).astype(np.float32)
    out["wgu"] = np.concatenate([gate, up], axis=0)
    out["wdown"] = rng(config_id, layer, T_WDOWN).normal(0.0, 0.02, (s.hidden, s.inter)).astype(np.float32)
    out["gamma_attn"] = rng(config_id, layer, T_GATTN).uniform(0.5, 1.5, s.hidden).astype(np.float32)
    out["gamma_ffn"] = rng(config_id, layer, T_GFFN).uniform(0.5, 1.5, s.hidden).astype(np.float32)
    return out


def activations(shape: BlockShape, config_id: int, batch: int, layer: int = 0,
                n_outliers: int = 2, outlier_scale: float = 20.0) -> tuple[np.ndarray, np.ndarray]:
    """BF16 block input x [batch, hidden]: N(0,1) with fixed outlier channels x20.

    The outlier channels are drawn once (seeded) and are the same for every row.
    Returns (uint16 bits, float32 values).
    """
    g = rng(config_id, layer, T_X)
    x = g.standard_normal((batch, shape.hidden)).astype(np.float32)
    ch = g.choice(shape.hidden, size=n_outliers, replace=False)
    x[:, ch] *= outlier_scale
    return _to_bf16(x)


def kv_history(shape: BlockShape, config_id: int, batch: int, length: int, layer: int = 0,
               n_outliers: int = 4, outlier_scale: float = 20.0, which: str = "k"
               ) -> tuple[np.ndarray, np.ndarray]:
    """BF16 K or V history [batch, length, n_kv, head_dim] (treated as post-RoPE).

    N(0,1) with ``n_outliers`` fixed channels per head scaled x20.
    Returns (uint16 bits, float32 values).
    """
    tid = T_K if which == "k" else T_V
    g = rng(config_id, layer, tid)
    a = g.standard_normal((batch, length, shape.n_kv, shape.head_dim)).astype(np.float32)
    for h in range(shape.n_kv):
        ch = g.choice(shape.head_dim, size=n_outliers, replace=False)
        a[:, :, h, ch] *= outlier_scale
    return _to_bf16(a)


def positions(batch: int, ctx: int, ragged: bool = False, seed: int = 0) -> np.ndarray:
    """Per-request history lengths L_b (the new token goes to position L_b)."""
    if not ragged:
        return np.full(batch, ctx, dtype=np.int32)
    g = rng(99, seed, T_POS)
    return g.integers(0, ctx + 1, size=batch).astype(np.int32)


def model_tensors(shape: BlockShape, config_id: int, vocab: int, batch: int) -> dict:
    """Embedding and LM head BF16 N(0, 0.02), final gain U(0.5, 1.5), token ids."""
    emb = rng(config_id, 0, T_EMB).normal(0.0, 0.02, (vocab, shape.hidden)).astype(np.float32)
    lm = rng(config_id, 0, T_LM).normal(0.0, 0.02, (vocab, shape.hidden)).astype(np.float32)
    emb_bits, emb_f = _to_bf16(emb)
    lm_bits, lm_f = _to_bf16(lm)
    gfin = rng(config_id, 0, T_GFINAL).uniform(0.5, 1.5, shape.hidden).astype(np.float32)
    tok = rng(config_id, 0, T_TOK).integers(0, vocab, size=batch).astype(np.int32)
    return {"emb_bits": emb_bits, "emb": emb_f, "lm_bits": lm_bits, "lm": lm_f,
            "gamma_final": gfin, "tokens": tok}


# ---------------------------------------------------------------------------
# Device-side draws for large timing workloads.  Same distributions as the
# NumPy draws above (weights N(0, 0.02), gains U(0.5, 1.5), activations and K/V
# history N(0, 1) with fixed outlier channels x20), drawn on the GPU from a
# seeded torch generator so that multi-GB workloads (70B layers, the 32-layer
# step, batch-32 histories) are ready in seconds.  Not bit-identical to the NumPy
# draws; used where only the shapes and value distributions matter (timing).

def _dev_gen(device, *seed_parts: int):
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence(list(seed_parts)).generate_state(1)[0]))
    return g


def device_layer_weights(shape: BlockShape, config_id: int, layer: int, device) -> dict:
    """FP32 device tensors with the layout of ``layer_weights``."""
    s = shape
    g = _dev_gen(device, config_id, layer, 1000)
    return {
        "wqkv": torch.empty((s.n_qkv, s.hidden), device=device).normal_(0.0, 0.02, generator=g),
        "wo": torch.empty((s.hidden, s.n_q * s.head_dim), device=device).normal_(0.0, 0.02, generator=g),
        "wgu": torch.empty((2 * s.inter, s.hidden), device=device).normal_(0.0, 0.02, generator=g),
        "wdown": torch.empty((s.hidden, s.inter), device=device).normal_(0.0, 0.02, generator=g),
        "gamma_attn": torch.empty(s.hidden, device=device).uniform_(0.5, 1.5, generator=g),
        "gamma_ffn": torch.empty(s.hidden, device=device).uniform_(0.5, 1.5, generator=g),
    }


def device_activations(shape: BlockShape, config_id: int, batch: int, device, n_outliers: int = 2,
                       outlier_scale: float = 20.0) -> torch.Tensor:
    """BF16 block input [batch, hidden] as int16 bits on the device."""
    g = _dev_gen(device, config_id, 0, 1010)
    x = torch.empty((batch, shape.hidden), device=device).normal_(0.0, 1.0, generator=g)
    ch = torch.randperm(shape.hidden, device=device, generator=g)[:n_outliers]
    x[:, ch] *= outlier_scale
    return x.to(torch.bfloat16).view(torch.int16)


def device_kv_history(shape: BlockShape, config_id: int, batch: int, t0: int, t1: int, which: str, device,
                      layer: int = 0, n_outliers: int = 4, outlier_scale: float = 20.0) -> torch.Tensor:
    """BF16 K or V history positions [t0, t1) as int16 bits [batch, t1 - t0, n_kv, head_dim]; the outlier
    channels of each head are fixed per (config, layer, K/V), the values per chunk."""
    gch = _dev_gen(device, config_id, layer, 1020 + (which == "v"))
    a = torch.empty((batch, t1 - t0, shape.n_kv, shape.head_dim), device=device)
    a.normal_(0.0, 1.0, generator=_dev_gen(device, config_id, layer, 1030 + (which == "v"), t0))
    for h in range(shape.n_kv):
        ch = torch.randperm(shape.head_dim, device=device, generator=gch)[:n_outliers]
        a[:, :, h, ch] *= outlier_scale
    return a.to(torch.bfloat16).view(torch.int16)


def device_model_tensors(shape: BlockShape, config_id: int, vocab: int, batch: int, device) -> dict:
    """Embedding and LM head BF16 N(0, 0.02) (int16 bits), final gain U(0.5, 1.5), token ids."""
    g = _dev_gen(device, config_id, 0, 1040)
    emb = torch.empty((vocab, shape.hidden), device=device).normal_(0.0, 0.02, generator=g)
    lm = torch.empty((vocab, shape.hidden), device=device).normal_(0.0, 0.02, generator=g)
    return {"emb_bits": emb.to(torch.bfloat16).view(torch.int16), "lm_bits": lm.to(torch.bfloat16).view(torch.int16),
            "gamma_final": torch.empty(shape.hidden, device=device).uniform_(0.5, 1.5, generator=g),
            "tokens": torch.randint(0, vocab, (batch,), device=device, generator=g, dtype=torch.int32)}
