"""Single-token decode step of one Llama-style block (oracle; test infrastructure only).

Steps, in the order the pages give them (summary page, sections "어떻게
동작하나" and "무엇과 다른가"), evaluated in FP64 from the INT4 codes:

1. rho_1 = (mean x^2 + eps)^(-1/2); QKV = rho_1 * W'_qkv x, with W' = W diag(gamma)
   quantised per (row, 128 inputs) -- the row factor is applied after the
   projection's accumulation ("어떻게 동작하나").
2. RoPE on q and k at the new position L_b (Llama block; reading in rope.py).
3. k~ = H k, v~ = H v per Hadamard block; quantise to INT4 + BF16 scale and
   place at position L_b ("무엇과 다른가"; "어떻게 동작하나" for the placement).
4. q~ = H q; each query head attends over positions 0..L_b of its KV head
   (h // G) using the decoded, still-rotated cache, including the new token read
   back from its INT4 copy; o = H o~ undoes the rotation (H is its own inverse).
5. h1 = x + W_o o;  rho_2 = (mean h1^2 + eps)^(-1/2).
6. [g; u] = rho_2 * W'_gu h1;  a = g * sigmoid(g) * u  (SwiGLU).
7. out = h1 + W_down a.

Readings taken where the pages are silent: eps, the
RoPE convention, the Hadamard choice, scale divisor 7, contiguous GQA groups,
the new token attending to its own quantised K/V.
"""
from __future__ import annotations

import numpy as np

from .weights import quantize_weight, int4_matvec
from .fp8 import quantize_weight_e4m3, e4m3_matvec
from .kv import kv_quantize, KVCacheOracle
from .quant import dequantize_groups
from .hadamard import blockdiag_apply
from .rope import rope_apply
from .attention import attend


class BlockWeightsOracle:
    """Codes and scales of one block's four projections, re-derived from FP32:
    INT4 (``fmt="int4"``) or E4M3 decode weights (``fmt="e4m3"``, summary page,
    "전제와 한계"); the rest of the block is the same for both."""

    def __init__(self, shape, w: dict, fmt: str = "int4"):
        self.shape = shape
        self.fmt = fmt
        quant = {"int4": quantize_weight, "e4m3": quantize_weight_e4m3}[fmt]
        self.matvec = {"int4": int4_matvec, "e4m3": e4m3_matvec}[fmt]
        self.qkv = quant(w["wqkv"], w["gamma_attn"])
        self.o = quant(w["wo"], None)
        self.gu = quant(w["wgu"], w["gamma_ffn"])
        self.down = quant(w["wdown"], None)


def rms_factor(x, eps: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)


def decode_block(shape, wts: BlockWeightsOracle, cache: KVCacheOracle, x, pos,
                 batch_idx=None, write_cache: bool = True) -> dict:
    """Run the block for requests ``batch_idx`` (default: all rows of x).

    x: [B, H] block input values (BF16 values widened to FP64, or an FP32/FP64
    residual); pos: [B] history lengths L_b.  When ``write_cache`` the new K/V
    codes are stored into ``cache`` at position L_b.
    Returns a dict of FP64 intermediates and the new token's codes.
    """
    s = shape
    x = np.asarray(x, dtype=np.float64)
    B = x.shape[0]
    rows = list(range(B)) if batch_idx is None else list(batch_idx)
    d, nq, nkv = s.head_dim, s.n_q, s.n_kv
    G = nq // nkv
    hb, kvg = s.hb, s.kvg
    xs = x[rows]
    res = {"rows": rows}

    rho1 = rms_factor(xs, s.rms_eps)
    qkv = rho1[:, None] * wts.matvec(*wts.qkv, xs)
    res["rho1"], res["qkv"] = rho1, qkv
    q = qkv[:, : nq * d].reshape(len(rows), nq, d)
    k = qkv[:, nq * d: (nq + nkv) * d].reshape(len(rows), nkv, d)
    v = qkv[:, (nq + nkv) * d:].reshape(len(rows), nkv, d)

    o = np.zeros((len(rows), nq * d))
    kc_new = np.zeros((len(rows), nkv, d), np.uint8)
    vc_new = np.zeros((len(rows), nkv, d), np.uint8)
    ks_new = np.zeros((len(rows), nkv, d // kvg), np.float32)
    vs_new = np.zeros((len(rows), nkv, d // kvg), np.float32)
    for i, b in enumerate(rows):
        L = int(pos[b])
        qr = rope_apply(q[i], L, s.rope_base)
        kr = rope_apply(k[i], L, s.rope_base)
        kc, ks, _ = kv_quantize(kr, hb, kvg)
        vc, vs, _ = kv_quantize(v[i], hb, kvg)
        kc_new[i], vc_new[i], ks_new[i], vs_new[i] = kc, vc, ks, vs
        if write_cache:
            cache.kc[b, :, L], cache.ks[b, :, L] = kc, ks
            cache.vc[b, :, L], cache.vs[b, :, L] = vc, vs
        qt = blockdiag_apply(qr, hb)
        for j in range(nkv):
            kh = np.concatenate([cache.k_hat(b, j, L), dequantize_groups(kc[j][None], ks[j][None], kvg)])
            vh = np.concatenate([cache.v_hat(b, j, L), dequantize_groups(vc[j][None], vs[j][None], kvg)])
            for hh in range(G):
                h = j * G + hh
                ot = attend(qt[h], kh, vh)
                o[i, h * d:(h + 1) * d] = blockdiag_apply(ot, hb)
    res.update(o=o, k_codes=kc_new, v_codes=vc_new, k_scales=ks_new, v_scales=vs_new)

    attn_delta = wts.matvec(*wts.o, o)
    h1 = xs + attn_delta
    rho2 = rms_factor(h1, s.rms_eps)
    gu = rho2[:, None] * wts.matvec(*wts.gu, h1)
    g, u = gu[:, : s.inter], gu[:, s.inter:]
    a = g / (1.0 + np.exp(-g)) * u
    mlp_delta = wts.matvec(*wts.down, a)
    out = h1 + mlp_delta
    res.update(attn_delta=attn_delta, h1=h1, rho2=rho2, a=a, mlp_delta=mlp_delta, out=out)
    return res
