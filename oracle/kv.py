"""Rotated INT4 KV cache (oracle; test infrastructure only).

Summary page, "무엇과 다른가": before cache quantisation the new K and V are
rotated by a block-diagonal Hadamard transform, then stored as INT4 with BF16
scales; "어떻게 동작하나": entries are placed directly at offset(request, head,
position, channel).  Readings: the rotation block is h_b channels of one head,
one BF16 scale per (token, head, K or V, kv_group channels), kv_group = h_b by
default; the rotated value is taken to FP32 (the kernels' decision precision)
before the quantiser's decisions.
"""
import numpy as np

from .hadamard import blockdiag_apply
from .quant import quantize_groups, dequantize_groups


def kv_quantize(x, had_block: int, kv_group: int):
    """Rotate the last axis of x (head_dim) per Hadamard block and quantise.

    Returns (codes uint8 [..., d], scales f32 [..., d / kv_group], rotated FP64).
    """
    rot = blockdiag_apply(np.asarray(x, dtype=np.float64), had_block)
    codes, scales = quantize_groups(rot.astype(np.float32), kv_group)
    return codes, scales, rot


class KVCacheOracle:
    """Logical cache: codes [B, n_kv, cap, d] and scales [B, n_kv, cap, d/kvg] for K and V."""

    def __init__(self, batch: int, n_kv: int, cap: int, head_dim: int, had_block: int, kv_group: int):
        self.d, self.hb, self.kvg = head_dim, had_block, kv_group
        self.kc = np.full((batch, n_kv, cap, head_dim), 8, dtype=np.uint8)
        self.vc = np.full((batch, n_kv, cap, head_dim), 8, dtype=np.uint8)
        self.ks = np.zeros((batch, n_kv, cap, head_dim // kv_group), dtype=np.float32)
        self.vs = np.zeros((batch, n_kv, cap, head_dim // kv_group), dtype=np.float32)

    def append(self, k, v, pos):
        """k, v: [B, T, n_kv, d] values (post-RoPE); pos: [B] first position."""
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        kc, ks, _ = kv_quantize(k, self.hb, self.kvg)
        vc, vs, _ = kv_quantize(v, self.hb, self.kvg)
        t = k.shape[1]
        for b in range(k.shape[0]):
            p0 = int(pos[b])
            self.kc[b, :, p0:p0 + t] = kc[b].transpose(1, 0, 2)
            self.vc[b, :, p0:p0 + t] = vc[b].transpose(1, 0, 2)
            self.ks[b, :, p0:p0 + t] = ks[b].transpose(1, 0, 2)
            self.vs[b, :, p0:p0 + t] = vs[b].transpose(1, 0, 2)

    def append_ragged(self, k, v, cu_seqlens, pos):
        """Packed variable-length requests (the prefill side's output): k, v [total, n_kv, d]
        values (post-RoPE); request b owns rows cu_seqlens[b] .. cu_seqlens[b+1] - 1, which go
        to positions pos[b] .. pos[b] + len_b - 1 of request b (summary page, "어떻게
        동작하나": direct placement at offset(request, head, position, channel) from the
        QKV epilogue).  Each token is quantised on its own, exactly as by append."""
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        for b in range(len(cu_seqlens) - 1):
            lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
            for i in range(lo, hi):
                p = int(pos[b]) + (i - lo)
                kc, ks, _ = kv_quantize(k[i], self.hb, self.kvg)
                vc, vs, _ = kv_quantize(v[i], self.hb, self.kvg)
                self.kc[b, :, p], self.ks[b, :, p] = kc, ks
                self.vc[b, :, p], self.vs[b, :, p] = vc, vs

    def k_hat(self, b: int, h: int, n: int) -> np.ndarray:
        """Decoded (still rotated) keys of positions 0..n-1, FP64 [n, d]."""
        return dequantize_groups(self.kc[b, h, :n], self.ks[b, h, :n], self.kvg)

    def v_hat(self, b: int, h: int, n: int) -> np.ndarray:
        return dequantize_groups(self.vc[b, h, :n], self.vs[b, h, :n], self.kvg)
