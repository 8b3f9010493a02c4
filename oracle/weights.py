"""INT4 projection weights: gain folding, quantisation and the exact product
(oracle; test infrastructure only).

* Gain folding (summary page, "어떻게 동작하나"): inference weights are fixed,
  so the RMSNorm gain is folded in before quantisation, W' = W diag(gamma).
  The product is formed in FP32 because it feeds the quantiser's integer
  decisions (the kernels form it in FP32 too).  gamma_attn is folded into the
  q/k/v rows and gamma_ffn into the gate/up rows; O and down use gamma = 1.
* Group quantisation per (output row, 128 consecutive input channels) with
  BF16 scales (summary page, "무엇과 다른가"; group size and scale type from
  the workload description).
* The product y = sum_g s_{o,g} sum_{i in g} (c_{o,i} - 8) x_i is evaluated in
  FP64 from the codes, i.e. the group scale is applied after each group's
  partial sum (summary page, "무엇과 다른가").
"""
import numpy as np

from .quant import quantize_groups

W_GROUP = 128


def quantize_weight(w, gamma=None, group: int = W_GROUP):
    """FP32 W [N_out, K_in] (+ optional gamma [K_in]) -> (codes [N,K] u8, scales [N, K/group] f32)."""
    w = np.asarray(w, dtype=np.float32)
    if gamma is not None:
        w = (w * np.asarray(gamma, dtype=np.float32)[None, :]).astype(np.float32)
    return quantize_groups(w, group)


def int4_matvec(codes, scales, x, group: int = W_GROUP, row_chunk: int = 2048) -> np.ndarray:
    """y[b, o] = sum_g s[o, g] * sum_{i in g} (codes[o, i] - 8) * x[b, i], in FP64.

    ``x`` is [B, K] (or [K]).  Rows are processed in chunks only to bound
    memory; each output is computed in full from its own row.
    """
    x = np.asarray(x, dtype=np.float64)
    squeeze = x.ndim == 1
    if squeeze:
        x = x[None, :]
    n, k = codes.shape
    ng = k // group
    xg = x.reshape(x.shape[0], ng, group)
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, row_chunk):
        r1 = min(n, r0 + row_chunk)
        c = codes[r0:r1].astype(np.float64).reshape(r1 - r0, ng, group) - 8.0
        # per-group partial sums part[g, o, b] = sum_i (c - 8)[o, g, i] x[b, g, i] ...
        part = np.matmul(c.transpose(1, 0, 2), xg.transpose(1, 2, 0))
        # ... then the group scale, summed over groups
        s = np.asarray(scales[r0:r1], dtype=np.float64)          # [o, g]
        y[:, r0:r1] = np.sum(part * s.T[:, :, None], axis=0).T
    return y[0] if squeeze else y
