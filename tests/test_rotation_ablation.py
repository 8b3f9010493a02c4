"""Rotation ablation on the oracle (CPU): what the block Hadamard rotation of K/V
buys before INT4 quantisation.

Summary page, "무엇과 다른가": K and V are rotated before the INT4 cache
quantisation so that outlier channels do not set every group's scale;
"전제와 한계" quotes the perplexity cost of the INT4 cache with the rotation
(+0.20) and without it (+0.54).  The synthetic stand-in is config 2's history
(8B layer shape, context 1024): N(0, 1) K/V with four fixed outlier channels
per head scaled x20.  Quantised attention with h_b = 128 (one rotation per
head), 16 and 1 (no rotation), all with 128-channel quantisation groups, is
compared with unquantised FP64 attention over the same K/V; queries are
N(0, 1).  The GPU-side counterpart (the kernels' own attention output with
h_b = 128 and h_b = 1) is tests/test_gpu_parity.py::test_rotation_ablation.
"""
import numpy as np
import pytest

import synth
from oracle.attention import attend
from oracle.hadamard import blockdiag_apply
from oracle.kv import KVCacheOracle


def _attention_error(hb: int, n_outliers: int = 4, ctx: int = 1024, seed: int = 5):
    """(attention output rel RMS error, K reconstruction rel RMS error) for rotation block hb."""
    s = synth.L8B
    d, nkv, G = s.head_dim, s.n_kv, s.n_q // s.n_kv
    _, kf = synth.kv_history(s, 2, 1, ctx, n_outliers=n_outliers, which="k")
    _, vf = synth.kv_history(s, 2, 1, ctx, n_outliers=n_outliers, which="v")
    q = np.random.default_rng(seed).standard_normal((s.n_q, d))
    cache = KVCacheOracle(1, nkv, ctx, d, hb, d)
    cache.append(kf, vf, np.zeros(1, int))
    num = den = 0.0
    for j in range(nkv):
        K, V = kf[0, :, j].astype(np.float64), vf[0, :, j].astype(np.float64)
        kh, vh = cache.k_hat(0, j, ctx), cache.v_hat(0, j, ctx)
        for hh in range(G):
            h = j * G + hh
            ref = attend(q[h], K, V)
            o = blockdiag_apply(attend(blockdiag_apply(q[h], hb), kh, vh), hb)
            num += float(np.sum((o - ref) ** 2))
            den += float(np.sum(ref ** 2))
    k_all = np.stack([blockdiag_apply(cache.k_hat(0, j, ctx), hb) for j in range(nkv)], axis=1)
    k_err = float(np.linalg.norm(k_all - kf[0]) / np.linalg.norm(kf[0]))
    return float(np.sqrt(num / den)), k_err


def test_rotation_lowers_int4_kv_attention_error():
    e128, k128 = _attention_error(128)
    e16, k16 = _attention_error(16)
    e1, k1 = _attention_error(1)
    print(f"attention rel RMS error: h_b=128 {e128:.4f}, h_b=16 {e16:.4f}, h_b=1 {e1:.4f}; "
          f"K reconstruction: {k128:.4f} / {k16:.4f} / {k1:.4f}")
    # wider rotations spread the outliers further: error falls monotonically with h_b
    assert e128 < e16 < e1 and k128 < k16 < k1
    # the effect is large (the pages' perplexity costs differ by 2.7x)
    assert e128 < 0.6 * e1 and k128 < 0.5 * k1


@pytest.mark.parametrize("hb", [128, 1])
def test_without_outliers_rotation_changes_little(hb):
    """Control: Gaussian K/V without outlier channels quantise about equally well with
    and without the rotation (the rotation of i.i.d. Gaussian channels is again i.i.d.
    Gaussian), so the gain above comes from the outliers."""
    e, k = _attention_error(hb, n_outliers=0)
    e_ref, k_ref = _attention_error(128 if hb == 1 else 1, n_outliers=0)
    assert abs(k - k_ref) < 0.15 * k_ref
    assert abs(e - e_ref) < 0.3 * e_ref
