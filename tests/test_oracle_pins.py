"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: printed
arithmetic from the pages (golden fixtures), closed forms, invariants, library
routines for special cases, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from oracle.block import BlockWeightsOracle, decode_block, rms_factor
from oracle.kv import KVCacheOracle, kv_quantize
from synth import BlockShape
from tests.conftest import golden_path


# ---------------------------------------------------------------- nibble decode
def test_nibble_decode_all_16_codes_golden():
    rows = [l.split() for l in open(golden_path("nibble_decode.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code, bits, val, dec in rows:
        c = int(code)
        assert int(bits, 16) == 0x4300 | c
        assert float(oracle.bf16_from_bits(np.array([int(bits, 16)], np.uint16))[0]) == float(val)
        assert oracle.nibble_decode_via_bf16(c) == float(dec) == c - 8
        # the oracle's dequantiser agrees with the pages' construction (scale 1)
        assert oracle.dequantize_groups(np.array([[c]], np.uint8), np.array([[1.0]]), 1)[0, 0] == c - 8


# ---------------------------------------------------------------- BF16 rounding
def test_bf16_rne_hand_cases():
    one = np.float32(1.0)
    cases = [
        (1.0, 1.0),
        (1.0 + 2.0 ** -8, 1.0),                        # exact tie -> even (1.0)
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),        # exact tie -> even mantissa 2
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),  # just above the tie
        (-(1.0 + 2.0 ** -8 + 2.0 ** -20), -(1.0 + 2.0 ** -7)),
        (0.0, 0.0),
    ]
    for x, want in cases:
        assert float(oracle.bf16_rne(np.float32(x))) == want, x
    assert one == 1.0


def test_bf16_rne_matches_torch_conversion():
    g = np.random.default_rng(0)
    x = (g.standard_normal(100000) * np.exp(g.uniform(-20, 20, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.bf16_rne(x), ref)


# ---------------------------------------------------------------- quantiser
def test_quantizer_golden_hand_cases():
    for line in open(golden_path("quantizer_hand_cases.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        vals, scale, codes = [p.split() for p in line.split("|")]
        x = np.array([float(v) for v in vals], np.float32)
        c, s = oracle.quantize_groups(x[None], 4)
        assert float(s[0, 0]) == float(scale[0])
        assert c[0].tolist() == [int(v) for v in codes]


def test_quantizer_brute_force_nearest_code():
    """Every unclamped code is the nearest representable (c-8)*s (ties to even)."""
    g = np.random.default_rng(1)
    x = (g.standard_normal((500, 128)) * g.uniform(0.001, 10, (500, 1))).astype(np.float32)
    x[0, :] = 0.0
    codes, s = oracle.quantize_groups(x, 128)
    assert np.all(codes[0] == 8) and s[0, 0] == 0
    for r in range(1, 60):
        sr = np.float32(s[r, 0])
        for i in range(128):
            t = np.float32(x[r, i] / sr)                 # FP32 decision, as stated
            cand = np.arange(-8, 8, dtype=np.float64)
            dist = np.abs(cand - float(t))
            best = cand[dist == dist.min()]
            want = best[0] if len(best) == 1 else best[np.argmin(np.abs(best) % 2)]  # tie -> even
            assert int(codes[r, i]) - 8 == want


def test_quantizer_invariants():
    g = np.random.default_rng(2)
    x = (g.standard_normal((300, 128)) * 3).astype(np.float32)
    codes, s = oracle.quantize_groups(x, 128)
    xh = oracle.dequantize_groups(codes, s, 128)
    # the element of largest magnitude decodes to +-7 s (amax/7 rounded to BF16 is within 2^-8)
    am = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(codes[np.arange(300), am].astype(int) - 8) == 7)
    # reconstruction error of every element is at most s/2
    assert np.all(np.abs(x - xh) <= s / 2 + 1e-12)
    # scale is BF16 and within 2^-8 relative of amax/7
    amax = np.max(np.abs(x), axis=1, keepdims=True)
    assert np.all(np.abs(s - amax / 7) <= (amax / 7) * 2.0 ** -8)
    assert np.all(oracle.bf16_rne(s) == s)


# ---------------------------------------------------------------- Hadamard
def _golden_hadamards():
    mats, cur, rows = {}, None, []
    for line in open(golden_path("hadamard_small.txt")):
        if line.startswith("#") or not line.strip():
            continue
        if line.startswith("order"):
            if cur:
                mats[cur] = np.array(rows, float)
            cur, rows = int(line.split()[1]), []
        else:
            rows.append([float(v) for v in line.split()])
    mats[cur] = np.array(rows, float)
    return mats


def test_hadamard_small_orders_golden():
    for n, m in _golden_hadamards().items():
        np.testing.assert_array_equal(oracle.sylvester(n) * np.sqrt(n), m)


@pytest.mark.parametrize("n", [1, 2, 4, 16, 64, 128])
def test_hadamard_orthogonal_symmetric_and_scipy(n):
    h = oracle.sylvester(n)
    np.testing.assert_allclose(h @ h.T, np.eye(n), atol=1e-15)
    np.testing.assert_array_equal(h, h.T)
    np.testing.assert_array_equal(h * np.sqrt(n), scipy.linalg.hadamard(n))


def test_rotation_preserves_dot_products_and_norms():
    g = np.random.default_rng(3)
    q, k = g.standard_normal((2, 50, 128))
    for hb in (16, 64, 128):
        qh, kh = oracle.blockdiag_apply(q, hb), oracle.blockdiag_apply(k, hb)
        np.testing.assert_allclose(np.sum(qh * kh, -1), np.sum(q * k, -1), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(qh, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-13)
        # self-inverse
        np.testing.assert_allclose(oracle.blockdiag_apply(qh, hb), q, atol=1e-13)


def test_rotation_is_block_diagonal():
    x = np.zeros(128)
    x[64:] = np.arange(64) + 1.0
    y = oracle.blockdiag_apply(x, 64)
    assert np.all(y[:64] == 0)
    np.testing.assert_allclose(y[64:], oracle.sylvester(64) @ x[64:], atol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_hand_case_and_complex_form():
    x = np.array([1.0, 0.0, 0.0, 0.0])
    np.testing.assert_allclose(oracle.rope_apply(x, 1, 100.0), [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    np.testing.assert_allclose(oracle.inv_freq(4, 100.0), [1.0, 0.1])
    g = np.random.default_rng(4)
    v = g.standard_normal(64)
    z = (v[:32] + 1j * v[32:]) * np.exp(1j * 37 * oracle.inv_freq(64, 10000.0))
    np.testing.assert_allclose(oracle.rope_apply(v, 37, 10000.0), np.concatenate([z.real, z.imag]), atol=1e-13)


def test_rope_identity_norm_and_relative_position():
    g = np.random.default_rng(5)
    q, k = g.standard_normal((2, 128))
    np.testing.assert_array_equal(oracle.rope_apply(q, 0, 5e5), q)
    np.testing.assert_allclose(np.linalg.norm(oracle.rope_apply(q, 999, 5e5)), np.linalg.norm(q), rtol=1e-13)
    a = oracle.rope_apply(q, 1000, 5e5) @ oracle.rope_apply(k, 990, 5e5)
    b = oracle.rope_apply(q, 13, 5e5) @ oracle.rope_apply(k, 3, 5e5)
    assert abs(a - b) < 1e-10


# ---------------------------------------------------------------- gain folding / row factor
def test_gain_folding_and_deferred_row_factor():
    g = np.random.default_rng(6)
    w = g.standard_normal((96, 256))
    gamma = g.uniform(0.5, 1.5, 256)
    x = g.standard_normal(256) * 5
    rho = 1.0 / np.sqrt(np.mean(x * x) + 1e-5)
    explicit = w @ (gamma * (rho * x))          # RMSNorm then matmul
    folded = rho * ((w * gamma[None, :]) @ x)    # W' = W diag(gamma), rho after accumulation
    np.testing.assert_allclose(folded, explicit, rtol=1e-12)
    # RMSNorm is scale invariant (eps -> 0)
    assert abs(rms_factor(3 * x, 0.0) * 3 - rms_factor(x, 0.0)) < 1e-12
    assert abs(rms_factor(np.array([3.0, 4.0]), 0.0) - 1 / math.sqrt(12.5)) < 1e-15


def test_int4_matvec_matches_dense_and_brute_force():
    g = np.random.default_rng(7)
    w = g.normal(0, 0.02, (40, 384)).astype(np.float32)
    gamma = g.uniform(0.5, 1.5, 384).astype(np.float32)
    codes, s = oracle.quantize_weight(w, gamma)
    x = g.standard_normal((3, 384))
    dense = oracle.dequantize_groups(codes, s, 128) @ x.T
    np.testing.assert_allclose(oracle.int4_matvec(codes, s, x, row_chunk=7), dense.T, rtol=1e-12)
    # brute force, one output
    o, b = 5, 1
    acc = 0.0
    for gi in range(3):
        part = sum((int(codes[o, gi * 128 + i]) - 8) * x[b, gi * 128 + i] for i in range(128))
        acc += float(s[o, gi]) * part
    assert abs(acc - oracle.int4_matvec(codes, s, x)[b, o]) < 1e-12
    # gamma is folded in FP32 before quantising
    c2, s2 = oracle.quantize_groups((w * gamma[None]).astype(np.float32), 128)
    np.testing.assert_array_equal(c2, codes)


# ---------------------------------------------------------------- attention
def _brute_attention(q, K, V):
    d = len(q)
    sc = [sum(q[c] * K[j][c] for c in range(d)) / math.sqrt(d) for j in range(len(K))]
    m = max(sc)
    e = [math.exp(v - m) for v in sc]
    z = sum(e)
    return [sum(e[j] * V[j][c] for j in range(len(K))) / z for c in range(d)]


def test_attention_brute_force_tiny():
    g = np.random.default_rng(8)
    q, K, V = g.standard_normal(8), g.standard_normal((5, 8)) * 2, g.standard_normal((5, 8))
    np.testing.assert_allclose(oracle.attend(q, K, V), _brute_attention(q, K, V), rtol=1e-13)


def test_attention_special_cases():
    g = np.random.default_rng(9)
    q, v = g.standard_normal(16), g.standard_normal(16)
    np.testing.assert_allclose(oracle.attend(q, g.standard_normal((1, 16)), v[None]), v, rtol=1e-15)
    k = g.standard_normal(16)
    V = g.standard_normal((6, 16))
    np.testing.assert_allclose(oracle.attend(q, np.tile(k, (6, 1)), V), V.mean(0), rtol=1e-13)


@pytest.mark.parametrize("n_split", [1, 2, 7, 64])
def test_split_kv_merge_invariance(n_split):
    g = np.random.default_rng(10)
    q, K, V = g.standard_normal(128), g.standard_normal((300, 128)) * 3, g.standard_normal((300, 128))
    np.testing.assert_allclose(oracle.attend_split(q, K, V, n_split), oracle.attend(q, K, V), rtol=1e-12, atol=1e-14)


def test_rotated_attention_equals_unrotated_without_quantisation():
    g = np.random.default_rng(11)
    q, K, V = g.standard_normal(128), g.standard_normal((40, 128)) * 2, g.standard_normal((40, 128))
    for hb in (32, 128):
        R = lambda a: oracle.blockdiag_apply(a, hb)
        ot = oracle.attend(R(q), R(K), R(V))
        np.testing.assert_allclose(R(ot), oracle.attend(q, K, V), rtol=1e-12, atol=1e-14)


def test_swiglu_closed_form():
    gg = np.array([0.0, 1.0, -2.0])
    u = np.array([3.0, 2.0, 1.0])
    a = gg / (1.0 + np.exp(-gg)) * u
    np.testing.assert_allclose(a, [0.0, 2.0 / (1.0 + math.exp(-1.0)), -2.0 / (1.0 + math.exp(2.0))], rtol=1e-15)


# ---------------------------------------------------------------- whole block
MINI = BlockShape(hidden=256, n_q=8, n_kv=2, head_dim=16, inter=256, rope_base=10000.0)


def _mini_setup(shape=MINI, B=2, L=5, seed=12, zero=(), fmt="int4"):
    g = np.random.default_rng(seed)
    w = {
        "wqkv": g.normal(0, 0.05, (shape.n_qkv, shape.hidden)).astype(np.float32),
        "wo": g.normal(0, 0.05, (shape.hidden, shape.n_q * shape.head_dim)).astype(np.float32),
        "wgu": g.normal(0, 0.05, (2 * shape.inter, shape.hidden)).astype(np.float32),
        "wdown": g.normal(0, 0.05, (shape.hidden, shape.inter)).astype(np.float32),
        "gamma_attn": g.uniform(0.5, 1.5, shape.hidden).astype(np.float32),
        "gamma_ffn": g.uniform(0.5, 1.5, shape.hidden).astype(np.float32),
    }
    for z in zero:
        w[z][:] = 0
    wts = BlockWeightsOracle(shape, w, fmt)
    cache = KVCacheOracle(B, shape.n_kv, L + 4, shape.head_dim, shape.hb, shape.kvg)
    if L:
        cache.append(g.standard_normal((B, L, shape.n_kv, shape.head_dim)),
                     g.standard_normal((B, L, shape.n_kv, shape.head_dim)), np.zeros(B, int))
    x = g.standard_normal((B, shape.hidden)) * 2
    return w, wts, cache, x


def test_block_residual_only_when_output_weights_zero():
    w, wts, cache, x = _mini_setup(zero=("wo", "wdown"))
    r = decode_block(MINI, wts, cache, x, np.array([5, 5]))
    np.testing.assert_array_equal(r["out"], x)
    w, wts, cache, x = _mini_setup(zero=("wdown",))
    r = decode_block(MINI, wts, cache, x, np.array([5, 5]))
    np.testing.assert_array_equal(r["out"], r["h1"])


def test_block_single_key_closed_form():
    """L_b = 0: each head attends to the new token only, so o_h = H * dequant(quant(H v))."""
    w, wts, cache, x = _mini_setup(L=0)
    r = decode_block(MINI, wts, cache, x, np.array([0, 0]))
    s = MINI
    for i in range(2):
        rho = 1 / np.sqrt(np.mean(x[i] ** 2) + s.rms_eps)
        wv = oracle.dequantize_groups(*wts.qkv, 128)[(s.n_q + s.n_kv) * s.head_dim:]
        v = (rho * (wv @ x[i])).reshape(s.n_kv, s.head_dim)
        for j in range(s.n_kv):
            c, sc, _ = kv_quantize(v[j], s.hb, s.kvg)
            vh = oracle.sylvester(s.hb) @ oracle.dequantize_groups(c, sc, s.kvg)
            for hh in range(s.n_q // s.n_kv):
                h = j * (s.n_q // s.n_kv) + hh
                np.testing.assert_allclose(r["o"][i, h * 16:(h + 1) * 16], vh, rtol=1e-12, atol=1e-14)


def test_block_output_projection_orientation():
    """A single nonzero W_o[r, c] moves exactly one residual channel by w * o[c]."""
    w, wts, cache, x = _mini_setup(zero=("wdown",))
    w["wo"][:] = 0
    w["wo"][7, 19] = 0.5
    wts = BlockWeightsOracle(MINI, w)
    r = decode_block(MINI, wts, cache, x, np.array([5, 5]))
    delta = r["h1"] - x
    assert np.count_nonzero(np.abs(delta) > 0) <= 2
    w_hat = oracle.dequantize_groups(*wts.o, 128)[7, 19]      # 0.5 after INT4 quantisation
    assert abs(w_hat - 0.5) <= 0.5 * 2.0 ** -8
    np.testing.assert_allclose(delta[:, 7], w_hat * r["o"][:, 19], rtol=1e-12)


def test_block_gqa_head_mapping():
    """Query head h reads KV head h // G (contiguous groups, no head expansion).

    KV head 1's history keys are made huge and its values constant, so any query
    head reading KV head 1 returns (almost exactly) that constant; heads of group 0
    must not."""
    w, wts, cache, x = _mini_setup(L=6)
    s = MINI
    G = s.n_q // s.n_kv
    cache.kc[:, 1] = 15
    cache.ks[:, 1] = 0.0
    cache.vc[:, 1] = 15                 # decoded value 7 * 0.25 = 1.75 in every rotated channel
    cache.vs[:, 1] = 0.25
    # zero keys for KV head 1 history -> uniform attention over history + new token
    r = decode_block(s, wts, cache, x, np.array([6, 6]), write_cache=False)
    const = oracle.sylvester(s.hb) @ np.full(s.head_dim, 1.75)
    for i in range(2):
        vnew = oracle.dequantize_groups(r["v_codes"][i, 1], r["v_scales"][i, 1], s.kvg)
        for h in range(G, 2 * G):
            # scores: history keys decode to 0 -> score 0; the new key has its own score
            qkv = r["qkv"][i]
            qt = oracle.blockdiag_apply(oracle.rope_apply(qkv[h * 16:(h + 1) * 16], 6, s.rope_base), s.hb)
            kn = oracle.dequantize_groups(r["k_codes"][i, 1], r["k_scales"][i, 1], s.kvg)
            sn = qt @ kn / 4.0
            p_new = math.exp(sn) / (6 + math.exp(sn))
            want = (1 - p_new) * const + p_new * (oracle.sylvester(s.hb) @ vnew)
            np.testing.assert_allclose(r["o"][i, h * 16:(h + 1) * 16], want, rtol=1e-12, atol=1e-13)
        for h in range(G):
            assert not np.allclose(r["o"][i, h * 16:(h + 1) * 16], const, atol=1e-3)


def _brute_block(shape, wts, cache, x, L):
    """Explicit-loop evaluation of the block for one request (tiny shapes only)."""
    s = shape
    H, d, nq, nkv = s.hidden, s.head_dim, s.n_q, s.n_kv
    G = nq // nkv
    def dequant(codes, scales):
        if wts.fmt == "e4m3":   # E4M3 values times the group scale, element by element
            return [[float(oracle.e4m3_decode(codes[r][i])) * float(scales[r][i // 128]) for i in range(len(codes[r]))]
                    for r in range(len(codes))]
        return oracle.dequantize_groups(codes, scales, 128)
    W = {k: dequant(*getattr(wts, k)) for k in ("qkv", "o", "gu", "down")}
    rho = 1 / math.sqrt(sum(v * v for v in x) / H + s.rms_eps)
    y = [rho * sum(W["qkv"][r][i] * x[i] for i in range(H)) for r in range(s.n_qkv)]

    def rope(vec):
        out = [0.0] * d
        for i in range(d // 2):
            a = L * s.rope_base ** (-2.0 * i / d)
            out[i] = vec[i] * math.cos(a) - vec[i + d // 2] * math.sin(a)
            out[i + d // 2] = vec[i + d // 2] * math.cos(a) + vec[i] * math.sin(a)
        return out

    def had(vec):
        n = s.hb
        out = []
        for b0 in range(0, d, n):
            for i in range(n):
                out.append(sum((-1) ** bin(i & j).count("1") * vec[b0 + j] for j in range(n)) / math.sqrt(n))
        return out

    def quant(vec):
        amax = max(abs(v) for v in vec)
        sc = float(oracle.bf16_rne(np.float32(np.float32(amax) / np.float32(7))))
        if sc == 0:
            return [0.0] * len(vec)
        return [sc * max(-8, min(7, float(np.rint(np.float32(np.float32(v) / np.float32(sc)))))) for v in vec]

    o = []
    for h in range(nq):
        j = h // G
        q = had(rope(y[h * d:(h + 1) * d]))
        kn = quant(had(rope(y[(nq + j) * d:(nq + j + 1) * d])))
        vn = quant(had(y[(nq + nkv + j) * d:(nq + nkv + j + 1) * d]))
        Ks = [list(cache.k_hat(0, j, L)[p]) for p in range(L)] + [kn]
        Vs = [list(cache.v_hat(0, j, L)[p]) for p in range(L)] + [vn]
        o += had(_brute_attention(q, Ks, Vs))
    h1 = [x[r] + sum(W["o"][r][c] * o[c] for c in range(nq * d)) for r in range(H)]
    rho2 = 1 / math.sqrt(sum(v * v for v in h1) / H + s.rms_eps)
    gu = [rho2 * sum(W["gu"][r][i] * h1[i] for i in range(H)) for r in range(2 * s.inter)]
    a = [gu[i] / (1 + math.exp(-gu[i])) * gu[s.inter + i] for i in range(s.inter)]
    return [h1[r] + sum(W["down"][r][i] * a[i] for i in range(s.inter)) for r in range(H)]


@pytest.mark.parametrize("fmt", ["int4", "e4m3"])
def test_block_brute_force_tiny(fmt):
    """The whole block (INT4 or E4M3 decode weights) against explicit loops."""
    shape = BlockShape(hidden=128, n_q=16, n_kv=4, head_dim=8, inter=128, rope_base=10000.0)
    w, wts, cache, x = _mini_setup(shape=shape, B=1, L=3, seed=13, fmt=fmt)
    r = decode_block(shape, wts, cache, x, np.array([3]), write_cache=False)
    want = _brute_block(shape, wts, cache, list(x[0]), 3)
    np.testing.assert_allclose(r["out"][0], want, rtol=1e-11, atol=1e-12)


def test_block_e4m3_residual_only_and_closer_to_dense():
    """E4M3 decode weights: zero output weights leave the residual; with the same FP32 weights
    the E4M3 block's MLP lies closer to the unquantised FP64 MLP (on the same h1) than the
    INT4 one (finer codes)."""
    w, wts, cache, x = _mini_setup(zero=("wo", "wdown"), fmt="e4m3")
    r = decode_block(MINI, wts, cache, x, np.array([5, 5]), write_cache=False)
    np.testing.assert_array_equal(r["out"], x)

    def mlp_error(fmt):
        w32, wq, cq, xq = _mini_setup(fmt=fmt, seed=21)
        res = decode_block(MINI, wq, cq, xq, np.array([5, 5]), write_cache=False)
        h1 = res["h1"]
        rho2 = 1.0 / np.sqrt(np.mean(h1 * h1, axis=-1) + MINI.rms_eps)
        wgu = w32["wgu"].astype(np.float64) * w32["gamma_ffn"].astype(np.float64)[None, :]
        gu = rho2[:, None] * (h1 @ wgu.T)
        g_, u_ = gu[:, :MINI.inter], gu[:, MINI.inter:]
        dense = (g_ / (1 + np.exp(-g_)) * u_) @ w32["wdown"].astype(np.float64).T
        return np.linalg.norm(res["mlp_delta"] - dense) / np.linalg.norm(dense)

    e8, e4 = mlp_error("e4m3"), mlp_error("int4")
    assert e8 < 0.5 * e4, (e8, e4)


# ---------------------------------------------------------------- KV cache placement
def test_kv_cache_append_places_each_token_at_its_position():
    """Distinct rows per (request, token, head) land at [request, head, pos0 + token]
    (offset(request, head, position, channel) placement); nothing else is touched."""
    B, T, nkv, d, cap = 3, 4, 2, 8, 14
    c = KVCacheOracle(B, nkv, cap, d, d, d)
    pos0 = np.array([0, 5, 9])
    g = np.random.default_rng(4)
    pat = g.standard_normal(d)
    k = np.empty((B, T, nkv, d))
    v = np.empty((B, T, nkv, d))
    for b in range(B):
        for t in range(T):
            for h in range(nkv):
                amp = 1.0 + 100 * b + 10 * t + h          # a different scale for every slot
                k[b, t, h] = amp * pat
                v[b, t, h] = -amp * pat[::-1]
    c.append(k, v, pos0)
    seen = np.zeros((B, nkv, cap), bool)
    for b in range(B):
        for t in range(T):
            for h in range(nkv):
                p = pos0[b] + t
                for cache_c, cache_s, row in ((c.kc, c.ks, k[b, t, h]), (c.vc, c.vs, v[b, t, h])):
                    codes, sc, _ = kv_quantize(row, d, d)   # the row quantised on its own
                    np.testing.assert_array_equal(cache_c[b, h, p], codes)
                    np.testing.assert_array_equal(cache_s[b, h, p], sc)
                seen[b, h, p] = True
    assert np.all(c.kc[~seen] == 8) and np.all(c.vc[~seen] == 8)
    assert np.all(c.ks[~seen] == 0) and np.all(c.vs[~seen] == 0)
    assert len(np.unique(c.ks[seen])) == seen.sum()
    # decoding reads the same slots back
    np.testing.assert_array_equal(c.k_hat(2, 1, 13)[9:], oracle.dequantize_groups(c.kc[2, 1, 9:13], c.ks[2, 1, 9:13], d))


# ---------------------------------------------------------------- full step
TINY_MODEL = BlockShape(hidden=128, n_q=16, n_kv=4, head_dim=8, inter=128, rope_base=10000.0)


def _tiny_model(n_layers=2, L=3, V=11, seed=21):
    layers, caches = [], []
    for li in range(n_layers):
        _, wts, cache, _ = _mini_setup(shape=TINY_MODEL, B=1, L=L, seed=seed + li)
        layers.append(wts)
        caches.append(cache)
    g = np.random.default_rng(seed + 100)
    emb = g.normal(0, 1.0, (V, TINY_MODEL.hidden))
    lm = g.normal(0, 0.05, (V, TINY_MODEL.hidden))
    gamma = g.uniform(0.5, 1.5, TINY_MODEL.hidden)
    return layers, caches, emb, lm, gamma, np.array([4])


def test_model_step_two_layers_brute_force():
    """Embedding lookup, two blocks, final RMSNorm and LM head against explicit loops."""
    s, L = TINY_MODEL, 3
    layers, caches, emb, lm, gamma, tokens = _tiny_model(L=L)
    x = [float(v) for v in emb[tokens[0]]]
    for wts, cache in zip(layers, caches):         # before model_step writes the new entries
        x = _brute_block(s, wts, cache, x, L)
    rho = 1 / math.sqrt(sum(v * v for v in x) / s.hidden + s.rms_eps)
    z = [gamma[i] * rho * x[i] for i in range(s.hidden)]
    want = [sum(lm[v][k] * z[k] for k in range(s.hidden)) for v in range(lm.shape[0])]
    logits, res = oracle.model_step(s, layers, caches, emb, lm, gamma, tokens, np.array([L]))
    assert len(res) == 2
    np.testing.assert_allclose(logits[0], want, rtol=1e-10, atol=1e-12)


def test_model_step_final_gain_axis_and_lm_head_orientation():
    """A one-hot final gain keeps one channel of z; a single nonzero W_lm[v, k]
    moves exactly logit v by W_lm[v, k] z[k]; teacher-forced inputs are used as given."""
    s, L = TINY_MODEL, 3
    layers, caches, emb, lm, gamma, tokens = _tiny_model(n_layers=1, L=L)
    xf = np.random.default_rng(3).standard_normal((1, s.hidden)) * 3
    rho = 1 / math.sqrt(float(np.mean(xf[0] ** 2)) + s.rms_eps)
    g1 = np.zeros(s.hidden)
    g1[37] = 1.0
    logits, _ = oracle.model_step(s, layers, caches, emb, lm, g1, tokens, np.array([L]), final_input=xf)
    np.testing.assert_allclose(logits[0], lm[:, 37] * rho * xf[0, 37], rtol=1e-13, atol=1e-300)
    lm1 = np.zeros_like(lm)
    lm1[5, 37] = 0.5
    logits, _ = oracle.model_step(s, layers, caches, emb, lm1, gamma, tokens, np.array([L]), final_input=xf)
    assert np.count_nonzero(logits[0]) == 1
    np.testing.assert_allclose(logits[0, 5], 0.5 * gamma[37] * rho * xf[0, 37], rtol=1e-13)
    xin = np.random.default_rng(8).standard_normal((1, s.hidden))
    _, res = oracle.model_step(s, layers, caches, emb, lm, gamma, tokens, np.array([L]), layer_inputs=[xin])
    np.testing.assert_allclose(res[0]["h1"] - res[0]["attn_delta"], xin, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(res[0]["rho1"], rms_factor(xin, s.rms_eps))


def test_kv_cache_append_ragged_places_each_token_and_matches_dense():
    """Ragged placement: packed token i of request b (cu_seqlens[b] <= i < cu_seqlens[b+1])
    lands at [b, head, pos[b] + i - cu_seqlens[b]]; zero-length requests write nothing;
    with equal lengths it is the dense append."""
    nkv, d, cap = 2, 8, 20
    lens = np.array([3, 0, 5, 1])
    cu = np.concatenate([[0], np.cumsum(lens)])
    pos = np.array([2, 7, 0, 19])
    B, total = len(lens), int(cu[-1])
    g = np.random.default_rng(9)
    pat = g.standard_normal(d)
    k = np.empty((total, nkv, d))
    v = np.empty((total, nkv, d))
    for i in range(total):
        for h in range(nkv):
            amp = 1.0 + 10 * i + h                     # a different scale for every row
            k[i, h] = amp * pat
            v[i, h] = -amp * pat[::-1]
    c = KVCacheOracle(B, nkv, cap, d, d, d)
    c.append_ragged(k, v, cu, pos)
    seen = np.zeros((B, nkv, cap), bool)
    for b in range(B):
        for t in range(lens[b]):
            for h in range(nkv):
                p = pos[b] + t
                row = cu[b] + t
                for cache_c, cache_s, vals in ((c.kc, c.ks, k[row, h]), (c.vc, c.vs, v[row, h])):
                    codes, sc, _ = kv_quantize(vals, d, d)
                    np.testing.assert_array_equal(cache_c[b, h, p], codes)
                    np.testing.assert_array_equal(cache_s[b, h, p], sc)
                seen[b, h, p] = True
    assert seen.sum() == total * nkv
    assert np.all(c.kc[~seen] == 8) and np.all(c.ks[~seen] == 0)
    # equal lengths: the same cache as the dense append of [B, T, n_kv, d]
    T = 4
    kd = g.standard_normal((3, T, nkv, d))
    vd = g.standard_normal((3, T, nkv, d))
    p3 = np.array([0, 6, 11])
    a = KVCacheOracle(3, nkv, cap, d, d, d)
    a.append(kd, vd, p3)
    r = KVCacheOracle(3, nkv, cap, d, d, d)
    r.append_ragged(kd.reshape(3 * T, nkv, d), vd.reshape(3 * T, nkv, d), np.arange(4) * T, p3)
    for x, y in ((a.kc, r.kc), (a.vc, r.vc), (a.ks, r.ks), (a.vs, r.vs)):
        np.testing.assert_array_equal(x, y)


# ---------------------------------------------------------------- E4M3 decode weights
def test_e4m3_decode_hand_values_and_all_codes_against_torch():
    """The codec against the format's definition: hand values, then all 256 codes
    against torch's float8_e4m3fn (a library decoding of the same format)."""
    from oracle.fp8 import e4m3_decode
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3F: 1.875,
            0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in hand.items():
        assert e4m3_decode(c) == v, hex(c)
    assert np.isnan(e4m3_decode(0x7F)) and np.isnan(e4m3_decode(0xFF))
    assert np.signbit(e4m3_decode(0x80)) and e4m3_decode(0x80) == 0.0
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode(np.arange(256))
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_encode_round_trip_ties_saturation_and_torch():
    from oracle.fp8 import e4m3_decode, e4m3_encode
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    vals = e4m3_decode(codes)
    np.testing.assert_array_equal(e4m3_encode(vals), codes)             # every finite code, +-0 included
    pos = e4m3_decode(np.arange(0x7F))
    mid = (pos[:-1] + pos[1:]) / 2                                       # exact midpoints (FP64)
    want = np.where(np.arange(1, 0x7F) % 2 == 0, np.arange(1, 0x7F), np.arange(0x7E))
    np.testing.assert_array_equal(e4m3_encode(mid), want)                # ties go to the even code
    np.testing.assert_array_equal(e4m3_encode(-mid), want | 0x80)
    assert e4m3_encode(449.0) == 0x7E and e4m3_encode(1e9) == 0x7E and e4m3_encode(-1e9) == 0xFE
    assert e4m3_encode(-1e-30) == 0x80 and e4m3_encode(1e-30) == 0x00
    g = np.random.default_rng(3)
    x = (g.standard_normal(20000) * np.exp(g.uniform(-12, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(e4m3_encode(x.astype(np.float64)), ref)


def test_e4m3_weight_quantiser_and_product():
    """Per (row, 128 inputs): the group's largest magnitude decodes to +-448 s, every
    weight to within half an E4M3 step, zero groups to zero; the product applies the
    group scale after each group's sum (against brute force)."""
    from oracle.fp8 import e4m3_decode, quantize_weight_e4m3, e4m3_matvec
    g = np.random.default_rng(11)
    w = (g.standard_normal((6, 384)) * 0.02).astype(np.float32)
    w[2, 128:256] = 0.0
    gamma = g.uniform(0.5, 1.5, 384).astype(np.float32)
    codes, s = quantize_weight_e4m3(w, gamma)
    wf = (w * gamma).astype(np.float32).astype(np.float64)
    deq = e4m3_decode(codes).reshape(6, 3, 128) * s[..., None]
    assert s[2, 1] == 0 and np.all(codes[2, 128:256] == 0)
    amax_at = np.argmax(np.abs(wf.reshape(6, 3, 128)), axis=-1)
    for o in range(6):
        for k in range(3):
            if s[o, k] == 0:
                continue
            c = codes[o, 128 * k + amax_at[o, k]]
            assert e4m3_decode(c & 0x7F) == 448.0
    err = np.abs(deq.reshape(6, 384) - wf)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, np.repeat(s, 128, axis=1) * 2.0 ** -10) * (1 + 2 ** -7)
    assert np.all(err <= bound + 1e-30)
    x = g.standard_normal((3, 384))
    y = e4m3_matvec(codes, s, x)
    brute = np.zeros((3, 6))
    for b in range(3):
        for o in range(6):
            for k in range(3):
                part = sum(float(e4m3_decode(codes[o, 128 * k + i])) * x[b, 128 * k + i] for i in range(128))
                brute[b, o] += float(s[o, k]) * part
    np.testing.assert_allclose(y, brute, rtol=1e-12, atol=1e-12)
