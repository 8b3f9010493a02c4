"""Shared set-up for GPU parity tests: build one decode-block problem from the
seeded inputs, run it through the C ABI, and run the CPU oracle on the same
inputs.  Nothing here computes the method: the GPU side calls the library and
the reference side calls oracle/."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import oracle
import synth
import int4_weight_kv_gb300 as ft
from int4_weight_kv_gb300 import runtime as rt
from oracle.block import BlockWeightsOracle, decode_block
from oracle.kv import KVCacheOracle


@dataclasses.dataclass
class Layer:
    shape: synth.BlockShape
    cfg: ft.BlockCfg
    w32: dict            # FP32 host weights (synth layout)
    packed: dict         # device packed roles
    wts: Optional[BlockWeightsOracle] = None

    def oracle_weights(self) -> BlockWeightsOracle:
        if self.wts is None:
            fmt = "e4m3" if self.cfg.weight_format == ft.FT_WFMT_E4M3 else "int4"
            self.wts = BlockWeightsOracle(self.shape, self.w32, fmt)
        return self.wts


def make_layer(shape: synth.BlockShape, config_id: int, layer: int = 0, weight_format: int = 0) -> Layer:
    cfg = ft.cfg_from_shape(shape)
    cfg.weight_format = weight_format
    w = synth.layer_weights(shape, config_id, layer)
    packed = rt.pack_layer(cfg, w)
    torch.cuda.synchronize()
    return Layer(shape, cfg, w, packed)


@dataclasses.dataclass
class Problem:
    layer: Layer
    B: int
    max_ctx: int
    pos: np.ndarray
    x_bits: np.ndarray
    x_f32: np.ndarray
    k_bits: np.ndarray
    v_bits: np.ndarray
    cache: torch.Tensor
    status: torch.Tensor


def make_problem(layer: Layer, config_id: int, B: int, ctx: int, pos: Optional[np.ndarray] = None,
                 max_ctx: Optional[int] = None) -> Problem:
    s = layer.shape
    pos = np.full(B, ctx, np.int32) if pos is None else np.asarray(pos, np.int32)
    hist = int(pos.max())
    max_ctx = max_ctx or hist + 1
    x_bits, x_f32 = synth.activations(s, config_id, B)
    kb, _ = synth.kv_history(s, config_id, B, max(hist, 1), which="k")
    vb, _ = synth.kv_history(s, config_id, B, max(hist, 1), which="v")
    cache = rt.alloc_cache(layer.cfg, B, max_ctx)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if hist > 0:
        rt.fill_history(layer.cfg, cache, B, max_ctx, kb[:, :hist], vb[:, :hist], status)
    torch.cuda.synchronize()
    return Problem(layer, B, max_ctx, pos, x_bits, x_f32, kb[:, :hist], vb[:, :hist], cache, status)


@dataclasses.dataclass
class GpuResult:
    out: np.ndarray          # FP32 [B, H] (or BF16 values widened)
    qkv: np.ndarray
    o: np.ndarray
    h1: np.ndarray
    a: np.ndarray
    status: int
    cache: torch.Tensor


def run_gpu(pb: Problem, act_dtype=ft.FT_F32, cache: Optional[torch.Tensor] = None) -> GpuResult:
    L = pb.layer
    s = L.shape
    cache = pb.cache.clone() if cache is None else cache
    pos = torch.from_numpy(pb.pos).cuda()
    if act_dtype == ft.FT_F32:
        x = torch.from_numpy(pb.x_f32).cuda()
        y = torch.empty_like(x)
    else:
        x = rt.bits_tensor(pb.x_bits)
        y = torch.empty_like(x)
    ws = rt.alloc_workspace(L.cfg, pb.B, pb.max_ctx)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ft.check(ft.ft_decode_block(L.cfg, L.packed, cache, pb.B, pb.max_ctx, x, y, act_dtype, pos, pb.B, ws, st),
             "ft_decode_block")
    torch.cuda.synchronize()
    lay = ft.ft_decode_workspace_layout(L.cfg, pb.B, pb.max_ctx)
    B, H = pb.B, s.hidden

    def view(off, n, dt):
        nbytes = n * torch.tensor([], dtype=dt).element_size()
        return ws[off:off + nbytes].view(dt).cpu().numpy()
    rho1 = view(lay.rho1, B, torch.float32)
    qkv = view(lay.qkv, B * s.n_qkv, torch.float32).reshape(B, s.n_qkv) * rho1[:, None]
    o = operand_decode(view(lay.o, B * s.n_q * s.head_dim, torch.float16), B)
    h1 = view(lay.h1, B * H, torch.float32).reshape(B, H)
    a = operand_decode(view(lay.a, B * s.inter, torch.float16), B)
    if act_dtype == ft.FT_F32:
        out = y.cpu().numpy()
    else:
        out = synth.bf16_bits_to_f32(y.cpu().numpy().view(np.uint16))
    return GpuResult(out, qkv, o, h1, a, int(st.item()), cache)


def operand_decode(x16: np.ndarray, B: int) -> np.ndarray:
    """Logical FP32 values [B, K] of B rows stored in the projections' grouped
    operand layout (include/ft.h: [K/64][B][64]; runs of 8 stored values
    permuted by XOR with row mod 8; within each 16 inputs the storage order is
    0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15 and inputs 8..15 hold value / 16)."""
    x = np.asarray(x16, np.float32).reshape(-1, B, 8, 8)           # [half group][row][stored run][8]
    runs = np.empty_like(x)
    for t in range(B):
        runs[:, t] = x[:, t, np.arange(8) ^ (t & 7)]                # logical run r sits at r ^ (t & 7)
    slots = runs.reshape(-1, B, 64).transpose(1, 0, 2).reshape(B, -1, 16)
    order = np.array([0, 1, 8, 9, 2, 3, 10, 11, 4, 5, 12, 13, 6, 7, 14, 15])
    out = np.empty_like(slots)
    out[..., order] = slots
    out[..., 8:] *= 16.0
    return out.reshape(B, -1)


def oracle_cache(pb: Problem) -> KVCacheOracle:
    s = pb.layer.shape
    c = KVCacheOracle(pb.B, s.n_kv, pb.max_ctx, s.head_dim, s.hb, s.kvg)
    hist = pb.k_bits.shape[1]
    if hist:
        c.append(synth.bf16_bits_to_f32(pb.k_bits), synth.bf16_bits_to_f32(pb.v_bits), np.zeros(pb.B, int))
    return c


def run_oracle(pb: Problem, rows=None) -> dict:
    s = pb.layer.shape
    return decode_block(s, pb.layer.oracle_weights(), oracle_cache(pb), pb.x_f32.astype(np.float64), pb.pos,
                        batch_idx=rows)


def rel_rms(y, ref) -> float:
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs_over_rms(y, ref) -> float:
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(y - ref)) / max(np.sqrt(np.mean(ref * ref)), 1e-300))


def assert_block_close(gpu: GpuResult, orc: dict, rows, tol_rms=5e-3, tol_max=2e-2) -> dict:
    """The block-output gates on `out` (rel RMS and max-abs over RMS); the sublayer deltas are gated at
    the same relative RMS."""
    rows = list(rows)
    out = gpu.out[rows]
    x = orc["h1"] - orc["attn_delta"]
    rep = {
        "out_rel_rms": rel_rms(out, orc["out"]),
        "out_max_over_rms": max_abs_over_rms(out, orc["out"]),
        "attn_delta_rel_rms": rel_rms(gpu.h1[rows] - x, orc["attn_delta"]),
        "mlp_delta_rel_rms": rel_rms(out - gpu.h1[rows], orc["mlp_delta"]),
        "qkv_rel_rms": rel_rms(gpu.qkv[rows], orc["qkv"]),
        "o_rel_rms": rel_rms(gpu.o[rows], orc["o"]),
    }
    assert gpu.status == 0, f"device status {gpu.status}"
    assert rep["out_rel_rms"] <= tol_rms, rep
    assert rep["out_max_over_rms"] <= tol_max, rep
    assert rep["attn_delta_rel_rms"] <= tol_rms, rep
    assert rep["mlp_delta_rel_rms"] <= tol_rms, rep
    return rep


def unpack_weights(layer: Layer, role: int):
    n, k = ft.ft_weight_shape(layer.cfg, role)
    codes = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    scales = torch.empty((n, k // 128), dtype=torch.int16, device="cuda")
    unpack = ft.ft_unpack_weights_e4m3 if layer.cfg.weight_format == ft.FT_WFMT_E4M3 else ft.ft_unpack_weights_int4
    ft.check(unpack(layer.cfg, role, layer.packed[rt.ROLE_NAMES[role]], codes, scales), "unpack weights")
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)


def unpack_cache(layer: Layer, cache, max_batch, max_ctx, B, length):
    s = layer.shape
    kc = torch.empty((B, s.n_kv, length, s.head_dim), dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty((B, s.n_kv, length, 1), dtype=torch.int16, device="cuda")
    vs = torch.empty_like(ks)
    ft.check(ft.ft_kv_unpack_int4(layer.cfg, cache, max_batch, max_ctx, B, length, kc, vc, ks, vs),
             "ft_kv_unpack_int4")
    torch.cuda.synchronize()
    return (kc.cpu().numpy(), vc.cpu().numpy(), synth.bf16_bits_to_f32(ks.cpu().numpy().view(np.uint16)),
            synth.bf16_bits_to_f32(vs.cpu().numpy().view(np.uint16)))


def compare_codes(gpu_codes, gpu_scales, x_ref, group):
    """Code parity against the oracle's quantisation of the FP32 values x_ref.

    Bit-exact, except: a code may differ by +-1 where the oracle's pre-rounding
    value t = x / s lies within 1e-3 of a rounding boundary (half-integer); a
    group's BF16 scale may differ by one BF16 step only where amax / 7 lies
    within 1e-3 (relative) of a BF16 rounding midpoint, and that group is then
    re-quantised with the GPU's scale and must match under the same +-1 rule.
    Returns (codes differing, scales differing)."""
    x32 = np.asarray(x_ref, np.float32)
    ref_codes, ref_scales = oracle.quantize_groups(x32, group)
    gpu_codes = np.asarray(gpu_codes).astype(np.int16).reshape(ref_codes.shape)
    gs = np.asarray(gpu_scales, np.float32).reshape(ref_scales.shape)
    xg = x32.reshape(x32.shape[:-1] + (-1, group))
    scale_diff = gs != ref_scales
    n_scale = int(scale_diff.sum())
    if n_scale:
        a = gs[scale_diff].view(np.int32).astype(np.int64)
        b = ref_scales[scale_diff].view(np.int32).astype(np.int64)
        assert np.all(np.abs(a - b) == 1 << 16), "scale differs by more than one BF16 step"
        q = (np.max(np.abs(xg[scale_diff]), axis=-1) / 7.0).astype(np.float64)
        lo = oracle.bf16_rne(q.astype(np.float32)).astype(np.float64)
        ulp = (np.abs(lo) * 2.0 ** -7)
        mid_dist = np.minimum(np.abs(q - (lo + ulp / 2)), np.abs(q - (lo - ulp / 2)))
        assert np.all(mid_dist <= 1e-3 * q), "scale differs away from a BF16 midpoint"
    # reference codes: the oracle's, or for groups with a differing scale the
    # oracle's re-quantisation with the GPU's scale
    s_used = np.where(scale_diff, gs, ref_scales).astype(np.float32)
    safe = np.where(s_used == 0, np.float32(1), s_used)
    t = (xg.astype(np.float64) / safe[..., None].astype(np.float64))
    re = np.clip(np.rint((xg / safe[..., None]).astype(np.float32)), -8, 7) + 8
    re = np.where((s_used == 0)[..., None], 8, re).reshape(ref_codes.shape).astype(np.int16)
    d = gpu_codes - re
    assert np.all(np.abs(d) <= 1), "code differs by more than 1"
    near = (np.abs(t - np.floor(t) - 0.5) < 1e-3).reshape(d.shape)
    unexplained = (d != 0) & ~near
    assert not np.any(unexplained), f"{int(unexplained.sum())} code mismatches away from a rounding boundary"
    return int((d != 0).sum()), n_scale
