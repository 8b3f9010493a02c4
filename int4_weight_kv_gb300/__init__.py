"""Python binding of the INT4-weight / Hadamard-rotated INT4-KV decode-block
library (``libft.so``, C ABI declared in ``include/ft.h``).

Argument marshalling only: every function here forwards to the C entry point of
the same name; all computation runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.  If the compiled library is missing the
calls raise instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_int, c_int32, c_size_t, c_uint, c_void_p, c_float, c_char_p, POINTER

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libft.so")

FT_OK, FT_ERR_INVALID_ARG, FT_ERR_UNSUPPORTED, FT_ERR_WORKSPACE, FT_ERR_CAPACITY, FT_ERR_CUDA = 0, -1, -2, -3, -4, -5
FT_DEV_CAPACITY, FT_DEV_TIMEOUT, FT_DEV_RANGE = 1, 2, 4
FT_BF16, FT_F32 = 0, 1
FT_WFMT_INT4, FT_WFMT_E4M3 = 0, 1
FT_W_QKV, FT_W_O, FT_W_GATEUP, FT_W_DOWN = 0, 1, 2, 3
FT_STAGE_PREP, FT_STAGE_QKV, FT_STAGE_ATTN, FT_STAGE_O = 1, 2, 4, 8
FT_STAGE_MID, FT_STAGE_GU, FT_STAGE_DOWN, FT_STAGE_ALL = 16, 32, 64, 127
ROLES = (FT_W_QKV, FT_W_O, FT_W_GATEUP, FT_W_DOWN)


class BlockCfg(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("n_q", c_int32), ("n_kv", c_int32), ("head_dim", c_int32),
                ("inter", c_int32), ("w_group", c_int32), ("had_block", c_int32), ("kv_group", c_int32),
                ("rms_eps", c_float), ("rope_base", c_float), ("weight_format", c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("qkv", c_void_p), ("o", c_void_p), ("gateup", c_void_p), ("down", c_void_p)]


class GemvInfo(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("ctas", "row_tiles", "warps", "col_tiles", "whole", "tensor_core", "stages",
                                       "groups_per_stage", "smem_bytes")]


class WsLayout(ctypes.Structure):
    _fields_ = [("qkv", c_size_t), ("rho1", c_size_t), ("o", c_size_t), ("h1", c_size_t), ("a", c_size_t),
                ("n_split", c_int32)]


class FTError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {ft_status_string(status)} ({status})")


_lib = None

# name -> (restype, argtypes)
_SIGS = {
    "ft_status_string": (c_char_p, [c_int]),
    "ft_validate_cfg": (c_int, [POINTER(BlockCfg)]),
    "ft_weight_shape": (c_int, [POINTER(BlockCfg), c_int, POINTER(c_int32), POINTER(c_int32)]),
    "ft_packed_weight_bytes": (c_size_t, [POINTER(BlockCfg), c_int]),
    "ft_pack_weights_int4": (c_int, [POINTER(BlockCfg), c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "ft_unpack_weights_int4": (c_int, [POINTER(BlockCfg), c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "ft_pack_weights_e4m3": (c_int, [POINTER(BlockCfg), c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "ft_unpack_weights_e4m3": (c_int, [POINTER(BlockCfg), c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "ft_kv_cache_bytes": (c_size_t, [POINTER(BlockCfg), c_int, c_int]),
    "ft_kv_append_int4": (c_int, [POINTER(BlockCfg), c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                  c_int, c_int, c_void_p, c_void_p]),
    "ft_kv_append_ragged_int4": (c_int, [POINTER(BlockCfg), c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_int, c_int, c_void_p, c_void_p]),
    "ft_kv_unpack_int4": (c_int, [POINTER(BlockCfg), c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p]),
    "ft_decode_workspace_bytes": (c_size_t, [POINTER(BlockCfg), c_int, c_int]),
    "ft_decode_block": (c_int, [POINTER(BlockCfg), POINTER(LayerWeights), c_void_p, c_int, c_int, c_void_p,
                                c_void_p, c_int, c_void_p, c_int, c_void_p, c_size_t, c_void_p, c_void_p]),
    "ft_decode_block_stages": (c_int, [POINTER(BlockCfg), POINTER(LayerWeights), c_void_p, c_int, c_int, c_void_p,
                                       c_void_p, c_int, c_void_p, c_int, c_void_p, c_size_t, c_void_p, c_uint,
                                       c_void_p]),
    "ft_decode_workspace_layout": (c_int, [POINTER(BlockCfg), c_int, c_int, POINTER(WsLayout)]),
    "ft_decode_block_static_ws": (c_int, [POINTER(BlockCfg), POINTER(LayerWeights), c_void_p, c_int, c_int,
                                          c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p]),
    "ft_embed_bf16": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "ft_lm_head_bf16": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_float, c_void_p]),
    "ft_rmsnorm_bf16": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_float, c_void_p]),
    "ft_read_device_status": (c_int, [c_void_p, c_void_p, c_void_p]),
    "ft_decode_plan_info": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p]),
    "ft_decode_block_launches": (c_int, [POINTER(BlockCfg), c_int]),
    "ft_set_pdl": (c_int, [c_int]),
}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run int4_weight_kv_gb300.build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_cfg(hidden, n_q, n_kv, head_dim, inter, had_block=0, kv_group=0, rms_eps=1e-5, rope_base=500000.0,
             w_group=128, weight_format=0) -> BlockCfg:
    hb = had_block or head_dim
    return BlockCfg(hidden, n_q, n_kv, head_dim, inter, w_group, hb, kv_group or head_dim, rms_eps, rope_base,
                    weight_format)


def cfg_from_shape(shape) -> BlockCfg:
    """BlockCfg from any object with the BlockShape attribute names."""
    return make_cfg(shape.hidden, shape.n_q, shape.n_kv, shape.head_dim, shape.inter,
                    getattr(shape, "had_block", 0), getattr(shape, "kv_group", 0),
                    shape.rms_eps, shape.rope_base, weight_format=getattr(shape, "weight_format", 0))


def check(status: int, what: str = "ft") -> None:
    if status != FT_OK:
        raise FTError(status, what)


# ---------------------------------------------------------------- the C ABI, same names
def ft_status_string(status: int) -> str:
    return lib().ft_status_string(status).decode()


def ft_validate_cfg(cfg: BlockCfg) -> int:
    return lib().ft_validate_cfg(ctypes.byref(cfg))


def ft_weight_shape(cfg: BlockCfg, role: int) -> tuple[int, int]:
    n, k = c_int32(), c_int32()
    check(lib().ft_weight_shape(ctypes.byref(cfg), role, ctypes.byref(n), ctypes.byref(k)), "ft_weight_shape")
    return n.value, k.value


def ft_packed_weight_bytes(cfg: BlockCfg, role: int) -> int:
    return lib().ft_packed_weight_bytes(ctypes.byref(cfg), role)


def ft_pack_weights_int4(cfg, role, W, gamma, packed, stream=None) -> int:
    return lib().ft_pack_weights_int4(ctypes.byref(cfg), role, _ptr(W), _ptr(gamma), _ptr(packed),
                                      packed.numel() * packed.element_size(), _stream(stream))


def ft_unpack_weights_int4(cfg, role, packed, codes, scales, stream=None) -> int:
    return lib().ft_unpack_weights_int4(ctypes.byref(cfg), role, _ptr(packed), _ptr(codes), _ptr(scales),
                                        _stream(stream))


def ft_pack_weights_e4m3(cfg, role, W, gamma, packed, stream=None) -> int:
    return lib().ft_pack_weights_e4m3(ctypes.byref(cfg), role, _ptr(W), _ptr(gamma), _ptr(packed),
                                      packed.numel() * packed.element_size(), _stream(stream))


def ft_unpack_weights_e4m3(cfg, role, packed, codes, scales, stream=None) -> int:
    return lib().ft_unpack_weights_e4m3(ctypes.byref(cfg), role, _ptr(packed), _ptr(codes), _ptr(scales),
                                        _stream(stream))


def ft_kv_cache_bytes(cfg, max_batch: int, max_ctx: int) -> int:
    return lib().ft_kv_cache_bytes(ctypes.byref(cfg), max_batch, max_ctx)


def ft_kv_append_int4(cfg, cache, max_batch, max_ctx, k_bits, v_bits, pos, B, T, dev_status=None,
                      stream=None) -> int:
    return lib().ft_kv_append_int4(ctypes.byref(cfg), _ptr(cache), max_batch, max_ctx, _ptr(k_bits), _ptr(v_bits),
                                   _ptr(pos), B, T, _ptr(dev_status), _stream(stream))


def ft_kv_append_ragged_int4(cfg, cache, max_batch, max_ctx, k_bits, v_bits, cu_seqlens, pos, B, total,
                             dev_status=None, stream=None) -> int:
    return lib().ft_kv_append_ragged_int4(ctypes.byref(cfg), _ptr(cache), max_batch, max_ctx, _ptr(k_bits),
                                          _ptr(v_bits), _ptr(cu_seqlens), _ptr(pos), B, total, _ptr(dev_status),
                                          _stream(stream))


def ft_kv_unpack_int4(cfg, cache, max_batch, max_ctx, B, length, k_codes, v_codes, k_scales, v_scales,
                      stream=None) -> int:
    return lib().ft_kv_unpack_int4(ctypes.byref(cfg), _ptr(cache), max_batch, max_ctx, B, length, _ptr(k_codes),
                                   _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _stream(stream))


def ft_decode_workspace_bytes(cfg, B: int, max_ctx: int) -> int:
    return lib().ft_decode_workspace_bytes(ctypes.byref(cfg), B, max_ctx)


def ft_decode_workspace_layout(cfg, B: int, max_ctx: int) -> WsLayout:
    out = WsLayout()
    check(lib().ft_decode_workspace_layout(ctypes.byref(cfg), B, max_ctx, ctypes.byref(out)),
          "ft_decode_workspace_layout")
    return out


def _layer(w) -> LayerWeights:
    if isinstance(w, LayerWeights):
        return w
    return LayerWeights(_ptr(w["qkv"]), _ptr(w["o"]), _ptr(w["gateup"]), _ptr(w["down"]))


def ft_decode_block(cfg, weights, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B, workspace,
                    dev_status=None, stream=None) -> int:
    lw = _layer(weights)
    return lib().ft_decode_block(ctypes.byref(cfg), ctypes.byref(lw), _ptr(cache), max_batch, max_ctx, _ptr(x_in),
                                 _ptr(x_out), act_dtype, _ptr(pos), B, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))


def ft_decode_block_stages(cfg, weights, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B, workspace,
                           stage_mask, dev_status=None, stream=None) -> int:
    lw = _layer(weights)
    return lib().ft_decode_block_stages(ctypes.byref(cfg), ctypes.byref(lw), _ptr(cache), max_batch, max_ctx,
                                        _ptr(x_in), _ptr(x_out), act_dtype, _ptr(pos), B, _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                        stage_mask, _stream(stream))


def ft_decode_block_static_ws(cfg, weights, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B,
                              dev_status=None, stream=None) -> int:
    """ft_decode_block with the library's fixed device scratch instead of a workspace."""
    lw = _layer(weights)
    return lib().ft_decode_block_static_ws(ctypes.byref(cfg), ctypes.byref(lw), _ptr(cache), max_batch, max_ctx,
                                           _ptr(x_in), _ptr(x_out), act_dtype, _ptr(pos), B, _ptr(dev_status),
                                           _stream(stream))


def ft_embed_bf16(table, tokens, x_out, B, V, H, dev_status=None, stream=None) -> int:
    return lib().ft_embed_bf16(_ptr(table), _ptr(tokens), _ptr(x_out), B, V, H, _ptr(dev_status), _stream(stream))


def ft_lm_head_bf16(x, gamma, W, logits, B, V, H, eps, stream=None) -> int:
    return lib().ft_lm_head_bf16(_ptr(x), _ptr(gamma), _ptr(W), _ptr(logits), B, V, H, eps, _stream(stream))


def ft_rmsnorm_bf16(x, gamma, z, B, H, eps, stream=None) -> int:
    return lib().ft_rmsnorm_bf16(_ptr(x), _ptr(gamma), _ptr(z), B, H, eps, _stream(stream))


def ft_read_device_status(dev_status, stream=None) -> int:
    """Waits for `stream` and returns the device status word (raises on a CUDA error)."""
    out = ctypes.c_int32(0)
    check(lib().ft_read_device_status(_ptr(dev_status), ctypes.byref(out), _stream(stream)), "ft_read_device_status")
    return int(out.value)


def ft_decode_plan_info(cfg, B: int, max_ctx: int, role: int) -> GemvInfo:
    out = GemvInfo()
    check(lib().ft_decode_plan_info(ctypes.byref(cfg), int(B), int(max_ctx), int(role), ctypes.byref(out)),
          "ft_decode_plan_info")
    return out


def ft_decode_block_launches(cfg, B: int = 1) -> int:
    return lib().ft_decode_block_launches(ctypes.byref(cfg), int(B))


def ft_set_pdl(enabled: bool) -> bool:
    return bool(lib().ft_set_pdl(1 if enabled else 0))
