"""The C-ABI library loads, exports every symbol include/ft.h declares, and its
host-side size queries and argument checks behave (no GPU needed: every call
here returns before touching the device)."""
import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ft():
    from int4_weight_kv_gb300 import build as b
    b.build()
    import int4_weight_kv_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "ft.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ft_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(ft):
    names = _declared()
    assert len(names) >= 15
    so = ctypes.CDLL(ft.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(ft.exported_symbols())


def test_status_strings(ft):
    for s in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(ft.ft_status_string(s), str) and ft.ft_status_string(s)


def _cfg8b(ft, **kw):
    c = dict(hidden=4096, n_q=32, n_kv=8, head_dim=128, inter=14336)
    c.update(kw)
    return ft.make_cfg(**c)


def test_cfg_validation(ft):
    assert ft.ft_validate_cfg(_cfg8b(ft)) == ft.FT_OK
    assert ft.ft_validate_cfg(ft.make_cfg(512, 8, 2, 64, 1408, rope_base=1e4)) == ft.FT_OK
    assert ft.ft_validate_cfg(_cfg8b(ft, n_q=30)) == ft.FT_ERR_INVALID_ARG          # n_q % n_kv
    assert ft.ft_validate_cfg(_cfg8b(ft, head_dim=96)) == ft.FT_ERR_UNSUPPORTED
    assert ft.ft_validate_cfg(_cfg8b(ft, had_block=48)) == ft.FT_ERR_INVALID_ARG    # not a power of two
    assert ft.ft_validate_cfg(_cfg8b(ft, hidden=4000)) == ft.FT_ERR_UNSUPPORTED
    assert ft.ft_validate_cfg(_cfg8b(ft, n_q=128, n_kv=8)) == ft.FT_ERR_UNSUPPORTED  # G > 8
    assert ft.ft_validate_cfg(_cfg8b(ft, w_group=64)) == ft.FT_ERR_UNSUPPORTED
    assert ft.ft_validate_cfg(_cfg8b(ft, had_block=1)) == ft.FT_OK                   # rotation off


def test_weight_shapes_and_packed_bytes(ft):
    c = _cfg8b(ft)
    shapes = {ft.FT_W_QKV: (6144, 4096), ft.FT_W_O: (4096, 4096), ft.FT_W_GATEUP: (28672, 4096),
              ft.FT_W_DOWN: (4096, 14336)}
    total = 0
    for role, (n, k) in shapes.items():
        assert ft.ft_weight_shape(c, role) == (n, k)
        nb = ft.ft_packed_weight_bytes(c, role)
        assert nb == n * k // 2 + n * k // 64        # nibbles + BF16 group-128 scales
        total += nb
    assert total == 112_459_776                      # 8B layer: codes + scales
    assert ft.ft_packed_weight_bytes(c, 9) == 0


def test_kv_and_workspace_sizes(ft):
    c = _cfg8b(ft)
    nb = ft.ft_kv_cache_bytes(c, 1, 1025)
    assert nb >= 1025 * 8 * (64 + 64 + 2 + 2)        # 1056 B per token per layer
    assert nb < 1025 * 8 * (64 + 64 + 2 + 2) + 4 * 256
    assert ft.ft_decode_workspace_bytes(c, 1, 1025) > 0
    assert ft.ft_decode_workspace_bytes(c, 33, 1025) == 0
    assert ft.ft_decode_workspace_bytes(c, 32, 4097) > ft.ft_decode_workspace_bytes(c, 1, 4097)
    lay = ft.ft_decode_workspace_layout(c, 4, 2048)
    assert lay.n_split >= 1 and len({lay.qkv, lay.rho1, lay.o, lay.h1, lay.a}) == 5


def test_argument_errors_return_before_launch(ft):
    c = _cfg8b(ft)
    lw = ft.LayerWeights(16, 16, 16, 16)
    lib = ft.lib()
    args = lambda **o: dict(dict(cache=4096, max_batch=4, max_ctx=64, x_in=8192, x_out=1 << 20, dt=ft.FT_BF16,
                                 pos=256, B=1, ws=1 << 24, wsb=1 << 30), **o)

    def call(**o):
        a = args(**o)
        return lib.ft_decode_block(ctypes.byref(c), ctypes.byref(lw), a["cache"], a["max_batch"], a["max_ctx"],
                                   a["x_in"], a["x_out"], a["dt"], a["pos"], a["B"], a["ws"], a["wsb"], None, None)
    assert call(B=33) == ft.FT_ERR_UNSUPPORTED
    assert call(B=5) == ft.FT_ERR_CAPACITY
    assert call(B=0) == ft.FT_ERR_INVALID_ARG
    assert call(cache=None) == ft.FT_ERR_INVALID_ARG
    assert call(x_in=8193) == ft.FT_ERR_INVALID_ARG           # misaligned
    assert call(x_out=8192 + 64) == ft.FT_ERR_INVALID_ARG     # overlaps x_in
    assert call(dt=7) == ft.FT_ERR_INVALID_ARG
    assert call(wsb=16) == ft.FT_ERR_WORKSPACE
    assert lib.ft_decode_block_stages(ctypes.byref(c), ctypes.byref(lw), 4096, 4, 64, 8192, 1 << 20, 0, 256, 1,
                                      1 << 24, 1 << 30, None, 0, None) == ft.FT_ERR_INVALID_ARG
    # pack / append / unpack argument checks
    assert lib.ft_pack_weights_int4(ctypes.byref(c), 0, None, None, 4096, 1 << 30, None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_pack_weights_int4(ctypes.byref(c), 0, 4096, None, 8192, 16, None) == ft.FT_ERR_WORKSPACE
    assert lib.ft_pack_weights_int4(ctypes.byref(c), 5, 4096, None, 8192, 1 << 30, None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_kv_append_int4(ctypes.byref(c), 4096, 2, 64, 16, 16, 16, 3, 1, None, None) == ft.FT_ERR_CAPACITY
    assert lib.ft_kv_append_int4(ctypes.byref(c), 4096, 2, 64, 16, 16, 16, 1, 65, None, None) == ft.FT_ERR_CAPACITY
    assert lib.ft_kv_append_int4(ctypes.byref(c), 4097, 2, 64, 16, 16, 16, 1, 1, None, None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_kv_unpack_int4(ctypes.byref(c), 4096, 2, 64, 3, 8, 16, 16, 16, 16, None) == ft.FT_ERR_INVALID_ARG
    assert ft.ft_decode_block_launches(c, 1) == 7 and ft.ft_decode_block_launches(c, 16) == 7
    assert ft.ft_decode_block_launches(c, 17) == 9 and ft.ft_decode_block_launches(c, 32) == 9
    assert ft.ft_decode_block_launches(c, 33) == 0
    # E4M3 decode weights: the tensor-core path at every batch; packs need the matching format
    e4 = ft.BlockCfg(*[getattr(c, f) for f, _ in ft.BlockCfg._fields_])
    e4.weight_format = ft.FT_WFMT_E4M3
    assert ft.ft_validate_cfg(e4) == ft.FT_OK
    assert ft.ft_decode_block_launches(e4, 1) == 7 and ft.ft_decode_block_launches(e4, 17) == 9
    assert ft.ft_packed_weight_bytes(e4, 0) == ft.ft_packed_weight_bytes(c, 0) * 2080 // 1056
    assert lib.ft_pack_weights_int4(ctypes.byref(e4), 0, 4096, None, 8192, 1 << 30, None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_pack_weights_e4m3(ctypes.byref(c), 0, 4096, None, 8192, 1 << 30, None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_pack_weights_e4m3(ctypes.byref(e4), 0, 4096, None, 8192, 16, None) == ft.FT_ERR_WORKSPACE
    bad = ft.BlockCfg(*[getattr(c, f) for f, _ in ft.BlockCfg._fields_])
    bad.weight_format = 7
    assert ft.ft_validate_cfg(bad) == ft.FT_ERR_INVALID_ARG
    # model-step helpers
    assert lib.ft_rmsnorm_bf16(None, 4096, 8192, 1, 64, ctypes.c_float(1e-5), None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_rmsnorm_bf16(4096, 4096, 8192, 0, 64, ctypes.c_float(1e-5), None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_rmsnorm_bf16(4096, 4096, 8192, 1, 64, ctypes.c_float(-1.0), None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_read_device_status(None, 4096, None) == ft.FT_ERR_INVALID_ARG
    prev = ft.ft_set_pdl(False)
    assert ft.ft_set_pdl(prev) is False


def test_plan_partitions(ft):
    """Host-side partition choices (no GPU needed): whole vs split sets, the
    tensor-core kernel for batches of 17-32, shared memory within one SM."""
    c8 = ft.cfg_from_shape(synth.workload("8b_b1_ctx1024").shape)
    c70 = ft.cfg_from_shape(synth.workload("70b_b1_ctx2048").shape)
    info = lambda c, B, role: ft.ft_decode_plan_info(c, B, 4097, role)
    for c in (c8, c70):
        for B in (1, 2, 8, 9, 16, 17, 32):
            for role in ft.ROLES:
                g = info(c, B, role)
                tc = B > 16
                assert g.tensor_core == (1 if tc else 0)
                assert g.col_tiles == (4 if tc else (B + 7) // 8)   # the tensor-core kernel always takes N = 32
                assert 2 <= g.stages <= 8 and 1 <= g.groups_per_stage
                assert 0 < g.smem_bytes <= 227 * 1024
                assert 1 <= g.ctas <= 148
                if tc:
                    assert g.row_tiles == 8                # one M = 128 tensor-core tile per set
                    assert g.whole == 0                    # units spread evenly, every piece to a slab
                elif role == ft.FT_W_GATEUP:
                    assert g.whole == 1                    # SwiGLU in the epilogue needs whole rows
                if role in (ft.FT_W_QKV, ft.FT_W_O):
                    assert g.whole == 0                    # split along K, one slab per piece
    # down: whole two-tile sets balance for the 8B shape, not for 70B (long K)
    assert info(c8, 1, ft.FT_W_DOWN).whole == 1 and info(c8, 1, ft.FT_W_DOWN).row_tiles == 2
    assert info(c70, 1, ft.FT_W_DOWN).whole == 0
    with pytest.raises(RuntimeError):
        info(c8, 33, ft.FT_W_QKV)


def test_ragged_append_argument_checks(ft):
    """Host-side checks of the ragged placement, before anything is enqueued."""
    cfg = ft.cfg_from_shape(synth.TINY)
    lib = ft.lib()
    fake = 4096  # never dereferenced: every call below returns before a launch
    call = lambda cache, mb, mc, k, cu, pos, B, total: lib.ft_kv_append_ragged_int4(
        ctypes.byref(cfg), cache, mb, mc, k, k, cu, pos, B, total, None, None)
    assert call(fake, 4, 16, fake, fake, fake, 5, 10) == ft.FT_ERR_CAPACITY       # B > max_batch
    assert call(fake, 4, 16, fake, fake, fake, 2, -1) == ft.FT_ERR_INVALID_ARG    # negative total
    assert call(None, 4, 16, fake, fake, fake, 2, 10) == ft.FT_ERR_INVALID_ARG    # no cache
    assert call(fake, 4, 16, fake, None, fake, 2, 10) == ft.FT_ERR_INVALID_ARG    # no map
    assert call(fake, 4, 16, None, fake, fake, 2, 10) == ft.FT_ERR_INVALID_ARG    # no rows
    assert call(fake + 8, 4, 16, fake, fake, fake, 2, 10) == ft.FT_ERR_INVALID_ARG  # misaligned cache
    assert call(fake, 4, 16, None, fake, fake, 2, 0) == ft.FT_OK                  # nothing to place


@pytest.mark.parametrize("fmt", [0, 1])
def test_plans_fit_shared_memory_for_every_batch(ft, fmt):
    """Host plans for INT4 and E4M3 weights at every batch 1..32 and the three shapes: every
    projection ring fits one SM's shared memory with at least two stages, and the partition
    covers every (row set, group) unit once (no launch could fail on its shared memory)."""
    for shape in (synth.TINY, synth.L8B, synth.L70B):
        cfg = ft.cfg_from_shape(shape)
        cfg.weight_format = fmt
        for B in range(1, 33):
            for role in ft.ROLES:
                g = ft.ft_decode_plan_info(cfg, B, 2049, role)
                assert 0 < g.smem_bytes <= 227 * 1024, (shape.hidden, B, role, g.smem_bytes)
                assert g.stages >= 2 and g.groups_per_stage >= 1
                assert g.tensor_core == (1 if B > 16 else 0)
            assert ft.ft_decode_block_launches(cfg, B) == (9 if B > 16 else 7)
