"""The allocation-free decode-block entry point agrees with ft_decode_block.

Some callers cannot allocate device memory at the moment they run a decode
step: an allocation policy that forbids new device allocations after start-up,
a host that hands the library only its input and output buffers, or a loop that
must not pay for cudaMalloc and its implicit synchronisation.  For them
ft_decode_block_static_ws takes its scratch space from a fixed device array
inside the library.  These checks compare it with the workspace entry point on
two calls in a row, and check that a problem too large for the array is
refused before anything runs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import int4_weight_kv_gb300 as ft
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_weight_kv_gb300 import build
    build.build()


STATIC_BYTES = 48 << 20  # the library's fixed scratch array


def _run_static(pb, cache):
    L = pb.layer
    x = torch.from_numpy(pb.x_f32).cuda()
    y = torch.empty_like(x)
    pos = torch.from_numpy(pb.pos).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ft.check(ft.ft_decode_block_static_ws(L.cfg, L.packed, cache, pb.B, pb.max_ctx, x, y, ft.FT_F32, pos, pb.B, st),
             "ft_decode_block_static_ws")
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("shape,cid,B,ctx", [(synth.TINY, 1, 3, 70), (synth.L8B, 2, 2, 300),
                                             (synth.L8B, 2, 32, 300)])
def test_static_workspace_matches_workspace_entry_point(shape, cid, B, ctx):
    layer = H.make_layer(shape, cid)
    pos = synth.positions(B, ctx, ragged=True, seed=7)
    pb = H.make_problem(layer, cid, B=B, ctx=ctx, pos=pos)
    ref = H.run_gpu(pb, ft.FT_F32)  # same problem through the caller-workspace entry point
    assert ref.status == 0
    n_hist = int(pb.pos.max()) + 1
    ref_cache = H.unpack_cache(layer, ref.cache, pb.B, pb.max_ctx, pb.B, n_hist)
    for _ in range(2):  # two calls in a row share the static array
        cache = pb.cache.clone()
        out, status = _run_static(pb, cache)
        assert status == 0
        # the block's parity tolerances ...
        assert H.rel_rms(out, ref.out) <= 5e-3
        assert H.max_abs_over_rms(out, ref.out) <= 2e-2
        # ... and, since both entry points run the same deterministic kernels
        # (no order-dependent floating-point reduction), the same bits
        np.testing.assert_array_equal(out, ref.out)
        # the new token's INT4 cache entry is written identically
        for a, b in zip(H.unpack_cache(layer, cache, pb.B, pb.max_ctx, pb.B, n_hist), ref_cache):
            np.testing.assert_array_equal(a, b)


def test_static_workspace_refuses_oversized_problem():
    cfg = ft.make_cfg(32768, 256, 32, 128, 131072)
    assert ft.ft_validate_cfg(cfg) == ft.FT_OK
    assert ft.ft_decode_workspace_bytes(cfg, 32, 4097) > STATIC_BYTES
    lw = ft.LayerWeights(16, 16, 16, 16)
    rc = ft.lib().ft_decode_block_static_ws(ctypes.byref(cfg), ctypes.byref(lw), 4096, 32, 4097, 8192, 1 << 24,
                                            ft.FT_BF16, 256, 32, None, None)
    assert rc == ft.FT_ERR_WORKSPACE
