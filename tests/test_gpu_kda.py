"""GPU parity of the per-channel-decay (KDA) verify, native snapshot and
all-layer commit, through the C ABI, against the fp64 oracle's KDA
functions and against the GPU native kernel (bit for bit): the same checks
as the scalar-gate path (tests/test_gpu_parity.py)."""
import gc

import numpy as np
import pytest
import torch

from spec_decode_recurrent_gb300 import api, build, workloads as wl
from tests._parity import GpuStep, bits, compare_full, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


SMALL = {
    "ragged_fused": dict(HK=2, HV=4, K=128, V=128, W=6, L=2, windows=[6, 4, 1, 3, 0, 6, 2],
                         accepted=[3, 4, 1, 2, 0, 6, 1], null_rows=(5,),
                         gaps=[1, 0, 2, 3, 0, 1, 0], shuffle_rows=True, fused=True,
                         qkv_dtype=wl.BF16),
    "extreme_gates": dict(HK=1, HV=2, K=128, V=128, W=6, L=1, windows=[6, 6, 5, 1],
                          accepted=[6, 3, 5, 1], gate_range=20.0, qkv_dtype=wl.BF16),
    "bf16_state": dict(HK=2, HV=4, K=128, V=128, W=4, L=2, windows=[4, 4, 2, 0],
                       accepted=[4, 1, 2, 0], qkv_dtype=wl.BF16, state_dtype=wl.BF16),
    "align_fp32": dict(HK=2, HV=4, K=128, V=128, W=4, L=2, windows=[4] * 8,
                       accepted=[1, 2, 3, 4, 4, 4, 2, 3], block_size=4,
                       seq_pos=[4, 5, 6, 7, 8, 9, 10, 11]),
    "align_bf16_state": dict(HK=1, HV=2, K=128, V=128, W=4, L=1, windows=[4] * 6,
                             accepted=[4, 3, 2, 1, 4, 3], block_size=4,
                             seq_pos=[4, 5, 6, 7, 9, 11], state_dtype=wl.BF16),
    "gqa4_k64_v32": dict(HK=1, HV=4, K=64, V=32, W=5, L=2, windows=[5, 3, 5], accepted=[2, 3, 5]),
    "k32_v64_two_tiles": dict(HK=1, HV=2, K=32, V=128, W=3, L=1, windows=[3, 2], accepted=[1, 2]),
    "k16_v16": dict(HK=2, HV=2, K=16, V=16, W=4, L=1, windows=[4, 4], accepted=[1, 3]),
    "max_window16": dict(HK=1, HV=2, K=128, V=128, W=16, L=1, windows=[16, 9], accepted=[16, 7]),
    # every window length under the unrolled 4-token build
    "w4_every_window": dict(HK=1, HV=2, K=128, V=128, W=4, L=1, windows=[1, 2, 3, 4],
                            accepted=[1, 2, 1, 3], qkv_dtype=wl.BF16),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_kda_small_step_full_oracle(name):
    sb = wl.custom(device="cuda", kda=True, **SMALL[name])
    gs = GpuStep(sb)
    assert gs.err == 0 and gs.verify_err == 0
    gs.check_bitwise()
    layers, pools, err = oracle_full(sb, gs.before)
    assert np.all(err == 0)
    compare_full(gs, layers, pools)


@pytest.mark.parametrize("state_dtype", [wl.F32, wl.BF16])
def test_kda_full_size_workload(state_dtype):
    # the benchmark's KDA configuration (all_layer shapes, 36 layers)
    sb = wl.kda_all_layer(device="cuda", state_dtype=state_dtype)
    try:
        gs = GpuStep(sb, units=12, unit_seed=3)
        assert gs.err == 0 and gs.verify_err == 0
        gs.check_bitwise()
        for l, r, h in gs.unit_list:
            gs.check_unit_against_oracle(l, r, h)
    finally:
        del sb
        gc.collect()
        torch.cuda.empty_cache()


def test_kda_uniform_channels_match_scalar_gate_kernels_bitwise():
    # Every channel carrying the scalar gate's input: the KDA kernels give
    # the scalar-gate kernels' outputs, records and committed states exactly
    # (the same fp32 operations on the same values).
    kw = dict(HK=1, HV=2, K=128, V=128, W=4, L=2, windows=[4, 3, 4], accepted=[2, 3, 4],
              qkv_dtype=wl.BF16)
    scal = wl.custom(device="cuda", **kw)
    kda = wl.custom(device="cuda", kda=True, **kw)
    for l in range(kda.L):
        kda.a[l] = scal.a[l][:, :, None].expand(-1, -1, kda.K).contiguous()
        kda.dt_bias[l] = scal.dt_bias[l][:, None].expand(-1, kda.K).contiguous()
        kda.q[l], kda.k[l], kda.v[l], kda.b[l] = scal.q[l], scal.k[l], scal.v[l], scal.b[l]
        kda.A_log[l] = scal.A_log[l]
        kda.pools[l].copy_(scal.pools[l])
    gs_s, gs_k = GpuStep(scal), GpuStep(kda)
    for l in range(kda.L):
        assert torch.equal(bits(gs_s.bufs.out[l]), bits(gs_k.bufs.out[l]))
        assert torch.equal(bits(gs_s.bufs.rec_u[l]), bits(gs_k.bufs.rec_u[l]))
        g = gs_s.bufs.rec_g[l][..., None].expand(-1, -1, -1, kda.K)
        assert torch.equal(bits(g.contiguous()), bits(gs_k.bufs.rec_g[l]))
        assert torch.equal(bits(scal.pools[l]), bits(kda.pools[l]))


def test_kda_commit_skips_rows_the_verify_rejected():
    sb = wl.custom(device="cuda", kda=True, HK=1, HV=2, K=128, V=128, W=4, L=1,
                   windows=[4, 3, 4], accepted=[2, 3, 4], qkv_dtype=wl.BF16)
    sb.token_start[1] = sb.T - 2
    gs = GpuStep(sb, native=False)
    assert gs.verify_err == api.ROW_ERR_TOKENS
    assert gs.err == api.ROW_ERR_TOKENS | api.ROW_ERR_REJECTED
    bad = int(sb.slot_table[1, 0])
    assert torch.equal(bits(sb.pools[0][bad]), bits(gs.before[0][bad]))
    assert torch.equal(gs.bufs.rec_g[0][1, :, 0, 0].cpu(), torch.full((sb.HV,), -1.0))


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("qkv_dtype", [wl.F32, wl.BF16])
def test_value_and_gate_rows_off_the_16_byte_grid(kda, qkv_dtype):
    # The library asks only element alignment of v (and 4 bytes of the KDA
    # gate inputs); the verify stages 16-byte pieces where rows allow it and
    # single elements elsewhere.  The same step with every value row and
    # gate input moved off the 16-byte grid must give the same bits.
    kw = dict(HK=1, HV=2, K=128, V=128, W=4, L=1, windows=[4, 3, 4], accepted=[2, 3, 4],
              qkv_dtype=qkv_dtype, kda=kda)
    ref = wl.custom(device="cuda", **kw)
    odd = wl.custom(device="cuda", **kw)
    T, HV, V = odd.v[0].shape
    buf = torch.empty((T, HV * V + 1), dtype=odd.v[0].dtype, device="cuda")
    v = buf[:, 1:].unflatten(1, (HV, V))      # odd row stride, base one element in
    v.copy_(odd.v[0])
    odd.v[0] = v
    assert v.stride(0) % 2 == 1
    if kda:
        def shifted(x):
            flat = torch.empty(x.numel() + 1, dtype=x.dtype, device="cuda")
            y = flat[1:].view(x.shape)        # 4 bytes off the 16-byte grid
            y.copy_(x)
            return y
        odd.a[0] = shifted(odd.a[0])
        odd.dt_bias[0] = shifted(odd.dt_bias[0])
        assert odd.a[0].data_ptr() % 16 != 0 and odd.dt_bias[0].data_ptr() % 16 != 0
    g_ref, g_odd = GpuStep(ref), GpuStep(odd)
    assert g_ref.err == 0 and g_odd.err == 0
    for name in ("out", "rec_u", "rec_k", "rec_g"):
        assert torch.equal(bits(getattr(g_ref.bufs, name)[0]), bits(getattr(g_odd.bufs, name)[0])), name
    assert torch.equal(bits(ref.pools[0]), bits(odd.pools[0]))
    g_odd.check_bitwise()
