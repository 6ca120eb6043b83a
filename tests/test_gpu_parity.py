"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle and
against the GPU native per-draft-snapshot kernel.

* small steps (oracle runs everything): every output element, record entry
  and committed state within tolerance, and untouched entries untouched;
* full-size workloads in the launch configuration the benchmark times:
  verify == native and commit == native snapshot n bit for bit over every
  layer, row and head (plus no stray pool writes), every native snapshot
  written exactly inside the live windows, and sampled (layer, row, head)
  units -- outputs, record, all snapshots and committed states --
  recomputed by the oracle.
"""
import gc

import numpy as np
import pytest
import torch

from spec_decode_recurrent_gb300 import api, build, step, workloads as wl
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


def _free():
    gc.collect()
    torch.cuda.empty_cache()


# ------------------------------------------------------------ small steps
def test_tiny_config_full_oracle():
    sb = wl.tiny(device="cuda")
    gs = GpuStep(sb)
    assert gs.err == 0 and gs.verify_err == 0
    gs.check_bitwise()
    layers, pools, err = oracle_full(sb, gs.before)
    assert np.all(err == 0)
    compare_full(gs, layers, pools)


SMALL = {
    # two 64-row tiles per head, ragged windows incl. decode-only (1) and padding (0),
    # a null-slot row, strided fused q/k/v, permuted rows with gaps
    "ragged_fp32": dict(HK=2, HV=4, K=128, V=128, W=6, L=2, windows=[6, 4, 1, 3, 0, 6, 2],
                        accepted=[3, 4, 1, 2, 0, 6, 1], null_rows=(5,), gaps=[1, 0, 2, 3, 0, 1, 0],
                        shuffle_rows=True, fused=True),
    "ragged_bf16_qkv": dict(HK=2, HV=4, K=128, V=128, W=6, L=2, windows=[6, 4, 1, 3, 0, 6, 2],
                            accepted=[6, 1, 1, 3, 0, 2, 2], gaps=[0, 2, 1, 0, 3, 1, 2],
                            shuffle_rows=True, fused=True, qkv_dtype=wl.BF16),
    "extreme_gates": dict(HK=1, HV=2, K=128, V=128, W=6, L=1, windows=[6, 6, 5, 1],
                          accepted=[6, 3, 5, 1], gate_range=20.0, qkv_dtype=wl.BF16),
    "bf16_state": dict(HK=2, HV=4, K=128, V=128, W=4, L=2, windows=[4, 4, 2, 0],
                       accepted=[4, 1, 2, 0], qkv_dtype=wl.BF16, state_dtype=wl.BF16),
    "gqa4_k64_v32": dict(HK=1, HV=4, K=64, V=32, W=5, L=2, windows=[5, 3, 5], accepted=[2, 3, 5]),
    "k32_v64": dict(HK=3, HV=6, K=32, V=64, W=4, L=1, windows=[4, 2], accepted=[1, 2]),
    "k16_v128": dict(HK=1, HV=1, K=16, V=128, W=3, L=1, windows=[3, 3], accepted=[3, 2]),
    "k128_v16": dict(HK=1, HV=2, K=128, V=16, W=3, L=1, windows=[3, 1], accepted=[2, 1]),
    "max_window16": dict(HK=1, HV=2, K=128, V=128, W=16, L=1, windows=[16, 9, 16],
                         accepted=[16, 9, 7]),
    "align_fp32": dict(HK=2, HV=4, K=128, V=128, W=4, L=2, windows=[4] * 8,
                       accepted=[1, 2, 3, 4, 4, 4, 2, 3], block_size=4,
                       seq_pos=[4, 5, 6, 7, 8, 9, 10, 11]),
    "align_bf16_state": dict(HK=2, HV=4, K=128, V=128, W=4, L=2, windows=[4] * 8,
                             accepted=[4, 3, 2, 1, 4, 4, 2, 3], block_size=4,
                             seq_pos=[4, 5, 6, 7, 8, 9, 10, 11], qkv_dtype=wl.BF16,
                             state_dtype=wl.BF16),
    "align_multi_boundary": dict(HK=1, HV=2, K=128, V=128, W=16, L=1, windows=[16, 16, 9, 12],
                                 accepted=[16, 13, 9, 12], block_size=4, seq_pos=[5, 8, 3, 1]),
    "align_block3_w6": dict(HK=1, HV=2, K=64, V=64, W=6, L=2, windows=[6, 6, 6, 3],
                            accepted=[6, 5, 3, 3], block_size=3, seq_pos=[1, 2, 3, 7]),
    # a head of one 64-row tile (K = 128, V = 64): the verify's one-tile path,
    # fp32 and bf16 state
    "two_tile_span": dict(HK=1, HV=2, K=128, V=64, W=5, L=2, windows=[5, 2, 1, 5],
                          accepted=[3, 2, 1, 5], qkv_dtype=wl.BF16),
    "two_tile_span_bf16_state": dict(HK=1, HV=2, K=128, V=64, W=4, L=1, windows=[4, 3, 4],
                                     accepted=[2, 3, 4], qkv_dtype=wl.BF16, state_dtype=wl.BF16),
    # four 32-row tiles per verify CTA (K = 64, V = 128): the 4-token build
    # and the generic one
    "k64_v128_four_tiles": dict(HK=1, HV=2, K=64, V=128, W=4, L=2, windows=[4, 3, 4],
                                accepted=[2, 3, 4], qkv_dtype=wl.BF16),
    "k64_v128_four_tiles_w5": dict(HK=1, HV=2, K=64, V=128, W=5, L=1, windows=[5, 2],
                                   accepted=[5, 1]),
    # bf16 states at narrow heads: the shared-memory-staged commit with a
    # tile taller than the head (ragged) and with two row tiles
    "k64_bf16_state": dict(HK=2, HV=4, K=64, V=64, W=4, L=2, windows=[4, 1, 4],
                           accepted=[4, 1, 3], state_dtype=wl.BF16),
    "k32_v128_bf16_state": dict(HK=1, HV=2, K=32, V=128, W=3, L=1, windows=[3, 2],
                                accepted=[1, 2], state_dtype=wl.BF16),
    # window 16 with a bf16 state: the staged commit needs more than 48 KiB of
    # shared memory per CTA (the opt-in path)
    "max_window16_bf16_state": dict(HK=1, HV=2, K=128, V=128, W=16, L=1, windows=[16, 11],
                                    accepted=[16, 5], qkv_dtype=wl.BF16, state_dtype=wl.BF16),
    "k16_bf16_state_align": dict(HK=1, HV=1, K=16, V=32, W=6, L=1, windows=[6, 6],
                                 accepted=[6, 4], block_size=2, seq_pos=[2, 5],
                                 state_dtype=wl.BF16),
    # every window length under the unrolled 4-token build
    "w4_every_window": dict(HK=1, HV=2, K=128, V=128, W=4, L=1, windows=[1, 2, 3, 4],
                            accepted=[1, 2, 1, 3], qkv_dtype=wl.BF16),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_step_full_oracle(name):
    sb = wl.custom(device="cuda", **SMALL[name])
    gs = GpuStep(sb)
    assert gs.err == 0 and gs.verify_err == 0
    gs.check_bitwise()
    layers, pools, err = oracle_full(sb, gs.before)
    assert np.all(err == 0)
    compare_full(gs, layers, pools)


# ------------------------------------------------------- full-size workloads
FULL = {
    "layer": lambda: wl.layer(device="cuda"),
    "all_layer": lambda: wl.all_layer(device="cuda"),
    "mtp5": lambda: wl.mtp5(device="cuda"),
    "long_ragged_seed30": lambda: wl.long_ragged(device="cuda", seed=30),
    "long_ragged_seed31": lambda: wl.long_ragged(device="cuda", seed=31),
    "long_ragged_seed32": lambda: wl.long_ragged(device="cuda", seed=32),
    "align_fp32": lambda: wl.align(device="cuda"),
    "align_bf16": lambda: wl.align(device="cuda", state_dtype=wl.BF16),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workload(name):
    sb = FULL[name]()
    try:
        gs = GpuStep(sb, units=12, unit_seed=len(name))
        assert gs.err == 0 and gs.verify_err == 0
        gs.check_bitwise()
        for l, r, h in gs.unit_list:
            gs.check_unit_against_oracle(l, r, h)
    finally:
        del sb
        _free()


# ------------------------------------------------------------- edge cases
def test_identity_gates_commit_leaves_state_bitwise():
    sb = wl.custom(device="cuda", HK=1, HV=2, K=128, V=128, W=4, L=2, windows=[4, 3],
                   accepted=[4, 2])
    for l in range(sb.L):
        sb.a[l].fill_(-1e4)     # softplus -> 0: decay 1
        sb.b[l].fill_(-1e4)     # sigmoid -> 0: no write
    gs = GpuStep(sb)
    for l in range(sb.L):
        assert torch.equal(sb.pools[l].view(torch.int32), gs.before[l].view(torch.int32))
        assert torch.count_nonzero(gs.bufs.rec_u[l][:, :, :3]) == 0


def test_accepted_zero_and_padding_rows_write_nothing():
    sb = wl.custom(device="cuda", HK=1, HV=2, K=64, V=64, W=4, L=2, windows=[4, 0, 4, 4],
                   accepted=[0, 0, 0, 2], null_rows=(2,))
    gs = GpuStep(sb)
    assert gs.err == 0
    gs.check_bitwise()
    for l in range(sb.L):
        # only row 3's slot may change
        changed = (sb.pools[l].view(torch.int32) != gs.before[l].view(torch.int32))
        slots = changed.flatten(1).any(1).nonzero().flatten().tolist()
        assert slots == [int(sb.slot_table[3, 0])]
        # the null row and the empty row wrote no outputs or records
        t0 = int(sb.token_start[2])
        assert torch.isnan(gs.bufs.out[l][t0:t0 + 4]).all()
        assert torch.isnan(gs.bufs.rec_u[l][1:3]).all()


def test_empty_batch_is_a_no_op():
    sb = wl.custom(device="cuda", HK=1, HV=2, K=64, V=64, W=4, L=1, windows=[4], accepted=[2])
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    bufs = step.StepBuffers(sb, fill=float("nan"))
    api.gdn_spec_verify(q=sb.q[0], k=sb.k[0], v=sb.v[0], a=sb.a[0], b=sb.b[0], A_log=sb.A_log[0],
                        dt_bias=sb.dt_bias[0], token_start=e, window_len=e,
                        state_pool=sb.pools[0], slot_table=e.view(0, 1), out=bufs.out[0],
                        rec_u=bufs.rec_u[0][:0], rec_k=bufs.rec_k[0][:0], rec_g=bufs.rec_g[0][:0],
                        max_window=sb.W)
    torch.cuda.synchronize()
    assert torch.isnan(bufs.out[0]).all()


def test_malformed_rows_are_flagged_and_skipped():
    # rows: fine | accepted > window | slot out of range | window > W | token rows past T
    sb = wl.custom(device="cuda", HK=1, HV=2, K=64, V=64, W=4, L=1, windows=[4, 2, 3, 4, 2],
                   accepted=[2, 1, 1, 1, 1])
    sb.accepted_len[1] = 3
    sb.slot_table[2, 0] = sb.num_slots + 5
    sb.window_len[3] = 5
    sb.token_start[4] = sb.T - 1   # the commit skips it by the verify's reject marker
    gs = GpuStep(sb, native=False)
    assert gs.verify_err == api.ROW_ERR_SLOT | api.ROW_ERR_WINDOW | api.ROW_ERR_TOKENS
    assert gs.err == (api.ROW_ERR_SLOT | api.ROW_ERR_WINDOW | api.ROW_ERR_TOKENS
                      | api.ROW_ERR_ACCEPTED | api.ROW_ERR_REJECTED)
    changed = (sb.pools[0].view(torch.int32) != gs.before[0].view(torch.int32))
    slots = changed.flatten(1).any(1).nonzero().flatten().tolist()
    assert slots == [int(sb.slot_table[0, 0])]


@pytest.mark.parametrize("state_dtype", [wl.F32, wl.BF16])
def test_commit_skips_rows_the_verify_rejected(state_dtype):
    # Row 1's window runs past the token rows: the verify rejects it and
    # leaves a stale (here NaN-filled) record.  The caller commits without
    # looking at the error word in between, with accepted_len > 0 for every
    # row; row 1's slot must stay bitwise unchanged in every layer while the
    # other rows commit as usual.
    sb = wl.custom(device="cuda", HK=1, HV=2, K=128, V=128, W=4, L=2, windows=[4, 3, 4],
                   accepted=[2, 3, 4], qkv_dtype=wl.BF16, state_dtype=state_dtype)
    sb.token_start[1] = sb.T - 2
    gs = GpuStep(sb, native=False)
    assert gs.verify_err == api.ROW_ERR_TOKENS
    assert gs.err == api.ROW_ERR_TOKENS | api.ROW_ERR_REJECTED
    bad = int(sb.slot_table[1, 0])
    for l in range(sb.L):
        assert torch.equal(bits(sb.pools[l][bad]), bits(gs.before[l][bad])), f"layer {l}"
        assert torch.equal(gs.bufs.rec_g[l][1, :, 0].cpu(), torch.full((sb.HV,), -1.0))
        changed = (bits(sb.pools[l]) != bits(gs.before[l])).flatten(1).any(1)
        assert changed.nonzero().flatten().tolist() == sorted(
            int(sb.slot_table[r, 0]) for r in (0, 2))


def test_align_missing_block_is_flagged():
    sb = wl.custom(device="cuda", HK=1, HV=2, K=64, V=64, W=4, L=1, windows=[4, 4],
                   accepted=[4, 4], block_size=4, seq_pos=[6, 4])
    final_col = (6 + 4 - 1) // 4
    sb.slot_table[0, final_col] = -1
    gs = GpuStep(sb, native=False)
    assert gs.verify_err == 0
    assert gs.err == api.ROW_ERR_BLOCK


def test_host_validation_rejects_bad_arguments():
    sb = wl.custom(device="cuda", HK=1, HV=2, K=64, V=64, W=4, L=1, windows=[4], accepted=[2])
    bufs = step.StepBuffers(sb)
    kw = dict(q=sb.q[0], k=sb.k[0], v=sb.v[0], a=sb.a[0], b=sb.b[0], A_log=sb.A_log[0],
              dt_bias=sb.dt_bias[0], token_start=sb.token_start, window_len=sb.window_len,
              state_pool=sb.pools[0], slot_table=sb.slot_table, out=bufs.out[0],
              rec_u=bufs.rec_u[0], rec_k=bufs.rec_k[0], rec_g=bufs.rec_g[0], max_window=sb.W)
    with pytest.raises(api.GDNError) as e:
        api.gdn_spec_verify(**dict(kw, max_window=17, rec_u=torch.zeros(1, 2, 17, 64, device="cuda"),
                                   rec_k=torch.zeros(1, 2, 17, 64, device="cuda"),
                                   rec_g=torch.zeros(1, 2, 17, device="cuda")))
    assert e.value.code == -2
    with pytest.raises(api.GDNError) as e:       # negative block size
        api.gdn_spec_verify(**dict(kw, block_size=-1, seq_pos=sb.window_len))
    assert e.value.code == -3
    with pytest.raises(api.GDNError) as e:       # a row stride shorter than a row
        api.gdn_spec_verify(**dict(kw, q=sb.q[0].as_strided(sb.q[0].shape, (32, 64, 1))))
    assert e.value.code == -3


def test_align_commit_repeatable_bitwise():
    # A boundary slot can be the checkpoint slot; the commit must not read a
    # tile another CTA already overwrote.  Run the same commit 20 times from
    # the same checkpoint and require identical results.
    sb = wl.align(device="cuda", L=4, batch=128)
    bufs = step.StepBuffers(sb)
    step.verify_all(sb, bufs)
    before = [p.clone() for p in sb.pools]
    results = None
    for _ in range(20):
        for p, b in zip(sb.pools, before):
            p.copy_(b)
        step.commit(sb, bufs)
        torch.cuda.synchronize()
        now = [p.view(torch.int32).clone() for p in sb.pools]
        if results is None:
            results = now
        else:
            for a, b in zip(results, now):
                assert torch.equal(a, b)
    assert int(bufs.err.item()) == 0


def test_graph_captured_step_matches_eager_bitwise():
    # The benchmark replays the per-layer verify calls from a CUDA graph
    # captured through the C ABI; replay must give the eager results bit
    # for bit (same kernels, same launch configuration).
    sb = wl.custom(device="cuda", sentinel=False, HK=2, HV=4, K=128, V=128, W=4, L=3,
                   windows=[4, 3, 0, 4], accepted=[2, 3, 0, 4])
    before = [p.clone() for p in sb.pools]
    eager = step.StepBuffers(sb, fill=float("nan"))
    step.verify_all(sb, eager)
    step.commit(sb, eager)
    torch.cuda.synchronize()
    eager_pools = [p.clone() for p in sb.pools]
    for p, b in zip(sb.pools, before):
        p.copy_(b)
    bufs = step.StepBuffers(sb, fill=float("nan"))
    step.verify_all(sb, bufs)                     # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.verify_all(sb, bufs)
    bufs.out_all.fill_(float("nan"))
    g.replay()
    step.commit(sb, bufs)
    torch.cuda.synchronize()
    for l in range(sb.L):
        assert torch.equal(bufs.out[l].view(torch.int32), eager.out[l].view(torch.int32))
        assert torch.equal(bufs.rec_u[l].view(torch.int32), eager.rec_u[l].view(torch.int32))
        assert torch.equal(sb.pools[l].view(torch.int32), eager_pools[l].view(torch.int32))


@pytest.mark.parametrize("kda", [False, True])
def test_verify_writes_into_a_strided_output_view(kda):
    # The verify writes o_t straight into the layer's output, which may be a
    # slice of a wider buffer (vLLM PR, Commits item 2: out=): the strided
    # result equals the contiguous one bit for bit, and the columns between
    # rows stay untouched.
    sb = wl.custom(device="cuda", kda=kda, HK=2, HV=4, K=128, V=128, W=4, L=1,
                   windows=[4, 2, 3], accepted=[2, 2, 3], qkv_dtype=wl.BF16)
    ref = step.StepBuffers(sb, fill=float("nan"))
    step.verify_all(sb, ref)
    pad = 96
    wide = torch.full((sb.T, sb.HV * sb.V + pad), float("nan"), device="cuda")
    view = wide[:, :sb.HV * sb.V].view(sb.T, sb.HV, sb.V)
    assert view.stride(0) == sb.HV * sb.V + pad
    bufs = step.StepBuffers(sb, fill=float("nan"))
    bufs.out[0] = view
    step.verify_all(sb, bufs)
    torch.cuda.synchronize()
    assert torch.equal(bits(view.contiguous()), bits(ref.out[0]))
    assert torch.isnan(wide[:, sb.HV * sb.V:]).all()
    for name in ("rec_u", "rec_k", "rec_g"):
        assert torch.equal(bits(getattr(bufs, name)[0]), bits(getattr(ref, name)[0]))


@pytest.mark.parametrize("kda", [False, True])
def test_verify_reads_inputs_the_previous_kernel_wrote(kda):
    # The verify is launched as a programmatic dependent of the stream's
    # previous kernel: its CTAs may start while that kernel's last CTAs run,
    # and must not read before it has finished.  Here the previous kernels
    # rewrite every input of the step (after a scramble) right before each
    # verify; the outputs must be the reference ones every time.
    sb = wl.custom(device="cuda", kda=kda, HK=2, HV=4, K=128, V=128, W=4, L=1,
                   windows=[4, 3, 4, 2], accepted=[2, 3, 4, 1], qkv_dtype=wl.BF16)
    ref = step.StepBuffers(sb, fill=float("nan"))
    step.verify_all(sb, ref)
    torch.cuda.synchronize()
    inputs = [sb.q[0], sb.k[0], sb.v[0], sb.a[0], sb.b[0]]
    saved = [x.clone() for x in inputs]
    for _ in range(20):
        bufs = step.StepBuffers(sb, fill=float("nan"))
        for x in inputs:
            x.fill_(7.0)
        for x, y in zip(inputs, saved):
            x.copy_(y)
        step.verify_all(sb, bufs)
        torch.cuda.synchronize()
        for name in ("out", "rec_u", "rec_k", "rec_g"):
            assert torch.equal(bits(getattr(ref, name)[0]), bits(getattr(bufs, name)[0])), name
