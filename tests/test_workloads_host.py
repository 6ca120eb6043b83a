"""CPU checks of the seeded input generators and of the host side of the
parity harness and the benchmark (no GPU): every workload the GPU tests and
the benchmark use can be drawn, is well formed, and the oracle runs on it."""
import numpy as np
import pytest
import torch

import oracle
from spec_decode_recurrent_gb300 import roofline, workloads as wl
from tests import test_gpu_parity as gp
from tests._parity import oracle_full, row_plan


def _check_layout(sb):
    assert sb.token_start.shape == (sb.B,) and sb.window_len.shape == (sb.B,)
    for r in range(sb.B):
        w, t0 = int(sb.window_len[r]), int(sb.token_start[r])
        assert 0 <= t0 and t0 + w <= sb.T
        src, writes = row_plan(sb, r)
        if w > 0 and src >= 0:
            pool = sb.pools[0][src].float()
            assert torch.isfinite(pool).all(), f"row {r} reads a sentinel slot"
        for slot, ntok in writes:
            assert 0 <= slot < sb.num_slots and 1 <= ntok <= int(sb.accepted_len[r])
    # no two live rows share a written slot
    seen = set()
    for r in range(sb.B):
        for slot, _ in row_plan(sb, r)[1]:
            assert slot not in seen
            seen.add(slot)


@pytest.mark.parametrize("name", sorted(gp.SMALL))
def test_small_cases_generate_and_run_on_the_oracle(name):
    sb = wl.custom(device="cpu", **gp.SMALL[name])
    _check_layout(sb)
    layers, pools, err = oracle_full(sb, sb.pools)
    assert np.all(err == 0)
    assert all(np.isfinite(x["out"][~np.isnan(x["out"])]).all() for x in layers)


def test_named_workloads_generate_small():
    for sb in (wl.tiny(), wl.layer(batch=4, HK=2, HV=4, KV=16, num_slots=8),
               wl.all_layer(L=2, batch=10, pad_rows=2, HK=2, HV=4, KV=16, num_slots=16),
               wl.long_ragged(L=2, batch=12, HK=2, HV=4, KV=16, num_slots=24),
               wl.align(L=2, batch=16, HK=2, HV=4, KV=16, num_slots=40),
               wl.align(L=1, batch=16, HK=2, HV=4, KV=16, num_slots=40, state_dtype=wl.BF16),
               wl.mtp5(L=2, batch=12, pad_rows=2, HK=2, HV=4, KV=16, num_slots=24)):
        _check_layout(sb)
        assert roofline.commit_bytes(sb) > 0 and roofline.verify_bytes_per_layer(sb) > 0


def test_align_workload_covers_every_boundary_case():
    sb = wl.align(L=1, batch=128, HK=1, HV=1, KV=16, num_slots=384)
    pairs = {(int(p) % 4, int(n)) for p, n in zip(sb.seq_pos, sb.accepted_len)}
    assert pairs == {(r, n) for r in range(4) for n in range(1, 5)}
    same = 0
    for r in range(sb.B):
        src, writes = row_plan(sb, r)
        same += any(s == src for s, _ in writes[1:])
    assert same > 0          # some boundary writes land in the checkpoint slot


def test_sentinels_are_nan_bit_patterns():
    f = wl.sentinel_like((3,), wl.F32, "cpu")
    b = wl.sentinel_like((3,), wl.BF16, "cpu")
    assert torch.isnan(f).all() and torch.isnan(b.float()).all()
    assert f.view(torch.int32)[0].item() == wl.SENTINEL_F32_BITS
    assert b.view(torch.int16)[0].item() == wl.SENTINEL_BF16_BITS


def test_bench_cpu_baseline_helpers_run_on_cpu():
    import bench
    sb = wl.all_layer(L=2, batch=6, pad_rows=1, HK=2, HV=4, KV=16, num_slots=12, sentinel=False)
    d = bench._compact_layer(sb, 0, list(range(sb.B)))
    bench._oracle_unit_of_work(oracle, d)
    res = bench.cpu_baseline(sb, 0.01, 0.01)
    assert res["value"] > 0 and res["cores"] >= 1
    assert res["single_core"]["cores"] == 1 and res["single_core"]["value"] > 0
    assert oracle.num_threads() == res["cores"]      # the thread count is restored


@pytest.mark.parametrize("fused", [False, True])
def test_pack_inputs_keeps_values_and_layout(fused):
    from spec_decode_recurrent_gb300 import step
    make = wl.long_ragged if fused else wl.all_layer
    kw = dict(L=2, batch=6, HK=2, HV=4, KV=16, num_slots=12, sentinel=False)
    if not fused:
        kw["pad_rows"] = 1
    sb = make(**kw)
    ref = {n: [(t.clone(), t.stride()) for t in getattr(sb, n)] for n in ("q", "k", "v", "a", "b")}
    meta = sb.slot_table.clone()
    arena = step.pack_inputs(sb)
    for n, ts in ref.items():
        for l, (t, stride) in enumerate(ts):
            got = getattr(sb, n)[l]
            assert got.shape == t.shape and got.stride() == stride and torch.equal(got, t)
            assert got.untyped_storage().data_ptr() == arena.untyped_storage().data_ptr()
    assert torch.equal(sb.slot_table, meta)


def test_conv_state_generator_and_oracle_on_cpu():
    sb = wl.long_ragged(L=2, batch=8, HK=2, HV=4, KV=16, num_slots=16, sentinel=False)
    pools, inputs = wl.conv_state(sb, state_len=3)
    C = 2 * sb.HK * sb.K + sb.HV * sb.V
    assert pools[0].shape == (sb.num_slots, C, 3) and inputs[0].shape == (sb.T, C)
    assert inputs[0].data_ptr() == sb.fused_qkv[0].data_ptr()      # fused rows reused
    ref, err = oracle.conv_commit(pools=np.stack([p.double().numpy() for p in pools]),
                                  inputs=np.stack([x.double().numpy() for x in inputs]),
                                  token_start=sb.token_start, window_len=sb.window_len,
                                  accepted_len=sb.accepted_len, slot_table=sb.slot_table,
                                  max_window=sb.W)
    assert np.all(err == 0)


def test_mtp5_acceptance_profile_matches_the_measured_rates():
    # the rates imply the mean accepted length printed beside them (3.941)
    assert abs(1 + sum(wl.MTP5_ACCEPT) - 3.941) < 1e-9
    n = 200_000
    lens = np.array(wl.accepted_from_profile(torch.Generator().manual_seed(0), wl.MTP5_ACCEPT, n))
    assert lens.min() >= 1 and lens.max() <= 6
    for i, p in enumerate(wl.MTP5_ACCEPT, start=1):
        sigma = (p * (1 - p) / n) ** 0.5
        assert abs((lens >= 1 + i).mean() - p) < 5 * sigma, (i, (lens >= 1 + i).mean(), p)
    assert abs(lens.mean() - 3.941) < 0.02
    sb = wl.mtp5(L=1, batch=64, pad_rows=8, HK=2, HV=4, KV=16, num_slots=128)
    live = sb.window_len > 0
    assert int(live.sum()) == 56 and sb.W == 6
    assert bool((sb.window_len[live] == 6).all())
    acc = sb.accepted_len[live]
    assert bool((acc >= 1).all() and (acc <= 6).all())
    assert bool((sb.accepted_len[~live] == 0).all())



def test_slot_exclusivity_check():
    from spec_decode_recurrent_gb300 import step
    # every benchmark workload commits to disjoint slots
    for sb in (wl.all_layer(L=1, batch=10, pad_rows=2, HK=2, HV=4, KV=16, num_slots=16),
               wl.align(L=1, batch=32, HK=1, HV=2, KV=16, num_slots=80),
               wl.long_ragged(L=1, batch=12, HK=2, HV=4, KV=16, num_slots=24)):
        step.check_slot_exclusivity(sb.window_len, sb.accepted_len, sb.slot_table, sb.seq_pos,
                                    sb.block_size)
    i32 = lambda x: torch.tensor(x, dtype=torch.int32)
    # two rows writing the same slot in place
    with pytest.raises(ValueError, match="slot 3"):
        step.check_slot_exclusivity(i32([4, 4]), i32([2, 1]), i32([[3], [3]]))
    # a null row, or a row with nothing accepted, may share (it writes nothing)
    step.check_slot_exclusivity(i32([4, 4]), i32([2, 0]), i32([[3], [3]]))
    step.check_slot_exclusivity(i32([4, 4]), i32([2, 1]), i32([[3], [-1]]))
    # align mode: row 0's boundary slot is row 1's checkpoint slot
    with pytest.raises(ValueError, match="slot 7"):
        step.check_slot_exclusivity(i32([4, 4]), i32([4, 1]), i32([[5, 7, 8], [7, 9, -1]]),
                                    i32([4, 4]), 4)
    # a row may write its own checkpoint slot (boundary = source)
    step.check_slot_exclusivity(i32([4]), i32([3]), i32([[5, 6, 7]]), i32([6]), 4)
