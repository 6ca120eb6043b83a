"""GPU parity of the grouped all-layer commit (layers split into KV-cache
groups, each with its own [batch, stride] state-index table): one launch,
bit-identical to the native per-token states of each layer under its
group's table, and within tolerance of the fp64 oracle's grouped commit."""
import gc

import numpy as np
import pytest
import torch

import oracle
from spec_decode_recurrent_gb300 import api, build, step, workloads as wl
from tests._parity import NAN, bits, cpu64
from tests._tol import check_close

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


def _case(G=3, L=6, seed=5):
    sb = wl.custom(device="cuda", sentinel=False, seed=seed, HK=2, HV=4, K=128, V=128, W=4, L=L,
                   windows=[4, 3, 4, 1, 0, 4], accepted=[2, 3, 4, 1, 0, 1], num_slots=24)
    gen = torch.Generator().manual_seed(seed)
    tables = [sb.slot_table.cpu()]
    for g in range(1, G):
        perm = torch.randperm(sb.num_slots, generator=gen)[:sb.B]
        tables.append(perm.view(-1, 1).to(torch.int32))
    tables[1][3, 0] = -1                      # this row is a padding row in group 1 only
    slot_tables = torch.stack(tables).to("cuda").contiguous()
    layer_group = torch.tensor([l % G for l in range(L)], dtype=torch.int32, device="cuda")
    return sb, slot_tables, layer_group


def _verify_layer(sb, bufs, l, table):
    api.gdn_spec_verify(q=sb.q[l], k=sb.k[l], v=sb.v[l], a=sb.a[l], b=sb.b[l], A_log=sb.A_log[l],
                        dt_bias=sb.dt_bias[l], token_start=sb.token_start, window_len=sb.window_len,
                        state_pool=sb.pools[l], slot_table=table, out=bufs.out[l],
                        rec_u=bufs.rec_u[l], rec_k=bufs.rec_k[l], rec_g=bufs.rec_g[l],
                        max_window=sb.W, err=bufs.err)


def test_grouped_commit_matches_native_and_oracle():
    sb, slot_tables, layer_group = _case()
    G = slot_tables.shape[0]
    before = [p.clone() for p in sb.pools]
    bufs = step.StepBuffers(sb, fill=NAN)
    expected = []
    for l in range(sb.L):
        g = int(layer_group[l])
        _verify_layer(sb, bufs, l, slot_tables[g])
        out, snaps = step.native_buffers(sb, fill=NAN)
        api.gdn_native_spec_snapshot(
            q=sb.q[l], k=sb.k[l], v=sb.v[l], a=sb.a[l], b=sb.b[l], A_log=sb.A_log[l],
            dt_bias=sb.dt_bias[l], token_start=sb.token_start, window_len=sb.window_len,
            state_pool=sb.pools[l], slot_table=slot_tables[g], out=out, snapshots=snaps,
            max_window=sb.W)
        exp = sb.pools[l].clone()
        for r in range(sb.B):
            src, writes = oracle.commit_plan(int(sb.window_len[r]), int(sb.accepted_len[r]),
                                             slot_tables[g, r].cpu(), 0, 0, sb.num_slots, sb.W)
            for slot, ntok in writes:
                exp[slot] = snaps[r, ntok - 1]
        expected.append(exp)
    api.gdn_replay_commit_grouped(table=bufs.table, num_k_heads=sb.HK, layer_group=layer_group,
                                  window_len=sb.window_len, accepted_len=sb.accepted_len,
                                  slot_tables=slot_tables, err=bufs.err)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    for l in range(sb.L):
        assert torch.equal(bits(sb.pools[l]), bits(expected[l])), f"layer {l}"

    # the oracle, from its own records
    recs = []
    for l in range(sb.L):
        g = int(layer_group[l])
        recs.append(oracle.spec_verify(
            q=sb.q[l].cpu(), k=sb.k[l].cpu(), v=sb.v[l].cpu(), a=sb.a[l].cpu(), b=sb.b[l].cpu(),
            A_log=sb.A_log[l].cpu(), dt_bias=sb.dt_bias[l].cpu(), token_start=sb.token_start.cpu(),
            window_len=sb.window_len.cpu(), pool=before[l].cpu(), slot_table=slot_tables[g].cpu(),
            max_window=sb.W))
    pools, err = oracle.replay_commit(
        pools=np.stack([cpu64(p) for p in before]), rec_u=np.stack([x["rec_u"] for x in recs]),
        rec_k=np.stack([x["rec_k"] for x in recs]), rec_g=np.stack([x["rec_g"] for x in recs]),
        window_len=sb.window_len.cpu(), accepted_len=sb.accepted_len.cpu(),
        slot_table=slot_tables.cpu(), layer_group=layer_group.cpu(), max_window=sb.W)
    assert np.all(err == 0)
    for l in range(sb.L):
        got, ref, was = cpu64(sb.pools[l]), pools[l], cpu64(before[l])
        changed = ref != was
        assert changed.any()
        assert np.array_equal(got[~changed], was[~changed])
        check_close(got[changed], ref[changed], f"layer {l} grouped commit")


def test_one_group_equals_plain_commit():
    sb, slot_tables, _ = _case(seed=6)
    bufs = step.StepBuffers(sb)
    step.verify_all(sb, bufs)
    before = [p.clone() for p in sb.pools]
    step.commit(sb, bufs)
    plain = [p.clone() for p in sb.pools]
    for p, b in zip(sb.pools, before):
        p.copy_(b)
    zeros = torch.zeros(sb.L, dtype=torch.int32, device="cuda")
    api.gdn_replay_commit_grouped(table=bufs.table, num_k_heads=sb.HK, layer_group=zeros,
                                  window_len=sb.window_len, accepted_len=sb.accepted_len,
                                  slot_tables=sb.slot_table.view(1, sb.B, -1).contiguous(),
                                  err=bufs.err)
    torch.cuda.synchronize()
    for a, b in zip(plain, sb.pools):
        assert torch.equal(bits(a), bits(b))


def test_bad_group_id_is_flagged_and_writes_nothing():
    sb, slot_tables, layer_group = _case(seed=7)
    bufs = step.StepBuffers(sb)
    for l in range(sb.L):
        _verify_layer(sb, bufs, l, slot_tables[int(layer_group[l])])
    layer_group[2] = 7
    before = sb.pools[2].clone()
    api.gdn_replay_commit_grouped(table=bufs.table, num_k_heads=sb.HK, layer_group=layer_group,
                                  window_len=sb.window_len, accepted_len=sb.accepted_len,
                                  slot_tables=slot_tables, err=bufs.err)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == api.ROW_ERR_GROUP
    assert torch.equal(bits(sb.pools[2]), bits(before))


def test_kda_grouped_commit_matches_native_and_oracle():
    # The per-channel-decay (KDA) records through the grouped commit: bit
    # for bit the native KDA snapshots of every layer under its group's
    # table, and within tolerance of the oracle's KDA commit of that layer.
    G, L, seed = 3, 6, 8
    sb = wl.custom(device="cuda", sentinel=False, seed=seed, kda=True, HK=2, HV=4, K=128, V=128,
                   W=4, L=L, windows=[4, 3, 4, 1, 0, 4], accepted=[2, 3, 4, 1, 0, 1], num_slots=24)
    gen = torch.Generator().manual_seed(seed)
    tables = [sb.slot_table.cpu()] + [
        torch.randperm(sb.num_slots, generator=gen)[:sb.B].view(-1, 1).to(torch.int32)
        for _ in range(1, G)]
    slot_tables = torch.stack(tables).to("cuda").contiguous()
    layer_group = torch.tensor([l % G for l in range(L)], dtype=torch.int32, device="cuda")
    before = [p.clone() for p in sb.pools]
    bufs = step.StepBuffers(sb, fill=NAN)
    expected = []
    for l in range(L):
        g = int(layer_group[l])
        kw = dict(q=sb.q[l], k=sb.k[l], v=sb.v[l], a=sb.a[l], b=sb.b[l], A_log=sb.A_log[l],
                  dt_bias=sb.dt_bias[l], token_start=sb.token_start, window_len=sb.window_len,
                  state_pool=sb.pools[l], slot_table=slot_tables[g], max_window=sb.W)
        api.gdn_kda_spec_verify(out=bufs.out[l], rec_u=bufs.rec_u[l], rec_k=bufs.rec_k[l],
                                rec_g=bufs.rec_g[l], err=bufs.err, **kw)
        out, snaps = step.native_buffers(sb, fill=NAN)
        api.gdn_kda_native_spec_snapshot(out=out, snapshots=snaps, **kw)
        exp = sb.pools[l].clone()
        for r in range(sb.B):
            src, writes = oracle.commit_plan(int(sb.window_len[r]), int(sb.accepted_len[r]),
                                             slot_tables[g, r].cpu(), 0, 0, sb.num_slots, sb.W)
            for slot, ntok in writes:
                exp[slot] = snaps[r, ntok - 1]
        expected.append(exp)
    api.gdn_replay_commit_grouped(table=bufs.table, num_k_heads=sb.HK, layer_group=layer_group,
                                  window_len=sb.window_len, accepted_len=sb.accepted_len,
                                  slot_tables=slot_tables, err=bufs.err)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    for l in range(L):
        assert torch.equal(bits(sb.pools[l]), bits(expected[l])), f"layer {l}"
        g = int(layer_group[l])
        rec = oracle.kda_spec_verify(
            q=sb.q[l].cpu(), k=sb.k[l].cpu(), v=sb.v[l].cpu(), a=sb.a[l].cpu(), b=sb.b[l].cpu(),
            A_log=sb.A_log[l].cpu(), dt_bias=sb.dt_bias[l].cpu(), token_start=sb.token_start.cpu(),
            window_len=sb.window_len.cpu(), pool=before[l].cpu(), slot_table=slot_tables[g].cpu(),
            max_window=sb.W)
        pools, err = oracle.kda_replay_commit(
            pools=cpu64(before[l])[None], rec_u=rec["rec_u"][None], rec_k=rec["rec_k"][None],
            rec_g=rec["rec_g"][None], window_len=sb.window_len.cpu(),
            accepted_len=sb.accepted_len.cpu(), slot_table=slot_tables[g].cpu(), max_window=sb.W)
        assert np.all(err == 0)
        got, ref, was = cpu64(sb.pools[l]), pools[0], cpu64(before[l])
        changed = ref != was
        assert changed.any()
        assert np.array_equal(got[~changed], was[~changed])
        check_close(got[changed], ref[changed], f"layer {l} KDA grouped commit")
