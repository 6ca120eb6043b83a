"""GPU parity of the short-conv state commit against the fp64 oracle.  The
commit only copies elements, so the bar is bit-exact: every stored value
equals the oracle's (which is an exact copy of an input), and every other
element is untouched."""
import gc

import numpy as np
import pytest
import torch

import oracle
from spec_decode_recurrent_gb300 import api, build, workloads as wl
from tests._parity import cpu64

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


def _run(sb, pools, inputs, slot_tables=None, layer_group=None):
    tab = api.ConvTable(pools, inputs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = sb.slot_table if slot_tables is None else slot_tables
    before = [p.clone() for p in pools]
    api.gdn_conv_state_commit(table=tab, token_start=sb.token_start, window_len=sb.window_len,
                              accepted_len=sb.accepted_len, slot_tables=st, max_window=sb.W,
                              layer_group=layer_group, seq_pos=sb.seq_pos,
                              block_size=sb.block_size, err=err)
    torch.cuda.synchronize()
    ref, row_err = oracle.conv_commit(
        pools=np.stack([cpu64(p) for p in before]), inputs=np.stack([cpu64(x) for x in inputs]),
        token_start=sb.token_start.cpu(), window_len=sb.window_len.cpu(),
        accepted_len=sb.accepted_len.cpu(), slot_table=st.cpu(),
        layer_group=None if layer_group is None else layer_group.cpu(),
        seq_pos=None if sb.seq_pos is None else sb.seq_pos.cpu(), block_size=sb.block_size,
        max_window=sb.W)
    return [cpu64(p) for p in pools], ref, int(err.item()), int(np.bitwise_or.reduce(row_err))


CASES = {
    "padding_rows_bf16": lambda: wl.all_layer(device="cuda", sentinel=False, L=2, batch=10,
                                              pad_rows=2, HK=2, HV=4, KV=128, num_slots=16),
    "ragged_fused_strided": lambda: wl.long_ragged(device="cuda", sentinel=False, L=2, batch=12,
                                                   HK=2, HV=4, KV=64, num_slots=24),
    "align_block4": lambda: wl.align(device="cuda", sentinel=False, L=2, batch=32, HK=1, HV=2,
                                     KV=64, num_slots=80),
    "align_multi_boundary": lambda: wl.custom(device="cuda", sentinel=False, HK=1, HV=2, K=64,
                                              V=64, W=16, L=1, windows=[16, 16, 9, 12],
                                              accepted=[16, 13, 9, 12], block_size=4,
                                              seq_pos=[5, 8, 3, 1]),
    "full_width_4_layers": lambda: wl.all_layer(device="cuda", sentinel=False, L=4),
}


# every small case at every dtype and state length; the full-width case only
# in the serving configuration (bf16 states, width-4 convolution)
PARAMS = [(n, d, sl) for n in sorted(CASES) if n != "full_width_4_layers"
          for d in ("bf16", "f32") for sl in (3, 1, 8)] + [("full_width_4_layers", "bf16", 3)]


@pytest.mark.parametrize("name,dtype,state_len", PARAMS)
def test_conv_commit_bit_exact(name, dtype, state_len):
    sb = CASES[name]()
    dt = wl.BF16 if dtype == "bf16" else wl.F32
    pools, inputs = wl.conv_state(sb, state_len=state_len, dtype=dt)
    got, ref, err, ref_err = _run(sb, pools, inputs)
    assert err == 0 and ref_err == 0
    for l, (g, r) in enumerate(zip(got, ref)):
        assert np.array_equal(g, r), f"layer {l}"


def test_conv_commit_grouped():
    sb = wl.custom(device="cuda", sentinel=False, HK=1, HV=2, K=64, V=64, W=4, L=6,
                   windows=[4, 3, 4, 0], accepted=[2, 3, 4, 0], num_slots=12)
    gen = torch.Generator().manual_seed(3)
    tables = torch.stack([sb.slot_table.cpu()] + [
        torch.randperm(sb.num_slots, generator=gen)[:sb.B].view(-1, 1).to(torch.int32)
        for _ in range(2)]).cuda().contiguous()
    layer_group = torch.tensor([0, 1, 2, 2, 1, 0], dtype=torch.int32, device="cuda")
    pools, inputs = wl.conv_state(sb, state_len=3)
    got, ref, err, ref_err = _run(sb, pools, inputs, tables, layer_group)
    assert err == 0 and ref_err == 0
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_conv_commit_flags_bad_rows():
    sb = wl.custom(device="cuda", sentinel=False, HK=1, HV=2, K=64, V=64, W=4, L=1,
                   windows=[4, 2, 3], accepted=[2, 1, 1])
    sb.accepted_len[1] = 3                  # more accepted than drafted
    sb.token_start[2] = sb.T - 1            # window runs past the token rows
    pools, inputs = wl.conv_state(sb, state_len=3)
    got, ref, err, ref_err = _run(sb, pools, inputs)
    assert err == ref_err == (api.ROW_ERR_ACCEPTED | api.ROW_ERR_TOKENS)
    assert np.array_equal(got[0], ref[0])
