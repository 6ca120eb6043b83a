"""Pins for the fp64 oracle: facts fixed by the method and by mathematics,
not by re-running the oracle's own formulas.

Each test is chosen so that a plausible slip in the oracle -- a dropped
decay, a wrong sign, a transposed outer product, a wrong GQA index, an
off-by-one in the align-mode block arithmetic -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests._tol import bf16_ulp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ gates
@pytest.mark.parametrize("x", [-30.0, -3.0, -0.5, 0.0, 0.7, 4.0, 30.0])
@pytest.mark.parametrize("A_log", [0.0, math.log(3.0), math.log(16.0)])
def test_decay_closed_form(x, A_log):
    # exp(-c * log(1 + e^x)) == (1 + e^x)^(-c): a different evaluation route.
    c = math.exp(A_log)
    expect = (1.0 + math.exp(x)) ** (-c)
    got = oracle.decay(x - 0.25, A_log, 0.25)   # the gate adds dt_bias to a
    assert got == pytest.approx(expect, rel=1e-12, abs=1e-300)


def test_decay_special_values():
    assert oracle.decay(0.0, 0.0, 0.0) == pytest.approx(0.5, rel=1e-15)
    # softplus -> 0 exactly for very negative inputs: the identity decay
    assert oracle.decay(-1e4, 0.3, 0.0) == 1.0
    # the decay is a contraction for any input
    for a in np.linspace(-20, 20, 41):
        assert 0.0 <= oracle.decay(a, 1.0, 0.5) <= 1.0


def test_softplus_closed_forms():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    for c in (1e-3, 0.5, 2.0, 10.0):
        assert oracle.softplus(math.log(math.expm1(c))) == pytest.approx(c, rel=1e-12)
    assert oracle.softplus(800.0) == 800.0           # no overflow
    assert oracle.softplus(-800.0) == 0.0
    assert oracle.softplus(-30.0) == pytest.approx(math.exp(-30.0), rel=1e-12)


def test_beta_closed_forms():
    assert oracle.beta(0.0) == 0.5
    assert oracle.beta(math.log(3.0)) == pytest.approx(0.75, rel=1e-15)
    assert oracle.beta(-math.log(3.0)) == pytest.approx(0.25, rel=1e-15)
    assert oracle.beta(1e4) == 1.0
    assert oracle.beta(-1e4) == 0.0


def test_l2norm():
    assert np.allclose(oracle.l2norm([3.0, 4.0]), [0.6, 0.8], rtol=0, atol=1e-7)
    # eps sits under the square root: |l2norm(x)|^2 = s / (s + eps) with
    # s = |x|^2, so a vector with s = eps comes out with squared norm 1/2.
    y = oracle.l2norm([1e-3, 0.0])
    assert float(y @ y) == pytest.approx(0.5, rel=1e-12)
    assert np.array_equal(oracle.l2norm(np.zeros(8)), np.zeros(8))
    x = rng.normal(size=128)
    y = oracle.l2norm(x)
    assert np.linalg.norm(y) == pytest.approx(1.0, abs=1e-7)
    assert np.allclose(y / np.linalg.norm(y), x / np.linalg.norm(x), rtol=0, atol=1e-15)


# ------------------------------------------------------- one-unit recurrence
def test_worked_example_golden():
    with open(os.path.join(GOLDEN, "worked_example_two_tokens.json")) as f:
        g = json.load(f)
    r = oracle.window(g["S0"], g["q"], g["k"], g["v"], g["a"], g["b"], g["A_log"], g["dt_bias"])
    tol = g["atol"]
    assert np.allclose(r["alpha"], g["expect_alpha"], rtol=0, atol=1e-15)
    assert np.allclose(r["u"], g["expect_u"], rtol=0, atol=tol)
    assert np.allclose(r["states"], g["expect_states"], rtol=0, atol=tol)
    assert np.allclose(r["o"], g["expect_o"], rtol=0, atol=tol)
    assert np.allclose(r["khat"], np.array(g["k"]) / math.sqrt(1.0 + 1e-6), rtol=0, atol=1e-15)


def _random_unit(K=16, V=16, w=5, seed=0):
    g = np.random.default_rng(seed)
    return dict(S0=g.normal(0, 0.1, (V, K)), q=g.normal(size=(w, K)), k=g.normal(size=(w, K)),
                v=g.normal(size=(w, V)), a=g.normal(size=w), b=g.normal(size=w),
                A_log=float(g.uniform(0, math.log(16))), dt_bias=float(g.uniform(-1, 1)))


def test_identity_gate_leaves_state_unchanged():
    u = _random_unit()
    w = len(u["a"])
    r = oracle.window(u["S0"], u["q"], u["k"], u["v"], np.full(w, -1e4), np.full(w, -1e4),
                      u["A_log"], 0.0)
    for t in range(w):
        assert np.array_equal(r["states"][t], u["S0"])           # bit for bit
        qh = oracle.l2norm(u["q"][t])
        assert np.allclose(r["o"][t], u["S0"] @ qh, rtol=1e-13, atol=1e-15)
    assert np.array_equal(r["u"], np.zeros_like(r["u"]))
    assert np.array_equal(r["alpha"], np.ones(w))


def test_zero_state_single_token_is_rank_one():
    # S0 = 0: S1 = beta * v khat^T and o1 = beta * (khat . qhat) * v.
    u = _random_unit(K=8, V=12, w=1, seed=3)
    r = oracle.window(np.zeros((12, 8)), u["q"], u["k"], u["v"], u["a"], u["b"],
                      u["A_log"], u["dt_bias"])
    be = 1.0 / (1.0 + math.exp(-u["b"][0]))
    kh, qh = oracle.l2norm(u["k"][0]), oracle.l2norm(u["q"][0])
    assert np.allclose(r["states"][0], be * np.outer(u["v"][0], kh), rtol=1e-13, atol=1e-15)
    assert np.allclose(r["o"][0], be * float(kh @ qh) * u["v"][0], rtol=1e-12, atol=1e-14)


def test_write_invariant_full_strength():
    # beta = 1: after each token the state maps the (normalised) key onto
    # its value, S_t khat_t = v_t, up to |khat|^2 = 1 - eps/(|k|^2 + eps).
    u = _random_unit(K=32, V=24, w=6, seed=5)
    w = len(u["a"])
    r = oracle.window(u["S0"], u["q"], u["k"], u["v"], u["a"], np.full(w, 1e4),
                      u["A_log"], u["dt_bias"])
    for t in range(w):
        kh = oracle.l2norm(u["k"][t])
        assert np.allclose(r["states"][t] @ kh, u["v"][t], rtol=0, atol=1e-6)


def test_orthonormal_keys_store_exact_memories():
    # alpha = 1, beta = 1, keys = distinct basis vectors: the delta rule
    # writes each value into its key's column and leaves the rest alone:
    # S_n = S0 + sum_t (v_t - S0 e_t) e_t^T.
    K, V, w = 10, 7, 4
    g = np.random.default_rng(7)
    S0 = g.normal(0, 0.1, (V, K))
    cols = [3, 0, 8, 5]
    k = np.zeros((w, K)); k[np.arange(w), cols] = 2.5      # scale is removed by the norm
    v = g.normal(size=(w, V)); q = g.normal(size=(w, K))
    r = oracle.window(S0, q, k, v, np.full(w, -1e4), np.full(w, 1e4), 0.0, 0.0)
    expect = S0.copy()
    for t, c in enumerate(cols):
        expect[:, c] = v[t]
    assert np.allclose(r["states"][-1], expect, rtol=0, atol=1e-6)


def test_pure_decay():
    # beta = 0: S_n = (prod alpha_t) S0, with alpha from the closed form.
    u = _random_unit(w=4, seed=9)
    r = oracle.window(u["S0"], u["q"], u["k"], u["v"], u["a"], np.full(4, -1e4),
                      u["A_log"], u["dt_bias"])
    c = math.exp(u["A_log"])
    prod = 1.0
    for t in range(4):
        prod *= (1.0 + math.exp(u["a"][t] + u["dt_bias"])) ** (-c)
        assert np.allclose(r["states"][t], prod * u["S0"], rtol=1e-12, atol=1e-300)


def test_replay_from_record_equals_recompute():
    u = _random_unit(K=16, V=16, w=6, seed=11)
    r = oracle.window(u["S0"], u["q"], u["k"], u["v"], u["a"], u["b"], u["A_log"], u["dt_bias"])
    assert np.array_equal(oracle.replay(u["S0"], r["u"][:0], r["khat"][:0], r["alpha"][:0]),
                          u["S0"])
    for n in range(1, 7):
        S = oracle.replay(u["S0"], r["u"][:n], r["khat"][:n], r["alpha"][:n])
        assert np.allclose(S, r["states"][n - 1], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------- align-mode plan
def _brute_force_writes(p0, n, Bk):
    """Walk the accepted tokens one by one: the block of token x (1-based
    position) ends up holding the state after the last accepted token that
    falls in it.  Returns {column: tokens folded}."""
    cols = {}
    for x in range(p0 + 1, p0 + n + 1):
        cols[(x - 1) // Bk] = x - p0
    return cols


@pytest.mark.parametrize("Bk", [1, 2, 3, 4, 8])
def test_align_plan_matches_brute_force(Bk):
    W = 6
    for p0 in range(1, 4 * Bk + 1):
        ncols = (p0 + W - 1) // Bk + 1
        table = [100 + c for c in range(ncols)]   # column c -> slot 100 + c
        for n in range(0, W + 1):
            src, writes = oracle.commit_plan(W, n, table, p0, Bk, 1000, W)
            assert src == table[(p0 - 1) // Bk]
            got = {s - 100: t for s, t in writes}
            assert len(got) == len(writes), "a slot written twice"
            assert got == _brute_force_writes(p0, n, Bk), (p0, n)
            if writes:
                assert writes[0] == (table[(p0 + n - 1) // Bk], n)   # final first


def test_plan_without_align_mode_updates_in_place():
    for n in range(0, 5):
        src, writes = oracle.commit_plan(4, n, [42], 0, 0, 64, 4)
        assert src == 42
        assert writes == ([] if n == 0 else [(42, n)])


def test_plan_null_and_errors():
    assert oracle.commit_plan(4, 2, [-1], 0, 0, 8, 4) == (-1, [])          # null slot
    assert oracle.commit_plan(0, 0, [3], 0, 0, 8, 4) == (-1, [])           # empty window
    with pytest.raises(ValueError) as e:
        oracle.commit_plan(4, 5, [3], 0, 0, 8, 4)
    assert e.value.args[0] == oracle.ERR_ACCEPTED
    with pytest.raises(ValueError) as e:
        oracle.commit_plan(5, 1, [3], 0, 0, 8, 4)
    assert e.value.args[0] == oracle.ERR_WINDOW
    with pytest.raises(ValueError) as e:
        oracle.commit_plan(4, 1, [8], 0, 0, 8, 4)
    assert e.value.args[0] == oracle.ERR_SLOT
    with pytest.raises(ValueError) as e:            # align: final block missing
        oracle.commit_plan(4, 2, [5, -1], 4, 4, 8, 4)
    assert e.value.args[0] == oracle.ERR_BLOCK
    with pytest.raises(ValueError) as e:            # align: column beyond the table
        oracle.commit_plan(4, 2, [5], 4, 4, 8, 4)
    assert e.value.args[0] == oracle.ERR_BLOCK
    with pytest.raises(ValueError) as e:
        oracle.commit_plan(4, 2, [5, 6], 0, 4, 8, 4)
    assert e.value.args[0] == oracle.ERR_SEQPOS


# ------------------------------------------------------------ batch level
def _batch(HK=2, HV=4, K=8, V=8, W=4, windows=(4, 2, 0, 3, 2), slots=(0, 2, -1, 3, -1), seed=0):
    g = np.random.default_rng(seed)
    B = len(windows)
    starts = np.cumsum([0] + list(windows[:-1])).astype(np.int32)
    T = int(sum(windows))
    return dict(q=g.normal(size=(T, HK, K)), k=g.normal(size=(T, HK, K)),
                v=g.normal(size=(T, HV, V)), a=g.normal(size=(T, HV)), b=g.normal(size=(T, HV)),
                A_log=g.uniform(0, math.log(16), HV), dt_bias=g.uniform(-1, 1, HV),
                token_start=starts, window_len=np.array(windows, np.int32),
                pool=g.normal(0, 0.1, (5, HV, V, K)), slot_table=np.array(slots, np.int32),
                max_window=W)


def test_gqa_uses_consecutive_key_groups():
    # HV = 2 * HK: value heads 2j and 2j+1 read key head j.  Expanding the
    # keys/queries to one per value head with repeat_interleave must give
    # the same result as the grouped run.
    d = _batch()
    grouped = oracle.spec_verify(**d)
    e = dict(d)
    e["q"] = np.repeat(d["q"], 2, axis=1)
    e["k"] = np.repeat(d["k"], 2, axis=1)
    expanded = oracle.spec_verify(**e)
    for key in ("out", "rec_u", "rec_k", "rec_g"):
        assert np.array_equal(grouped[key], expanded[key], equal_nan=True), key
    e["q"] = np.tile(d["q"], (1, 2, 1))        # the other plausible mapping differs
    e["k"] = np.tile(d["k"], (1, 2, 1))
    tiled = oracle.spec_verify(**e)
    assert not np.allclose(np.nan_to_num(grouped["out"]), np.nan_to_num(tiled["out"]))


def test_verify_writes_only_live_rows():
    d = _batch()
    r = oracle.spec_verify(**d, snapshots=True)
    assert np.all(r["row_err"] == 0)
    starts, windows = d["token_start"], d["window_len"]
    for row, (s, w) in enumerate(zip(starts, windows)):
        live = w > 0 and d["slot_table"][row] >= 0
        blk = r["out"][s:s + w]
        assert np.all(np.isfinite(blk)) if live else np.all(np.isnan(blk))
        rec = r["rec_u"][row, :, :w]
        assert np.all(np.isfinite(rec)) if live else np.all(np.isnan(rec))
        assert np.all(np.isnan(r["rec_u"][row, :, w:]))      # beyond the window
        assert np.all(np.isnan(r["snaps"][row, w:]))


def test_commit_equals_native_snapshot_states():
    # Commit after n accepted tokens (replay from records) equals the
    # recomputed state after n tokens, for every n, and writes only the
    # final slot; slots of null rows stay unchanged.
    d = _batch()
    B = len(d["window_len"])
    v = oracle.spec_verify(**d, snapshots=True)
    for n_first in range(0, 5):
        acc = np.array([n_first, 2, 0, 1, 2], np.int32)
        pools, err = oracle.replay_commit(
            pools=d["pool"][None], rec_u=v["rec_u"][None], rec_k=v["rec_k"][None],
            rec_g=v["rec_g"][None], window_len=d["window_len"], accepted_len=acc,
            slot_table=d["slot_table"], max_window=4)
        assert np.all(err == 0)
        expect = d["pool"].copy()
        for r in range(B):
            s, n = d["slot_table"][r], acc[r]
            if s >= 0 and n > 0:
                expect[s] = v["snaps"][r, n - 1]
        assert np.allclose(pools[0], expect, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("Bk,W", [(4, 4), (3, 6), (2, 5)])
def test_align_commit_writes_snapshots_into_boundary_and_final_slots(Bk, W):
    # Align mode: the commit stores the state after p - p0 tokens into the
    # slot of every block boundary p crossed, and the state after n tokens
    # into the final slot.  Which slot gets which state comes from the
    # token-by-token block walk (_brute_force_writes), the states from the
    # oracle's own recompute (native snapshots): the commit replays records,
    # so a wrong slot, a boundary off by one, a boundary fold that started
    # from an already-written slot or a dropped final write all fail here.
    # Rows cover every checkpoint offset p0 % Bk and every n in 1..W; when
    # p0 % Bk != 0 and the window crosses a boundary, the boundary slot is
    # the row's own checkpoint slot.
    g = np.random.default_rng(7 + Bk)
    HK, HV, K, V = 1, 2, 8, 8
    combos = [(r, n) for r in range(Bk) for n in range(1, W + 1)]
    B = len(combos)
    seq_pos = np.array([Bk * (1 + i % 3) + r for i, (r, _) in enumerate(combos)], np.int32)
    acc = np.array([n for _, n in combos], np.int32)
    windows = np.full(B, W, np.int32)
    stride = int((seq_pos.max() + W - 1) // Bk + 1)
    table = np.full((B, stride), -1, np.int32)
    nxt = 0
    for r in range(B):
        for col in range((seq_pos[r] - 1) // Bk, (seq_pos[r] + W - 1) // Bk + 1):
            table[r, col] = nxt
            nxt += 1
    T = B * W
    d = dict(q=g.normal(size=(T, HK, K)), k=g.normal(size=(T, HK, K)), v=g.normal(size=(T, HV, V)),
             a=g.normal(size=(T, HV)), b=g.normal(size=(T, HV)), A_log=g.uniform(0, 2.7, HV),
             dt_bias=g.uniform(-1, 1, HV), token_start=np.arange(0, T, W, dtype=np.int32),
             window_len=windows, pool=g.normal(0, 0.1, (nxt, HV, V, K)), slot_table=table,
             seq_pos=seq_pos, block_size=Bk, max_window=W)
    v = oracle.spec_verify(**d, snapshots=True)
    assert np.all(v["row_err"] == 0)
    pools, err = oracle.replay_commit(
        pools=d["pool"][None], rec_u=v["rec_u"][None], rec_k=v["rec_k"][None],
        rec_g=v["rec_g"][None], window_len=windows, accepted_len=acc, slot_table=table,
        seq_pos=seq_pos, block_size=Bk, max_window=W)
    assert np.all(err == 0)
    expect = d["pool"].copy()
    src_reused = 0
    for r in range(B):
        p0, n = int(seq_pos[r]), int(acc[r])
        cols = _brute_force_writes(p0, n, Bk)
        for col, ntok in cols.items():
            expect[table[r, col]] = v["snaps"][r, ntok - 1]
        src_reused += int((p0 - 1) // Bk in cols)
    assert src_reused > 0, "no row whose boundary slot is its checkpoint slot"
    assert np.allclose(pools[0], expect, rtol=1e-12, atol=1e-14)
    # slots no row writes keep the checkpoint bit for bit
    written = {int(table[r, c]) for r in range(B)
               for c in _brute_force_writes(int(seq_pos[r]), int(acc[r]), Bk)}
    for s in range(nxt):
        if s not in written:
            assert np.array_equal(pools[0][s], d["pool"][s])


def test_config_tiny_checkpoint_untouched_and_consistent():
    from spec_decode_recurrent_gb300 import workloads
    sb = workloads.tiny()
    pool = sb.pools[0].clone()
    r = oracle.spec_verify(q=sb.q[0], k=sb.k[0], v=sb.v[0], a=sb.a[0], b=sb.b[0],
                           A_log=sb.A_log[0], dt_bias=sb.dt_bias[0],
                           token_start=sb.token_start, window_len=sb.window_len,
                           pool=sb.pools[0], slot_table=sb.slot_table, max_window=sb.W,
                           snapshots=True)
    assert torch.equal(pool.view(torch.int32), sb.pools[0].view(torch.int32))
    assert np.all(np.isfinite(r["out"])) and np.all(np.isfinite(r["rec_u"]))
    # The normalised key in the record has unit norm (up to eps).
    assert np.allclose(np.linalg.norm(r["rec_k"], axis=-1), 1.0, atol=1e-6)


# ------------------------------------------------------------- bf16 grid
def test_bf16_ulp_values():
    assert bf16_ulp(1.0) == 2.0 ** -7
    assert bf16_ulp(1.99) == 2.0 ** -7
    assert bf16_ulp(2.0) == 2.0 ** -6
    assert bf16_ulp(0.1) == 2.0 ** -11
    assert bf16_ulp(-3.0) == 2.0 ** -6
    assert bf16_ulp(0.0) == 2.0 ** -133


def test_bf16_ulp_is_grid_spacing():
    x = torch.tensor(rng.normal(0, 0.3, 4096), dtype=torch.float32)
    xb = x.to(torch.bfloat16)
    nxt = (xb.view(torch.int16) + 1).view(torch.bfloat16)   # next value away from zero
    spacing = (nxt.double() - xb.double()).abs().numpy()
    assert np.array_equal(spacing, bf16_ulp(xb.double().numpy()))
    assert np.all(np.abs(xb.double().numpy() - x.double().numpy())
                  <= 0.5 * bf16_ulp(xb.double().numpy()) + 0.0)


# ------------------------------------------------------- grouped commit
def test_grouped_commit_reduces_to_per_layer_commits():
    # Layers in KV-cache groups, each group with its own [batch, stride]
    # slot table: the grouped commit must equal committing each layer on
    # its own with its group's table.
    g = np.random.default_rng(21)
    L, G, B, HV, K, V, W, slots = 6, 3, 4, 2, 8, 8, 4, 12
    pools = g.normal(0, 0.1, (L, slots, HV, V, K))
    rec_u, rec_k = g.normal(size=(L, B, HV, W, V)), g.normal(size=(L, B, HV, W, K))
    rec_g = g.uniform(0.1, 1.0, (L, B, HV, W))
    win = np.array([4, 3, 0, 4], np.int32)
    acc = np.array([2, 3, 0, 4], np.int32)
    tables = np.stack([g.permutation(slots)[:B].reshape(B, 1) for _ in range(G)]).astype(np.int32)
    tables[1, 3, 0] = -1                        # a null slot in one group only
    layer_group = np.array([0, 1, 2, 0, 1, 2], np.int32)
    got, err = oracle.replay_commit(pools=pools, rec_u=rec_u, rec_k=rec_k, rec_g=rec_g,
                                    window_len=win, accepted_len=acc, slot_table=tables,
                                    layer_group=layer_group, max_window=W)
    assert np.all(err == 0)
    for l in range(L):
        one, e1 = oracle.replay_commit(pools=pools[l:l + 1], rec_u=rec_u[l:l + 1],
                                       rec_k=rec_k[l:l + 1], rec_g=rec_g[l:l + 1],
                                       window_len=win, accepted_len=acc,
                                       slot_table=tables[layer_group[l]], max_window=W)
        assert np.array_equal(got[l], one[0])
    # one group whose table every layer shares is the plain all-layer commit
    plain, _ = oracle.replay_commit(pools=pools, rec_u=rec_u, rec_k=rec_k, rec_g=rec_g,
                                    window_len=win, accepted_len=acc, slot_table=tables[0],
                                    max_window=W)
    same, _ = oracle.replay_commit(pools=pools, rec_u=rec_u, rec_k=rec_k, rec_g=rec_g,
                                   window_len=win, accepted_len=acc,
                                   slot_table=np.stack([tables[0]] * G),
                                   layer_group=layer_group, max_window=W)
    assert np.array_equal(plain, same)


# ------------------------------------------------------ short-conv commit
def _shift_register(old, xs):
    """Brute force: push the accepted inputs one at a time into a shift
    register that drops its oldest entry."""
    state = list(old)
    for x in xs:
        state = state[1:] + [x]
    return state


@pytest.mark.parametrize("SL", [1, 3, 5])
def test_conv_commit_matches_shift_register(SL):
    g = np.random.default_rng(SL)
    C, W, B, slots = 6, 6, 5, 9
    win = np.array([6, 4, 0, 1, 6], np.int32)
    acc = np.array([6, 2, 0, 1, 0], np.int32)
    starts = np.array([0, 7, 11, 11, 13], np.int32)       # rows with gaps, any order
    T = 20
    pools = g.normal(size=(1, slots, C, SL))
    inputs = g.normal(size=(1, T, C))
    table = np.array([[3], [0], [-1], [5], [7]], np.int32)
    got, err = oracle.conv_commit(pools=pools, inputs=inputs, token_start=starts, window_len=win,
                                  accepted_len=acc, slot_table=table, max_window=W)
    assert np.all(err == 0)
    expect = pools.copy()
    for r in range(B):
        s = table[r, 0]
        if s < 0 or acc[r] == 0:
            continue
        for c in range(C):
            xs = [inputs[0, starts[r] + i, c] for i in range(acc[r])]
            expect[0, s, c] = _shift_register(list(pools[0, s, c]), xs)
    assert np.array_equal(got, expect)


def test_conv_commit_composes_and_aligns():
    # committing n1 tokens and then n2 more from the new checkpoint equals
    # committing n1 + n2 at once; align mode writes each block's last state
    g = np.random.default_rng(3)
    C, SL, W, slots = 4, 3, 6, 8
    pools = g.normal(size=(1, slots, C, SL))
    inputs = g.normal(size=(1, 12, C))
    one, _ = oracle.conv_commit(pools=pools, inputs=inputs, token_start=[0], window_len=[5],
                                accepted_len=[5], slot_table=[[2]], max_window=W)
    a, _ = oracle.conv_commit(pools=pools, inputs=inputs, token_start=[0], window_len=[2],
                              accepted_len=[2], slot_table=[[2]], max_window=W)
    b, _ = oracle.conv_commit(pools=a, inputs=inputs, token_start=[2], window_len=[3],
                              accepted_len=[3], slot_table=[[2]], max_window=W)
    assert np.array_equal(one, b)
    # align: block 4, checkpoint after 5 tokens (column 1), 5 accepted -> the
    # state after token 8 goes to column 1, after token 10 to column 2
    table = np.array([[-1, 4, 6, -1]], np.int32)
    al, err = oracle.conv_commit(pools=pools, inputs=inputs, token_start=[0], window_len=[6],
                                 accepted_len=[5], slot_table=table, seq_pos=[5], block_size=4,
                                 max_window=W)
    assert np.all(err == 0)
    s3, _ = oracle.conv_commit(pools=pools, inputs=inputs, token_start=[0], window_len=[6],
                               accepted_len=[3], slot_table=[[4]], max_window=W)
    s5, _ = oracle.conv_commit(pools=pools, inputs=inputs, token_start=[0], window_len=[6],
                               accepted_len=[5], slot_table=[[4]], max_window=W)
    assert np.array_equal(al[0, 4], s3[0, 4]) and np.array_equal(al[0, 6], s5[0, 4])
