"""Pins for the oracle's per-channel-decay (KDA) functions: facts fixed by
the reading of the method and by mathematics, not by re-running the
oracle's own formulas.

Reading (the pages name KDA as the protocol's origin but print no formula):
the decay of the gated delta rule becomes a vector over the K key channels,
H = S diag(alpha_t), and the replay record keeps the whole gate vector.
Each pin is chosen so that a plausible slip -- the decay applied along the
value rows, a per-head instead of per-channel bias, a wrong gate offset in
the batch layout -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit(K=8, V=12, w=5, seed=0):
    g = np.random.default_rng(seed)
    return dict(S0=g.normal(0, 0.1, (V, K)), q=g.normal(size=(w, K)), k=g.normal(size=(w, K)),
                v=g.normal(size=(w, V)), a=g.normal(size=(w, K)), b=g.normal(size=w),
                A_log=float(g.uniform(0, math.log(16))), dt_bias=g.uniform(-1, 1, K))


def _run(u, **over):
    d = dict(u, **over)
    return oracle.kda_window(d["S0"], d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                             d["dt_bias"])


def test_kda_worked_example_golden():
    with open(os.path.join(GOLDEN, "kda_worked_example_two_tokens.json")) as f:
        g = json.load(f)
    r = oracle.kda_window(g["S0"], g["q"], g["k"], g["v"], g["a"], g["b"], g["A_log"],
                          g["dt_bias"])
    tol = g["atol"]
    assert np.allclose(r["alpha"], g["expect_alpha"], rtol=0, atol=1e-15)
    assert np.allclose(r["u"], g["expect_u"], rtol=0, atol=tol)
    assert np.allclose(r["states"], g["expect_states"], rtol=0, atol=tol)
    assert np.allclose(r["o"], g["expect_o"], rtol=0, atol=tol)


def test_kda_decay_closed_form_per_channel():
    # alpha_t[j] = (1 + e^{a_t[j] + dt_bias[j]})^(-exp(A_log)): a different
    # evaluation route of exp(-exp(A_log) softplus(.)), channel by channel.
    u = _unit(seed=1)
    r = _run(u)
    c = math.exp(u["A_log"])
    expect = (1.0 + np.exp(u["a"] + u["dt_bias"][None, :])) ** (-c)
    assert np.allclose(r["alpha"], expect, rtol=1e-12, atol=0)


def test_kda_uniform_channels_reproduce_the_scalar_gate_bit_for_bit():
    # Every channel given the scalar gate's input: the KDA recurrence, its
    # records and its commit equal the scalar-gate (GDN) oracle exactly.
    g = np.random.default_rng(2)
    HK, HV, K, V, W = 2, 4, 8, 6, 4
    windows = np.array([4, 2, 0, 3], np.int32)
    B = len(windows)
    T = int(windows.sum())
    starts = np.concatenate([[0], np.cumsum(windows)[:-1]]).astype(np.int32)
    a = g.normal(size=(T, HV))
    dt = g.uniform(-1, 1, HV)
    common = dict(q=g.normal(size=(T, HK, K)), k=g.normal(size=(T, HK, K)),
                  v=g.normal(size=(T, HV, V)), b=g.normal(size=(T, HV)),
                  A_log=g.uniform(0, 2.7, HV), token_start=starts, window_len=windows,
                  pool=g.normal(0, 0.1, (6, HV, V, K)),
                  slot_table=np.array([0, 3, -1, 5], np.int32), max_window=W)
    scal = oracle.spec_verify(a=a, dt_bias=dt, snapshots=True, **common)
    kda = oracle.kda_spec_verify(a=np.repeat(a[:, :, None], K, axis=2),
                                 dt_bias=np.repeat(dt[:, None], K, axis=1), snapshots=True,
                                 **common)
    for key in ("out", "rec_u", "rec_k", "snaps"):
        assert np.array_equal(scal[key], kda[key], equal_nan=True), key
    assert np.array_equal(np.repeat(scal["rec_g"][..., None], K, axis=3), kda["rec_g"],
                          equal_nan=True)
    acc = np.array([3, 2, 0, 1], np.int32)
    p_s, e_s = oracle.replay_commit(pools=common["pool"][None], rec_u=scal["rec_u"][None],
                                    rec_k=scal["rec_k"][None], rec_g=scal["rec_g"][None],
                                    window_len=windows, accepted_len=acc,
                                    slot_table=common["slot_table"], max_window=W)
    p_k, e_k = oracle.kda_replay_commit(pools=common["pool"][None], rec_u=kda["rec_u"][None],
                                        rec_k=kda["rec_k"][None], rec_g=kda["rec_g"][None],
                                        window_len=windows, accepted_len=acc,
                                        slot_table=common["slot_table"], max_window=W)
    assert np.array_equal(p_s, p_k) and np.array_equal(e_s, e_k)


def test_kda_identity_gate_leaves_state_unchanged():
    u = _unit(seed=3)
    w = len(u["b"])
    r = _run(u, a=np.full((w, 8), -1e4), b=np.full(w, -1e4))
    for t in range(w):
        assert np.array_equal(r["states"][t], u["S0"])                 # bit for bit
        assert np.allclose(r["o"][t], u["S0"] @ oracle.l2norm(u["q"][t]), rtol=1e-13, atol=1e-15)
    assert np.array_equal(r["u"], np.zeros_like(r["u"]))
    assert np.array_equal(r["alpha"], np.ones((w, 8)))


@pytest.mark.parametrize("K,V", [(8, 8), (8, 12), (16, 4)])
def test_kda_pure_decay_scales_key_columns(K, V):
    # beta = 0: S_t = S0 diag(prod_{s<=t} alpha_s): column j (key channel)
    # scaled by its own running product, rows untouched.
    u = _unit(K=K, V=V, w=4, seed=4)
    r = _run(u, b=np.full(4, -1e4))
    c = math.exp(u["A_log"])
    prod = np.ones(K)
    for t in range(4):
        prod = prod * (1.0 + np.exp(u["a"][t] + u["dt_bias"])) ** (-c)
        assert np.allclose(r["states"][t], u["S0"] * prod[None, :], rtol=1e-12, atol=1e-300)


def test_kda_write_invariant_full_strength():
    # beta = 1: S_t khat_t = v_t after every token (|khat| = 1 up to eps).
    u = _unit(K=32, V=24, w=6, seed=5)
    r = _run(u, b=np.full(6, 1e4))
    for t in range(6):
        assert np.allclose(r["states"][t] @ oracle.l2norm(u["k"][t]), u["v"][t], rtol=0, atol=1e-6)


def test_kda_replay_from_record_equals_recompute():
    u = _unit(K=16, V=16, w=6, seed=6)
    r = _run(u)
    for n in range(1, 7):
        S = oracle.kda_replay(u["S0"], r["u"][:n], r["khat"][:n], r["alpha"][:n])
        assert np.allclose(S, r["states"][n - 1], rtol=1e-12, atol=1e-14)


def _batch(seed=7, block_size=0):
    g = np.random.default_rng(seed)
    HK, HV, K, V, W = 1, 2, 8, 6, 4
    windows = np.array([4, 3, 4, 0, 2], np.int32)
    B = len(windows)
    T = int(windows.sum()) + 3
    starts = np.array([3, 0, 7, 0, 11], np.int32)          # rows out of order, gaps
    if block_size:
        seq_pos = np.array([4, 5, 7, 1, 2], np.int32)
        table = np.full((B, int((seq_pos.max() + W - 1) // block_size) + 1), -1, np.int32)
        nxt = 0
        for r in range(B):
            for col in range((seq_pos[r] - 1) // block_size,
                             (seq_pos[r] + W - 1) // block_size + 1):
                table[r, col] = nxt
                nxt += 1
    else:
        seq_pos = None
        table = np.array([[2], [0], [4], [-1], [1]], np.int32)
        nxt = 6
    return dict(q=g.normal(size=(T, HK, K)), k=g.normal(size=(T, HK, K)),
                v=g.normal(size=(T, HV, V)), a=g.normal(size=(T, HV, K)),
                b=g.normal(size=(T, HV)), A_log=g.uniform(0, 2.7, HV),
                dt_bias=g.uniform(-1, 1, (HV, K)), token_start=starts, window_len=windows,
                pool=g.normal(0, 0.1, (max(nxt, 1), HV, V, K)), slot_table=table,
                seq_pos=seq_pos, block_size=block_size, max_window=W)


def test_kda_batch_layout_matches_unit_windows():
    # Every (row, value head) of the batch equals the one-unit window run on
    # that unit's slices: pins the gate offsets (a [T, HV, K], dt_bias
    # [HV, K]), the GQA key head, the token rows and the record layout.
    d = _batch()
    r = oracle.kda_spec_verify(snapshots=True, **d)
    assert np.all(r["row_err"] == 0)
    for row in range(len(d["window_len"])):
        w, t0, slot = int(d["window_len"][row]), int(d["token_start"][row]), int(d["slot_table"][row, 0])
        for h in range(2):
            if w == 0 or slot < 0:
                assert np.all(np.isnan(r["rec_g"][row, h]))
                continue
            sl = slice(t0, t0 + w)
            u = oracle.kda_window(d["pool"][slot, h], d["q"][sl, 0], d["k"][sl, 0], d["v"][sl, h],
                                  d["a"][sl, h], d["b"][sl, h], d["A_log"][h], d["dt_bias"][h])
            assert np.array_equal(r["out"][sl, h], u["o"])
            assert np.array_equal(r["rec_u"][row, h, :w], u["u"])
            assert np.array_equal(r["rec_g"][row, h, :w], u["alpha"])
            assert np.array_equal(r["snaps"][row, :w, h], u["states"])
            assert np.all(np.isnan(r["rec_g"][row, h, w:]))


@pytest.mark.parametrize("block_size", [0, 2])
def test_kda_commit_equals_native_snapshot_states(block_size):
    # The commit replays records: after n accepted tokens the final slot
    # holds the recomputed state after n tokens and, in align mode, every
    # crossed boundary's slot the state after p - p0 tokens.
    d = _batch(seed=8, block_size=block_size)
    v = oracle.kda_spec_verify(snapshots=True, **d)
    acc = np.array([3, 3, 4, 0, 1], np.int32)
    pools, err = oracle.kda_replay_commit(
        pools=d["pool"][None], rec_u=v["rec_u"][None], rec_k=v["rec_k"][None],
        rec_g=v["rec_g"][None], window_len=d["window_len"], accepted_len=acc,
        slot_table=d["slot_table"], seq_pos=d["seq_pos"], block_size=block_size, max_window=4)
    assert np.all(err == 0)
    expect = d["pool"].copy()
    for r in range(len(acc)):
        n = int(acc[r])
        if n == 0 or d["window_len"][r] == 0:
            continue
        if block_size == 0:
            if d["slot_table"][r, 0] >= 0:
                expect[d["slot_table"][r, 0]] = v["snaps"][r, n - 1]
            continue
        p0 = int(d["seq_pos"][r])
        for x in range(p0 + 1, p0 + n + 1):               # block of each accepted token
            expect[d["slot_table"][r, (x - 1) // block_size]] = v["snaps"][r, x - p0 - 1]
    assert np.allclose(pools[0], expect, rtol=1e-12, atol=1e-14)
