"""fp64 CPU oracle for GDN speculative verify and replay commit.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``spec_decode_recurrent_gb300``) never imports it, and it never
imports the product.  The arithmetic lives in ``gdn_oracle.c`` (plain fp64
loops, token by token); this module only compiles it with gcc, converts
arrays to float64 and marshals pointers.

Parity pins for every function here are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

# Row error bits (same contract as the library's optional error word).
ERR_WINDOW, ERR_ACCEPTED, ERR_SLOT, ERR_BLOCK, ERR_SEQPOS, ERR_TOKENS = 1, 2, 4, 8, 16, 32

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)
_i = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into a shared object (gcc, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.gdn_oracle_softplus.restype = ctypes.c_double
            lib.gdn_oracle_softplus.argtypes = [ctypes.c_double]
            lib.gdn_oracle_decay.restype = ctypes.c_double
            lib.gdn_oracle_decay.argtypes = [ctypes.c_double] * 3
            lib.gdn_oracle_beta.restype = ctypes.c_double
            lib.gdn_oracle_beta.argtypes = [ctypes.c_double]
            lib.gdn_oracle_l2norm.restype = None
            lib.gdn_oracle_l2norm.argtypes = [_i, _D, _D]
            lib.gdn_oracle_window.restype = None
            lib.gdn_oracle_window.argtypes = [_i, _i, _i, _D, _D, _D, _D, _D, _D,
                                              ctypes.c_double, ctypes.c_double,
                                              _D, _D, _D, _D, _D]
            lib.gdn_oracle_replay.restype = None
            lib.gdn_oracle_replay.argtypes = [_i, _i, _i, _D, _D, _D, _D]
            lib.gdn_oracle_source_slot.restype = _i
            lib.gdn_oracle_source_slot.argtypes = [_i, _I, _i, _i, _i, _i, _i]
            lib.gdn_oracle_commit_plan.restype = _i
            lib.gdn_oracle_commit_plan.argtypes = [_i, _i, _I, _i, _i, _i, _i, _i,
                                                   _I, _I, _I, _i]
            lib.gdn_oracle_spec_verify.restype = _i
            lib.gdn_oracle_spec_verify.argtypes = (
                [_i] * 8 + [_D] * 7 + [_I, _I, _D, _I, _i, _I, _i] + [_D] * 5 + [_I])
            lib.gdn_oracle_replay_commit.restype = _i
            lib.gdn_oracle_replay_commit.argtypes = (
                [_i] * 7 + [_D] * 5 + [_I, _I, _I, _i, _I, _i, _I])
            lib.gdn_oracle_replay_commit_grouped.restype = _i
            lib.gdn_oracle_replay_commit_grouped.argtypes = (
                [_i] * 7 + [_D] * 5 + [_I, _I, _I, _i, ctypes.c_long, _I, _i, _I, _i, _I])
            lib.gdn_oracle_conv_commit.restype = _i
            lib.gdn_oracle_conv_commit.argtypes = (
                [_i] * 7 + [_D] * 3 + [_I, _I, _I, _I, _i, ctypes.c_long, _I, _i, _I, _i, _I])
            lib.gdn_oracle_kda_window.restype = None
            lib.gdn_oracle_kda_window.argtypes = [_i, _i, _i, _D, _D, _D, _D, _D, _D,
                                                  ctypes.c_double, _D, _D, _D, _D, _D, _D]
            lib.gdn_oracle_kda_replay.restype = None
            lib.gdn_oracle_kda_replay.argtypes = [_i, _i, _i, _D, _D, _D, _D]
            lib.gdn_oracle_kda_spec_verify.restype = _i
            lib.gdn_oracle_kda_spec_verify.argtypes = (
                [_i] * 8 + [_D] * 7 + [_I, _I, _D, _I, _i, _I, _i] + [_D] * 5 + [_I])
            lib.gdn_oracle_kda_replay_commit.restype = _i
            lib.gdn_oracle_kda_replay_commit.argtypes = (
                [_i] * 7 + [_D] * 5 + [_I, _I, _I, _i, _I, _i, _I])
            lib.gdn_oracle_num_threads.restype = _i
            lib.gdn_oracle_num_threads.argtypes = []
            lib.gdn_oracle_set_num_threads.restype = None
            lib.gdn_oracle_set_num_threads.argtypes = [_i]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Contiguous float64 copy of a numpy array or CPU torch tensor (exact widening)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dp(a):
    return None if a is None else a.ctypes.data_as(_D)


def _ip(a):
    return None if a is None else a.ctypes.data_as(_I)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().gdn_oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on."""
    _load().gdn_oracle_set_num_threads(int(n))


# ---------------------------------------------------------------- scalars
def softplus(x: float) -> float:
    return _load().gdn_oracle_softplus(float(x))


def decay(a: float, A_log: float, dt_bias: float) -> float:
    """alpha = exp(-exp(A_log) * softplus(a + dt_bias))."""
    return _load().gdn_oracle_decay(float(a), float(A_log), float(dt_bias))


def beta(b: float) -> float:
    """beta = sigmoid(b)."""
    return _load().gdn_oracle_beta(float(b))


def l2norm(x) -> np.ndarray:
    x = _f64(x).reshape(-1)
    out = np.empty_like(x)
    _load().gdn_oracle_l2norm(x.size, _dp(x), _dp(out))
    return out


# ------------------------------------------------------------ one unit
def window(S0, q, k, v, a, b, A_log: float, dt_bias: float):
    """Verify window of one (request, value head) unit.

    S0 [V, K]; q, k [w, K]; v [w, V]; a, b [w].
    Returns dict with o [w, V], u [w, V], khat [w, K], alpha [w] and
    states [w, V, K] (state after each token).
    """
    S0 = _f64(S0)
    V, K = S0.shape
    q, k, v, a, b = (_f64(t) for t in (q, k, v, a, b))
    w = a.shape[0]
    o = np.empty((w, V)); u = np.empty((w, V)); kh = np.empty((w, K))
    al = np.empty(w); st = np.empty((w, V, K))
    _load().gdn_oracle_window(K, V, w, _dp(S0), _dp(q), _dp(k), _dp(v), _dp(a),
                              _dp(b), float(A_log), float(dt_bias), _dp(o), _dp(u),
                              _dp(kh), _dp(al), _dp(st))
    return {"o": o, "u": u, "khat": kh, "alpha": al, "states": st}


def replay(S0, u, khat, alpha) -> np.ndarray:
    """Fold len(alpha) records into a copy of S0 [V, K]; returns the new state."""
    S = _f64(S0).copy()
    V, K = S.shape
    u, khat, alpha = _f64(u), _f64(khat), _f64(alpha).reshape(-1)
    _load().gdn_oracle_replay(K, V, alpha.shape[0], _dp(S), _dp(u), _dp(khat), _dp(alpha))
    return S


def source_slot(window_len, table_row, seq_pos, block_size, num_slots, max_window):
    """Checkpoint slot of a row (>= -1) or -(1 + error bits)."""
    row = _i32(table_row).reshape(-1)
    return int(_load().gdn_oracle_source_slot(int(window_len), _ip(row), row.size,
                                              int(seq_pos), int(block_size),
                                              int(num_slots), int(max_window)))


def commit_plan(window_len, accepted_len, table_row, seq_pos, block_size,
                num_slots, max_window):
    """Commit plan of one row.

    Returns (src_slot, [(slot, tokens_folded), ...]) with the final write
    first, or raises ValueError(error_bits) for a malformed row.
    """
    row = _i32(table_row).reshape(-1)
    src = (ctypes.c_int32 * 1)()
    cap = 2 + int(max_window)
    slots = (ctypes.c_int32 * cap)()
    ntok = (ctypes.c_int32 * cap)()
    nw = _load().gdn_oracle_commit_plan(int(window_len), int(accepted_len), _ip(row),
                                        row.size, int(seq_pos), int(block_size),
                                        int(num_slots), int(max_window),
                                        ctypes.cast(src, _I), ctypes.cast(slots, _I),
                                        ctypes.cast(ntok, _I), cap)
    if nw < 0:
        raise ValueError(-nw - 1)
    return int(src[0]), [(int(slots[i]), int(ntok[i])) for i in range(nw)]


# ------------------------------------------------------------- batches
def spec_verify(*, q, k, v, a, b, A_log, dt_bias, token_start, window_len, pool,
                slot_table, seq_pos=None, block_size=0, max_window, snapshots=False,
                out=None, rec_u=None, rec_k=None, rec_g=None, snaps=None):
    """Verify for one layer (plus native per-draft snapshots if requested).

    q, k [T, HK, K]; v [T, HV, V]; a, b [T, HV]; A_log, dt_bias [HV];
    pool [num_slots, HV, V, K]; slot_table [B, stride].
    Outputs are float64 arrays; pass pre-filled arrays (e.g. NaN) to see
    which entries are written.  Returns dict with out, rec_u, rec_k, rec_g,
    snaps (or None) and row_err.
    """
    q, k, v, a, b = (_f64(t) for t in (q, k, v, a, b))
    A_log, dt_bias, pool = _f64(A_log), _f64(dt_bias), _f64(pool)
    token_start, window_len = _i32(token_start), _i32(window_len)
    slot_table = _i32(slot_table)
    if slot_table.ndim == 1:
        slot_table = slot_table.reshape(-1, 1)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    B = window_len.shape[0]
    W = int(max_window)
    num_slots = pool.shape[0]
    sp = None if seq_pos is None else _i32(seq_pos)
    nan = np.nan
    out = np.full((T, HV, V), nan) if out is None else out
    rec_u = np.full((B, HV, W, V), nan) if rec_u is None else rec_u
    rec_k = np.full((B, HV, W, K), nan) if rec_k is None else rec_k
    rec_g = np.full((B, HV, W), nan) if rec_g is None else rec_g
    if snapshots and snaps is None:
        snaps = np.full((B, W, HV, V, K), nan)
    row_err = np.zeros(B, dtype=np.int32)
    rc = _load().gdn_oracle_spec_verify(
        HK, HV, K, V, W, B, T, num_slots, _dp(q), _dp(k), _dp(v), _dp(a), _dp(b),
        _dp(A_log), _dp(dt_bias), _ip(token_start), _ip(window_len), _dp(pool),
        _ip(slot_table), slot_table.shape[1], _ip(sp), int(block_size),
        _dp(out), _dp(rec_u), _dp(rec_k), _dp(rec_g), _dp(snaps if snapshots else None),
        _ip(row_err))
    if rc != 0:
        raise ValueError(f"oracle spec_verify rejected the shape ({rc})")
    return {"out": out, "rec_u": rec_u, "rec_k": rec_k, "rec_g": rec_g,
            "snaps": snaps if snapshots else None, "row_err": row_err}


def replay_commit(*, pools, rec_u, rec_k, rec_g, window_len, accepted_len, slot_table,
                  seq_pos=None, block_size=0, max_window, layer_group=None):
    """All-layer commit from records.

    pools [L, num_slots, HV, V, K]; rec_u [L, B, HV, W, V]; rec_k [L, B, HV, W, K];
    rec_g [L, B, HV, W].  slot_table [B, stride], or [G, B, stride] with
    layer_group [L] naming each layer's group.  Returns (new_pools float64,
    row_err).
    """
    pools_in = _f64(pools)
    pools_out = pools_in.copy()
    rec_u, rec_k, rec_g = _f64(rec_u), _f64(rec_k), _f64(rec_g)
    window_len, accepted_len = _i32(window_len), _i32(accepted_len)
    slot_table = _i32(slot_table)
    if slot_table.ndim == 1:
        slot_table = slot_table.reshape(-1, 1)
    if slot_table.ndim == 2:
        slot_table = slot_table[None]
    G = slot_table.shape[0]
    lg = None if layer_group is None else _i32(layer_group)
    L, num_slots, HV, V, K = pools_in.shape
    B = window_len.shape[0]
    sp = None if seq_pos is None else _i32(seq_pos)
    row_err = np.zeros(B, dtype=np.int32)
    rc = _load().gdn_oracle_replay_commit_grouped(
        L, HV, K, V, int(max_window), B, num_slots, _dp(pools_in), _dp(pools_out),
        _dp(rec_u), _dp(rec_k), _dp(rec_g), _ip(window_len), _ip(accepted_len),
        _ip(lg), G, slot_table.shape[1] * slot_table.shape[2], _ip(slot_table),
        slot_table.shape[2], _ip(sp), int(block_size), _ip(row_err))
    if rc != 0:
        raise ValueError(f"oracle replay_commit rejected the shape ({rc})")
    return pools_out, row_err


def conv_commit(*, pools, inputs, token_start, window_len, accepted_len, slot_table,
                seq_pos=None, block_size=0, max_window, layer_group=None):
    """Short-conv state commit.

    pools [L, num_slots, C, SL] (last SL conv inputs per channel, oldest
    first); inputs [L, T, C]; slot_table [B, stride] or [G, B, stride] with
    layer_group [L].  Returns (new_pools float64, row_err).
    """
    pools_in = _f64(pools)
    pools_out = pools_in.copy()
    inputs = _f64(inputs)
    token_start, window_len, accepted_len = _i32(token_start), _i32(window_len), _i32(accepted_len)
    slot_table = _i32(slot_table)
    if slot_table.ndim == 1:
        slot_table = slot_table.reshape(-1, 1)
    if slot_table.ndim == 2:
        slot_table = slot_table[None]
    G = slot_table.shape[0]
    lg = None if layer_group is None else _i32(layer_group)
    L, num_slots, C, SL = pools_in.shape
    T = inputs.shape[1]
    B = window_len.shape[0]
    sp = None if seq_pos is None else _i32(seq_pos)
    row_err = np.zeros(B, dtype=np.int32)
    rc = _load().gdn_oracle_conv_commit(
        L, C, SL, int(max_window), B, T, num_slots, _dp(pools_in), _dp(pools_out), _dp(inputs),
        _ip(token_start), _ip(window_len), _ip(accepted_len), _ip(lg), G,
        slot_table.shape[1] * slot_table.shape[2], _ip(slot_table), slot_table.shape[2], _ip(sp),
        int(block_size), _ip(row_err))
    if rc != 0:
        raise ValueError(f"oracle conv_commit rejected the shape ({rc})")
    return pools_out, row_err


# --------------------------------------------------- KDA (per-channel decay)
def kda_window(S0, q, k, v, a, b, A_log: float, dt_bias):
    """KDA verify window of one unit: a [w, K] per-channel gate inputs,
    dt_bias [K]; otherwise as window().  alpha comes back as [w, K]."""
    S0 = _f64(S0)
    V, K = S0.shape
    q, k, v, a, b, dt_bias = (_f64(t) for t in (q, k, v, a, b, dt_bias))
    w = b.shape[0]
    o = np.empty((w, V)); u = np.empty((w, V)); kh = np.empty((w, K))
    al = np.empty((w, K)); st = np.empty((w, V, K))
    _load().gdn_oracle_kda_window(K, V, w, _dp(S0), _dp(q), _dp(k), _dp(v), _dp(a), _dp(b),
                                  float(A_log), _dp(dt_bias), _dp(o), _dp(u), _dp(kh),
                                  _dp(al), _dp(st))
    return {"o": o, "u": u, "khat": kh, "alpha": al, "states": st}


def kda_replay(S0, u, khat, alpha) -> np.ndarray:
    """Fold len(alpha) KDA records (alpha [n, K]) into a copy of S0 [V, K]."""
    S = _f64(S0).copy()
    V, K = S.shape
    u, khat, alpha = _f64(u), _f64(khat), _f64(alpha).reshape(-1, K)
    _load().gdn_oracle_kda_replay(K, V, alpha.shape[0], _dp(S), _dp(u), _dp(khat), _dp(alpha))
    return S


def kda_spec_verify(*, q, k, v, a, b, A_log, dt_bias, token_start, window_len, pool,
                    slot_table, seq_pos=None, block_size=0, max_window, snapshots=False):
    """KDA verify for one layer: a [T, HV, K], dt_bias [HV, K]; returns the
    same dict as spec_verify with rec_g [B, HV, W, K]."""
    q, k, v, a, b = (_f64(t) for t in (q, k, v, a, b))
    A_log, dt_bias, pool = _f64(A_log), _f64(dt_bias), _f64(pool)
    token_start, window_len = _i32(token_start), _i32(window_len)
    slot_table = _i32(slot_table)
    if slot_table.ndim == 1:
        slot_table = slot_table.reshape(-1, 1)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    B = window_len.shape[0]
    W = int(max_window)
    sp = None if seq_pos is None else _i32(seq_pos)
    nan = np.nan
    out = np.full((T, HV, V), nan)
    rec_u = np.full((B, HV, W, V), nan)
    rec_k = np.full((B, HV, W, K), nan)
    rec_g = np.full((B, HV, W, K), nan)
    snaps = np.full((B, W, HV, V, K), nan) if snapshots else None
    row_err = np.zeros(B, dtype=np.int32)
    rc = _load().gdn_oracle_kda_spec_verify(
        HK, HV, K, V, W, B, T, pool.shape[0], _dp(q), _dp(k), _dp(v), _dp(a), _dp(b),
        _dp(A_log), _dp(dt_bias), _ip(token_start), _ip(window_len), _dp(pool),
        _ip(slot_table), slot_table.shape[1], _ip(sp), int(block_size),
        _dp(out), _dp(rec_u), _dp(rec_k), _dp(rec_g), _dp(snaps), _ip(row_err))
    if rc != 0:
        raise ValueError(f"oracle kda_spec_verify rejected the shape ({rc})")
    return {"out": out, "rec_u": rec_u, "rec_k": rec_k, "rec_g": rec_g, "snaps": snaps,
            "row_err": row_err}


def kda_replay_commit(*, pools, rec_u, rec_k, rec_g, window_len, accepted_len, slot_table,
                      seq_pos=None, block_size=0, max_window):
    """All-layer KDA commit from records: rec_g [L, B, HV, W, K].
    Returns (new_pools float64, row_err)."""
    pools_in = _f64(pools)
    pools_out = pools_in.copy()
    rec_u, rec_k, rec_g = _f64(rec_u), _f64(rec_k), _f64(rec_g)
    window_len, accepted_len = _i32(window_len), _i32(accepted_len)
    slot_table = _i32(slot_table)
    if slot_table.ndim == 1:
        slot_table = slot_table.reshape(-1, 1)
    L, num_slots, HV, V, K = pools_in.shape
    B = window_len.shape[0]
    sp = None if seq_pos is None else _i32(seq_pos)
    row_err = np.zeros(B, dtype=np.int32)
    rc = _load().gdn_oracle_kda_replay_commit(
        L, HV, K, V, int(max_window), B, num_slots, _dp(pools_in), _dp(pools_out),
        _dp(rec_u), _dp(rec_k), _dp(rec_g), _ip(window_len), _ip(accepted_len),
        _ip(slot_table), slot_table.shape[1], _ip(sp), int(block_size), _ip(row_err))
    if rc != 0:
        raise ValueError(f"oracle kda_replay_commit rejected the shape ({rc})")
    return pools_out, row_err
