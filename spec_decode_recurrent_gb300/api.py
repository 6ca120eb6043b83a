"""Thin Python binding of libgdn_spec.so: argument marshalling only.

Each function takes torch CUDA tensors, checks that their layout is the one
the C ABI documents (include/gdn_spec.h), and passes raw device pointers,
sizes and the current CUDA stream to the library function of the same
name.  Every step of the computation runs in the library's kernels; there
is no fallback.  A missing library raises at the first call.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

from . import build as _build

GDN_DTYPE_F32, GDN_DTYPE_BF16 = 0, 1
ROW_ERR_WINDOW, ROW_ERR_ACCEPTED, ROW_ERR_SLOT = 1, 2, 4
ROW_ERR_BLOCK, ROW_ERR_SEQPOS, ROW_ERR_TOKENS = 8, 16, 32
ROW_ERR_GROUP, ROW_ERR_REJECTED = 64, 128
ENTRY_POINTS = ("gdn_spec_verify", "gdn_replay_commit", "gdn_replay_commit_grouped",
                "gdn_conv_state_commit", "gdn_native_spec_snapshot", "gdn_kda_spec_verify",
                "gdn_kda_native_spec_snapshot", "gdn_kda_replay_commit",
                "gdn_kda_replay_commit_grouped")

_ERRORS = {-1: "null pointer", -2: "unsupported shape or dtype",
           -3: "invalid count, stride, alignment or block size", -4: "CUDA launch failed"}


class GDNError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({_ERRORS.get(code, 'unknown')})")
        self.code = code


class gdn_shape(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k", ctypes.c_int32), ("head_v", ctypes.c_int32),
                ("max_window", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_VERIFY_HEAD = [ctypes.POINTER(gdn_shape), _I32, _I32, _I32, _P, _I64, _P, _I64, _P, _I64,
                _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32, _P, _I64]


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libgdn_spec.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with spec_decode_recurrent_gb300.build.build()")
            lib = ctypes.CDLL(path)
            lib.gdn_spec_verify.restype = ctypes.c_int
            lib.gdn_spec_verify.argtypes = _VERIFY_HEAD + [_P, _P, _P, _P, _P]
            lib.gdn_native_spec_snapshot.restype = ctypes.c_int
            lib.gdn_native_spec_snapshot.argtypes = _VERIFY_HEAD + [_P, _P, _P]
            lib.gdn_replay_commit.restype = ctypes.c_int
            lib.gdn_replay_commit.argtypes = [ctypes.POINTER(gdn_shape), _I32, _I32, _I32,
                                              _P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32,
                                              _P, _P]
            lib.gdn_kda_spec_verify.restype = ctypes.c_int
            lib.gdn_kda_spec_verify.argtypes = lib.gdn_spec_verify.argtypes
            lib.gdn_kda_native_spec_snapshot.restype = ctypes.c_int
            lib.gdn_kda_native_spec_snapshot.argtypes = lib.gdn_native_spec_snapshot.argtypes
            lib.gdn_kda_replay_commit.restype = ctypes.c_int
            lib.gdn_kda_replay_commit.argtypes = lib.gdn_replay_commit.argtypes
            lib.gdn_conv_state_commit.restype = ctypes.c_int
            lib.gdn_conv_state_commit.argtypes = [
                _I32, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I64, _P, _P,
                _P, _P, _I32, _I64, _P, _I32, _P, _P]
            lib.gdn_replay_commit_grouped.restype = ctypes.c_int
            lib.gdn_replay_commit_grouped.argtypes = [
                ctypes.POINTER(gdn_shape), _I32, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _P,
                _P, _I32, _I64, _P, _I32, _P, _P]
            lib.gdn_kda_replay_commit_grouped.restype = ctypes.c_int
            lib.gdn_kda_replay_commit_grouped.argtypes = lib.gdn_replay_commit_grouped.argtypes
            _lib = lib
    return _lib


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return GDN_DTYPE_F32
    if t == torch.bfloat16:
        return GDN_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _rows(t: torch.Tensor, name: str, dtype=None):
    """[rows, heads, width] view with contiguous heads; returns the row stride."""
    _need(t.dim() == 3 and t.is_cuda, f"{name} must be a 3-d CUDA tensor")
    _need(t.stride(2) == 1 and t.stride(1) == t.shape[2], f"{name}: heads must be contiguous")
    if dtype is not None:
        _need(t.dtype == dtype, f"{name} must be {dtype}")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1] * t.shape[2]


def _contig(t: torch.Tensor, name: str, dtype):
    _need(t.is_cuda and t.is_contiguous() and t.dtype == dtype,
          f"{name} must be a contiguous CUDA {dtype} tensor")


def _verify_args(q, k, v, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                 slot_table, seq_pos, block_size, out, max_window, kda=False):
    T, HK, K = q.shape
    _need(k.shape == q.shape and k.dtype == q.dtype, "k must match q")
    _need(v.shape[0] == T and v.dtype == q.dtype, "v must have q's rows and dtype")
    HV, V = v.shape[1], v.shape[2]
    qs, ks, vs = _rows(q, "q"), _rows(k, "k"), _rows(v, "v")
    os_ = _rows(out, "out", torch.float32)
    _need(out.shape == (T, HV, V), "out must be [num_tokens, HV, V]")
    _need(state_pool.dim() == 4 and state_pool.shape[1:] == (HV, V, K), "pool must be [slots, HV, V, K]")
    _contig(state_pool, "state_pool", state_pool.dtype)
    # per-channel (KDA) gates: a [T, HV, K] and dt_bias [HV, K]
    G = K if kda else 1
    _contig(a, "a", torch.float32)
    _need(a.numel() == T * HV * G and a.shape[:2] == (T, HV),
          "a must be [num_tokens, HV]" + (", K]" if kda else ""))
    _contig(b, "b", torch.float32)
    _need(b.shape == (T, HV), "b must be [num_tokens, HV]")
    _contig(A_log, "A_log", torch.float32)
    _need(A_log.numel() == HV, "A_log must have HV entries")
    _contig(dt_bias, "dt_bias", torch.float32)
    _need(dt_bias.numel() == HV * G, "dt_bias must have HV" + (" * K" if kda else "") + " entries")
    B = window_len.shape[0]
    for name, t in (("token_start", token_start), ("window_len", window_len)):
        _contig(t, name, torch.int32)
        _need(t.shape == (B,), f"{name} must be [batch]")
    st = slot_table if slot_table.dim() == 2 else slot_table.view(-1, 1)
    _contig(st, "slot_table", torch.int32)
    _need(st.shape[0] == B, "slot_table must have one row per request")
    if block_size:
        _contig(seq_pos, "seq_pos", torch.int32)
    shape = gdn_shape(HK, HV, K, V, int(max_window), _dtype_code(q.dtype),
                      _dtype_code(state_pool.dtype))
    head = [ctypes.byref(shape), B, T, state_pool.shape[0], _ptr(q), qs, _ptr(k), ks, _ptr(v), vs,
            _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(token_start), _ptr(window_len),
            _ptr(state_pool), _ptr(st), st.shape[1], _ptr(seq_pos if block_size else None),
            int(block_size), _ptr(out), os_]
    return shape, head, B, HV, V, K


def _verify(fn, kda, q, k, v, a, b, A_log, dt_bias, token_start, window_len, state_pool,
            slot_table, out, rec_u, rec_k, rec_g, max_window, seq_pos, block_size, err, stream):
    shape, head, B, HV, V, K = _verify_args(q, k, v, a, b, A_log, dt_bias, token_start,
                                            window_len, state_pool, slot_table, seq_pos,
                                            block_size, out, max_window, kda)
    W = int(max_window)
    for name, t, shp in (("rec_u", rec_u, (B, HV, W, V)), ("rec_k", rec_k, (B, HV, W, K)),
                         ("rec_g", rec_g, (B, HV, W, K) if kda else (B, HV, W))):
        _contig(t, name, torch.float32)
        _need(tuple(t.shape) == shp, f"{name} must be {shp}")
    if err is not None:
        _contig(err, "err", torch.int32)
    rc = getattr(load(), fn)(*head, _ptr(rec_u), _ptr(rec_k), _ptr(rec_g), _ptr(err),
                             _stream(stream))
    if rc != 0:
        raise GDNError(fn, rc)


def _native(fn, kda, q, k, v, a, b, A_log, dt_bias, token_start, window_len, state_pool,
            slot_table, out, snapshots, max_window, seq_pos, block_size, err, stream):
    shape, head, B, HV, V, K = _verify_args(q, k, v, a, b, A_log, dt_bias, token_start,
                                            window_len, state_pool, slot_table, seq_pos,
                                            block_size, out, max_window, kda)
    W = int(max_window)
    _contig(snapshots, "snapshots", state_pool.dtype)
    _need(tuple(snapshots.shape) == (B, W, HV, V, K), "snapshots must be [batch, W, HV, V, K]")
    if err is not None:
        _contig(err, "err", torch.int32)
    rc = getattr(load(), fn)(*head, _ptr(snapshots), _ptr(err), _stream(stream))
    if rc != 0:
        raise GDNError(fn, rc)


def gdn_spec_verify(*, q, k, v, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                    slot_table, out, rec_u, rec_k, rec_g, max_window, seq_pos=None,
                    block_size=0, err=None, stream=None) -> None:
    """Verify one layer: writes out and the replay record, never the pool."""
    _verify("gdn_spec_verify", False, q, k, v, a, b, A_log, dt_bias, token_start, window_len,
            state_pool, slot_table, out, rec_u, rec_k, rec_g, max_window, seq_pos, block_size,
            err, stream)


def gdn_kda_spec_verify(*, q, k, v, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                        slot_table, out, rec_u, rec_k, rec_g, max_window, seq_pos=None,
                        block_size=0, err=None, stream=None) -> None:
    """Per-channel-decay (KDA) verify of one layer: a [T, HV, K], dt_bias
    [HV, K], rec_g [B, HV, W, K]; otherwise as gdn_spec_verify."""
    _verify("gdn_kda_spec_verify", True, q, k, v, a, b, A_log, dt_bias, token_start, window_len,
            state_pool, slot_table, out, rec_u, rec_k, rec_g, max_window, seq_pos, block_size,
            err, stream)


def gdn_native_spec_snapshot(*, q, k, v, a, b, A_log, dt_bias, token_start, window_len,
                             state_pool, slot_table, out, snapshots, max_window, seq_pos=None,
                             block_size=0, err=None, stream=None) -> None:
    """Native baseline of one layer: writes out and the state after every token."""
    _native("gdn_native_spec_snapshot", False, q, k, v, a, b, A_log, dt_bias, token_start,
            window_len, state_pool, slot_table, out, snapshots, max_window, seq_pos, block_size,
            err, stream)


def gdn_kda_native_spec_snapshot(*, q, k, v, a, b, A_log, dt_bias, token_start, window_len,
                                 state_pool, slot_table, out, snapshots, max_window,
                                 seq_pos=None, block_size=0, err=None, stream=None) -> None:
    """Native baseline of one layer with the per-channel (KDA) decay."""
    _native("gdn_kda_native_spec_snapshot", True, q, k, v, a, b, A_log, dt_bias, token_start,
            window_len, state_pool, slot_table, out, snapshots, max_window, seq_pos, block_size,
            err, stream)


class LayerTable:
    """Device arrays of per-layer pointers (pools and records) for the
    all-layer commit.  Build once per set of buffers and reuse."""

    def __init__(self, pools: Sequence[torch.Tensor], rec_u: Sequence[torch.Tensor],
                 rec_k: Sequence[torch.Tensor], rec_g: Sequence[torch.Tensor]):
        L = len(pools)
        _need(L >= 1 and len(rec_u) == len(rec_k) == len(rec_g) == L, "one entry per layer")
        p0 = pools[0]
        for t in pools:
            _contig(t, "pool", p0.dtype)
            _need(t.shape == p0.shape and t.device == p0.device, "pools must share shape")
        for name, lst in (("rec_u", rec_u), ("rec_k", rec_k), ("rec_g", rec_g)):
            for t in lst:
                _contig(t, name, torch.float32)
        dev = p0.device
        mk = lambda ts: torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device=dev)
        self.pools, self.rec_u, self.rec_k, self.rec_g = list(pools), list(rec_u), list(rec_k), list(rec_g)
        self.d_pools, self.d_rec_u, self.d_rec_k, self.d_rec_g = mk(pools), mk(rec_u), mk(rec_k), mk(rec_g)
        self.num_layers = L
        self.num_slots, self.HV, self.V, self.K = p0.shape
        self.state_dtype = p0.dtype
        self.B, _, self.W, _ = rec_u[0].shape
        self.kda = rec_g[0].dim() == 4        # per-channel gate records [B, HV, W, K]


def gdn_replay_commit(*, table: LayerTable, num_k_heads: int, window_len, accepted_len,
                      slot_table, seq_pos=None, block_size=0, err=None, stream=None) -> None:
    """All-layer commit in one launch: replays the accepted prefix of every
    row of every layer and writes each state once (plus align boundaries).
    A table of per-channel gate records (KDA) calls gdn_kda_replay_commit."""
    B = window_len.shape[0]
    _need(B == table.B, "batch must match the record buffers")
    for name, t in (("window_len", window_len), ("accepted_len", accepted_len)):
        _contig(t, name, torch.int32)
        _need(t.shape == (B,), f"{name} must be [batch]")
    st = slot_table if slot_table.dim() == 2 else slot_table.view(-1, 1)
    _contig(st, "slot_table", torch.int32)
    if block_size:
        _contig(seq_pos, "seq_pos", torch.int32)
    if err is not None:
        _contig(err, "err", torch.int32)
    # the commit reads no q/k/v: qkv_dtype is a placeholder
    shape = gdn_shape(int(num_k_heads), table.HV, table.K, table.V, table.W, GDN_DTYPE_F32,
                      _dtype_code(table.state_dtype))
    fn = "gdn_kda_replay_commit" if table.kda else "gdn_replay_commit"
    rc = getattr(load(), fn)(
        ctypes.byref(shape), table.num_layers, B, table.num_slots, _ptr(table.d_pools),
        _ptr(table.d_rec_u), _ptr(table.d_rec_k), _ptr(table.d_rec_g), _ptr(window_len),
        _ptr(accepted_len), _ptr(st), st.shape[1], _ptr(seq_pos if block_size else None),
        int(block_size), _ptr(err), _stream(stream))
    if rc != 0:
        raise GDNError(fn, rc)


def gdn_replay_commit_grouped(*, table: LayerTable, num_k_heads: int, layer_group, window_len,
                              accepted_len, slot_tables, seq_pos=None, block_size=0, err=None,
                              stream=None) -> None:
    """All-layer commit in one launch for layers split into KV-cache groups:
    layer l uses slot_tables[layer_group[l]] ([groups, batch, stride]).  A
    table of per-channel gate records (KDA) calls gdn_kda_replay_commit_grouped."""
    B = window_len.shape[0]
    _need(B == table.B, "batch must match the record buffers")
    for name, t in (("window_len", window_len), ("accepted_len", accepted_len)):
        _contig(t, name, torch.int32)
        _need(t.shape == (B,), f"{name} must be [batch]")
    _contig(layer_group, "layer_group", torch.int32)
    _need(layer_group.shape == (table.num_layers,), "layer_group must be [num_layers]")
    _contig(slot_tables, "slot_tables", torch.int32)
    _need(slot_tables.dim() == 3 and slot_tables.shape[1] == B, "slot_tables must be [groups, batch, stride]")
    if block_size:
        _contig(seq_pos, "seq_pos", torch.int32)
    if err is not None:
        _contig(err, "err", torch.int32)
    G, _, stride = slot_tables.shape
    shape = gdn_shape(int(num_k_heads), table.HV, table.K, table.V, table.W, GDN_DTYPE_F32,
                      _dtype_code(table.state_dtype))
    fn = "gdn_kda_replay_commit_grouped" if table.kda else "gdn_replay_commit_grouped"
    rc = getattr(load(), fn)(
        ctypes.byref(shape), table.num_layers, G, _ptr(layer_group), B, table.num_slots,
        _ptr(table.d_pools), _ptr(table.d_rec_u), _ptr(table.d_rec_k), _ptr(table.d_rec_g),
        _ptr(window_len), _ptr(accepted_len), _ptr(slot_tables), stride, B * stride,
        _ptr(seq_pos if block_size else None), int(block_size), _ptr(err), _stream(stream))
    if rc != 0:
        raise GDNError(fn, rc)


class ConvTable:
    """Device arrays of per-layer pointers for the short-conv state commit:
    pools [num_slots, C, SL] and the layer's convolution inputs [T, C]
    (token rows may be strided; every layer the same row stride)."""

    def __init__(self, pools: Sequence[torch.Tensor], inputs: Sequence[torch.Tensor]):
        _need(len(pools) >= 1 and len(pools) == len(inputs), "one pool and one input per layer")
        p0, x0 = pools[0], inputs[0]
        for t in pools:
            _contig(t, "conv pool", p0.dtype)
            _need(t.shape == p0.shape and t.dim() == 3, "conv pools must share [slots, C, SL]")
        for x in inputs:
            _need(x.is_cuda and x.dim() == 2 and x.dtype == p0.dtype and x.stride(1) == 1,
                  "conv inputs must be [T, C] rows of the pools' dtype")
            _need(x.shape == x0.shape and x.stride(0) == x0.stride(0), "conv inputs must share layout")
        _need(x0.shape[1] == p0.shape[1], "conv inputs must have C channels")
        dev = p0.device
        mk = lambda ts: torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device=dev)
        self.pools, self.inputs = list(pools), list(inputs)
        self.d_pools, self.d_inputs = mk(pools), mk(inputs)
        self.num_layers = len(pools)
        self.num_slots, self.C, self.SL = p0.shape
        self.dtype = p0.dtype
        self.num_tokens = x0.shape[0]
        self.in_stride = x0.stride(0) if x0.shape[0] > 1 else x0.shape[1]


def gdn_conv_state_commit(*, table: ConvTable, token_start, window_len, accepted_len,
                          slot_tables, max_window, layer_group=None, seq_pos=None,
                          block_size=0, err=None, stream=None) -> None:
    """Short-conv state commit of every layer in one launch, with the same
    plan as the recurrent-state commit."""
    B = window_len.shape[0]
    for name, t in (("token_start", token_start), ("window_len", window_len),
                    ("accepted_len", accepted_len)):
        _contig(t, name, torch.int32)
        _need(t.shape == (B,), f"{name} must be [batch]")
    st = slot_tables if slot_tables.dim() == 3 else slot_tables.view(1, B, -1)
    _contig(st, "slot_tables", torch.int32)
    G, _, stride = st.shape
    if layer_group is not None:
        _contig(layer_group, "layer_group", torch.int32)
        _need(layer_group.shape == (table.num_layers,), "layer_group must be [num_layers]")
    if block_size:
        _contig(seq_pos, "seq_pos", torch.int32)
    if err is not None:
        _contig(err, "err", torch.int32)
    rc = load().gdn_conv_state_commit(
        table.num_layers, G, _ptr(layer_group), B, table.num_tokens, table.num_slots, table.C,
        table.SL, _dtype_code(table.dtype), int(max_window), _ptr(table.d_pools),
        _ptr(table.d_inputs), table.in_stride, _ptr(token_start), _ptr(window_len),
        _ptr(accepted_len), _ptr(st), stride, B * stride, _ptr(seq_pos if block_size else None),
        int(block_size), _ptr(err), _stream(stream))
    if rc != 0:
        raise GDNError("gdn_conv_state_commit", rc)
