"""Algorithmic HBM bytes of each kernel for a given step (the method's own
bytes, not the traffic of any particular implementation).

Per live (layer, row r, value head) unit, with e = state element bytes,
q = q/k/v element bytes, w = window_len[r], n = accepted_len[r] and G the
gate width (1 for the scalar decay, K for the per-channel KDA decay):
  commit   V*K*e read + (1 + boundaries) * V*K*e written + n*(V+K+G)*4 record read
  verify   V*K*e read + w*(V*4 out + (V+K+G)*4 record + V*q value + 4*G + 4 gates)
           plus, per (row, key head), w*2*K*q for q and k
  native   V*K*e read + w*V*K*e snapshots + w*(V*4 out + V*q value + 4*G + 4 gates)
           plus the same q and k bytes
Rows with a null slot, an empty window or n = 0 move no bytes.
"""
from __future__ import annotations

from .workloads import SpecBatch


def _rows(sb: SpecBatch):
    win = sb.window_len.tolist()
    acc = sb.accepted_len.tolist()
    table = sb.slot_table.tolist()
    pos = sb.seq_pos.tolist() if sb.seq_pos is not None else [0] * sb.B
    for r in range(sb.B):
        w, n = win[r], acc[r]
        if w <= 0:
            continue
        if sb.block_size == 0:
            src = table[r][0]
        else:
            src = table[r][(pos[r] - 1) // sb.block_size]
        if src < 0:
            continue
        yield r, w, n, pos[r]


def state_bytes(sb: SpecBatch) -> int:
    return sb.V * sb.K * (2 if sb.state_dtype.itemsize == 2 else 4)


def gate_width(sb: SpecBatch) -> int:
    return sb.K if getattr(sb, "kda", False) else 1


def commit_bytes(sb: SpecBatch) -> int:
    S = state_bytes(sb)
    rec = (sb.V + sb.K + gate_width(sb)) * 4
    total = 0
    for r, w, n, p0 in _rows(sb):
        if n <= 0:
            continue
        bounds = 0
        if sb.block_size > 0:
            bounds = sum(1 for j in range(1, n) if (p0 + j) % sb.block_size == 0)
        total += S + (1 + bounds) * S + n * rec
    return total * sb.HV * sb.L


def verify_bytes_per_layer(sb: SpecBatch) -> int:
    S = state_bytes(sb)
    qb = sb.qkv_dtype.itemsize
    G = gate_width(sb)
    per_tok = sb.V * 4 + (sb.V + sb.K + G) * 4 + sb.V * qb + 4 * G + 4
    total = 0
    for r, w, n, p0 in _rows(sb):
        total += sb.HV * (S + w * per_tok) + sb.HK * w * 2 * sb.K * qb
    return total


def native_bytes_per_layer(sb: SpecBatch) -> int:
    S = state_bytes(sb)
    qb = sb.qkv_dtype.itemsize
    per_tok = S + sb.V * 4 + sb.V * qb + 4 * gate_width(sb) + 4
    total = 0
    for r, w, n, p0 in _rows(sb):
        total += sb.HV * (S + w * per_tok) + sb.HK * w * 2 * sb.K * qb
    return total


def verify_flops_per_layer(sb: SpecBatch) -> int:
    """fp32 operations of the recurrence (decay multiply, two dot products,
    rank-1 update: 4 per state element per token, an FMA counted once)."""
    return sum(sb.HV * w * 4 * sb.V * sb.K for r, w, n, p0 in _rows(sb))


def conv_commit_bytes(sb: SpecBatch, C: int, state_len: int, elem_bytes: int) -> int:
    """Short-conv state commit: per live (layer, row) C*SL*e read, n*C*e
    inputs read and (1 + boundaries)*C*SL*e written."""
    S = C * state_len * elem_bytes
    total = 0
    for r, w, n, p0 in _rows(sb):
        if n <= 0:
            continue
        bounds = 0
        if sb.block_size > 0:
            bounds = sum(1 for j in range(1, n) if (p0 + j) % sb.block_size == 0)
        total += S + n * C * elem_bytes + (1 + bounds) * S
    return total * sb.L
