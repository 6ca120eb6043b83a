"""One speculative step of an L-layer GDN stack through the C ABI.

``StepBuffers`` owns the per-layer outputs and replay records of a
``workloads.SpecBatch``; ``verify_all`` runs the verify of every layer
(one launch per layer, as a model forward would), ``commit`` runs the
single all-layer commit launch, and ``native_layer`` runs the native
per-draft-snapshot baseline of one layer.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import api
from .workloads import SpecBatch


class StepBuffers:
    def __init__(self, sb: SpecBatch, fill: Optional[float] = None):
        dev = sb.device
        make = (lambda shape: torch.full(shape, fill, dtype=torch.float32, device=dev)) \
            if fill is not None else (lambda shape: torch.empty(shape, dtype=torch.float32, device=dev))
        # every layer's output in one tensor, so a step's result is one copy
        self.out_all = make((sb.L, sb.T, sb.HV, sb.V))
        self.out = list(self.out_all.unbind(0))
        self.rec_u = [make((sb.B, sb.HV, sb.W, sb.V)) for _ in range(sb.L)]
        self.rec_k = [make((sb.B, sb.HV, sb.W, sb.K)) for _ in range(sb.L)]
        gshape = (sb.B, sb.HV, sb.W, sb.K) if sb.kda else (sb.B, sb.HV, sb.W)
        self.rec_g = [make(gshape) for _ in range(sb.L)]
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.table = api.LayerTable(sb.pools, self.rec_u, self.rec_k, self.rec_g)


def verify_layer(sb: SpecBatch, bufs: StepBuffers, layer: int, stream=None) -> None:
    fn = api.gdn_kda_spec_verify if sb.kda else api.gdn_spec_verify
    fn(
        q=sb.q[layer], k=sb.k[layer], v=sb.v[layer], a=sb.a[layer], b=sb.b[layer],
        A_log=sb.A_log[layer], dt_bias=sb.dt_bias[layer], token_start=sb.token_start,
        window_len=sb.window_len, state_pool=sb.pools[layer], slot_table=sb.slot_table,
        seq_pos=sb.seq_pos, block_size=sb.block_size, out=bufs.out[layer],
        rec_u=bufs.rec_u[layer], rec_k=bufs.rec_k[layer], rec_g=bufs.rec_g[layer],
        max_window=sb.W, err=bufs.err, stream=stream)


def verify_all(sb: SpecBatch, bufs: StepBuffers, stream=None) -> None:
    for layer in range(sb.L):
        verify_layer(sb, bufs, layer, stream)


def commit(sb: SpecBatch, bufs: StepBuffers, stream=None, check_slots: bool = False) -> None:
    """The all-layer commit.  check_slots (a debug aid: it copies the row
    metadata to the host and synchronises) first verifies that no live row
    writes a slot another live row reads or writes."""
    if check_slots:
        check_slot_exclusivity(sb.window_len, sb.accepted_len, sb.slot_table, sb.seq_pos,
                               sb.block_size)
    api.gdn_replay_commit(table=bufs.table, num_k_heads=sb.HK, window_len=sb.window_len,
                          accepted_len=sb.accepted_len, slot_table=sb.slot_table,
                          seq_pos=sb.seq_pos, block_size=sb.block_size, err=bufs.err,
                          stream=stream)


def check_slot_exclusivity(window_len, accepted_len, slot_table, seq_pos=None,
                           block_size: int = 0) -> None:
    """Raise ValueError if a slot one live row of a commit writes (its final
    or a boundary slot) is read or written by another live row: the rows of
    one launch run concurrently with no ordering between them, so such a
    call has no defined result.  A row may write its own checkpoint slot.
    Rows the commit would skip or flag (null slot, nothing accepted, a
    malformed row) are left out.  Host-side, for debugging."""
    win = [int(x) for x in window_len.tolist()]
    acc = [int(x) for x in accepted_len.tolist()]
    table = slot_table.view(len(win), -1).tolist()
    pos = [int(x) for x in seq_pos.tolist()] if (block_size and seq_pos is not None) else None

    def slot_after(row, x):
        if block_size == 0:
            return row[0]
        col = (x - 1) // block_size
        return row[col] if 1 <= x and col < len(row) else None

    reads, writes = {}, {}
    for r, (w, n) in enumerate(zip(win, acc)):
        if w <= 0 or n <= 0 or n > w:
            continue
        p0 = pos[r] if pos is not None else 0
        src = slot_after(table[r], p0)
        if src is None or src < 0:
            continue
        mine = set()
        for j in range(1, n + 1):           # the block of every accepted token
            if block_size == 0 and j < n:
                continue
            s_ = slot_after(table[r], p0 + j)
            if s_ is not None and s_ >= 0:
                mine.add(s_)
        reads.setdefault(src, set()).add(r)
        for s_ in mine:
            writes.setdefault(s_, set()).add(r)
    for s_, rows in writes.items():
        others = (rows | reads.get(s_, set()))
        if len(others) > 1:
            raise ValueError(f"slot {s_} is written by row(s) {sorted(rows)} and used by rows "
                             f"{sorted(others)} in the same commit")


def native_layer(sb: SpecBatch, layer: int, out: torch.Tensor, snapshots: torch.Tensor,
                 err: Optional[torch.Tensor] = None, stream=None) -> None:
    fn = api.gdn_kda_native_spec_snapshot if sb.kda else api.gdn_native_spec_snapshot
    fn(
        q=sb.q[layer], k=sb.k[layer], v=sb.v[layer], a=sb.a[layer], b=sb.b[layer],
        A_log=sb.A_log[layer], dt_bias=sb.dt_bias[layer], token_start=sb.token_start,
        window_len=sb.window_len, state_pool=sb.pools[layer], slot_table=sb.slot_table,
        seq_pos=sb.seq_pos, block_size=sb.block_size, out=out, snapshots=snapshots,
        max_window=sb.W, err=err, stream=stream)


def native_buffers(sb: SpecBatch, fill: Optional[float] = None):
    dev = sb.device
    out = torch.empty((sb.T, sb.HV, sb.V), dtype=torch.float32, device=dev)
    snaps = torch.empty((sb.B, sb.W, sb.HV, sb.V, sb.K), dtype=sb.state_dtype, device=dev)
    if fill is not None:
        out.fill_(fill)
        snaps.fill_(fill)
    return out, snaps


def pack_inputs(sb: SpecBatch) -> torch.Tensor:
    """Move every per-step input of `sb` (q/k/v or the fused projection,
    a, b and the row metadata of all layers) into one contiguous device
    byte arena and rebind `sb`'s tensors to views of it, keeping shapes and
    strides.  A step's inputs can then arrive with a single host-to-device
    copy.  Returns the arena."""
    roots = []          # (owner list, index or None, tensor) for tensors owning storage
    for l in range(sb.L):
        if sb.fused_qkv:
            roots.append(("fused_qkv", l, sb.fused_qkv[l]))
        else:
            roots += [("q", l, sb.q[l]), ("k", l, sb.k[l]), ("v", l, sb.v[l])]
        roots += [("a", l, sb.a[l]), ("b", l, sb.b[l])]
    for name in ("token_start", "window_len", "accepted_len", "slot_table", "seq_pos"):
        if getattr(sb, name) is not None:
            roots.append((name, None, getattr(sb, name)))
    align = 256
    offsets, total = [], 0
    for _, _, t in roots:
        assert t.is_contiguous()
        offsets.append(total)
        total += -(-t.numel() * t.element_size() // align) * align
    arena = torch.empty(total, dtype=torch.uint8, device=sb.device)
    for (name, l, t), off in zip(roots, offsets):
        nbytes = t.numel() * t.element_size()
        view = arena[off:off + nbytes].view(t.dtype).view(t.shape)
        view.copy_(t)
        if l is None:
            setattr(sb, name, view)
        else:
            getattr(sb, name)[l] = view
    if sb.fused_qkv:
        HK, HV, K, V = sb.HK, sb.HV, sb.K, sb.V
        for l, buf in enumerate(sb.fused_qkv):
            sb.q[l] = buf[:, :HK * K].unflatten(1, (HK, K))
            sb.k[l] = buf[:, HK * K:2 * HK * K].unflatten(1, (HK, K))
            sb.v[l] = buf[:, 2 * HK * K:].unflatten(1, (HV, V))
    return arena
