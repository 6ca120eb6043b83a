"""Seeded synthetic inputs for GDN speculative verify / replay commit.

This module only draws random numbers and lays out index tables; it holds
none of the method's arithmetic (no gates, no normalisation, no recurrence),
so both the CUDA path and the fp64 oracle can be fed from it.

Distributions (the same for every workload unless stated):
  q, k, v      ~ N(0, 1), raw; the method L2-normalises q and k itself
  a, b         ~ N(0, 1) fp32   (extreme-gate workload: U(-20, 20))
  A_log        ~ U(0, ln 16) fp32, dt_bias ~ U(-1, 1) fp32, per value head
  state        ~ N(0, 0.1) (std 0.1) in the slots rows read
Slots that no row reads can be filled with a NaN sentinel so that a stray
read poisons the outputs and a stray write shows up bit for bit.

Named workloads (sizes are those of the five benchmark configurations):
  tiny          1 layer, batch 2, HK=HV=2, K=V=16, window 4, accepted [1, 3]
  layer         1 layer, HK=16, HV=32, K=V=128, batch 16, window 4, bf16 q/k/v
  all_layer     36 layers, batch 64 (8 graph-padding rows), 256-slot pools
  long_ragged   36 layers, batch 256, window 6 mixed with ragged 4/1/3,
                non-contiguous strided rows, extreme gates, three seeds
  align         36 layers, batch 128, window 4, block size 4, align mode,
                fp32 or bf16 state
  kda_all_layer the all_layer shapes with a per-channel (KDA) decay
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

F32, BF16 = torch.float32, torch.bfloat16
SENTINEL_F32_BITS = 0x7FBADBAD   # a NaN payload no arithmetic produces
SENTINEL_BF16_BITS = 0x7FBA


@dataclasses.dataclass
class SpecBatch:
    """One speculative step of an L-layer GDN stack.

    Per layer: q, k [T, HK, K] and v [T, HV, V] (views; rows may be strided),
    a, b [T, HV] fp32, A_log, dt_bias [HV] fp32, pool [num_slots, HV, V, K].
    Per row: token_start, window_len, accepted_len, seq_pos [B] int32 and
    slot_table [B, table_stride] int32 (-1 = null).
    """
    name: str
    HK: int
    HV: int
    K: int
    V: int
    W: int
    L: int
    B: int
    T: int
    num_slots: int
    block_size: int
    qkv_dtype: torch.dtype
    state_dtype: torch.dtype
    q: List[torch.Tensor]
    k: List[torch.Tensor]
    v: List[torch.Tensor]
    a: List[torch.Tensor]
    b: List[torch.Tensor]
    A_log: List[torch.Tensor]
    dt_bias: List[torch.Tensor]
    pools: List[torch.Tensor]
    token_start: torch.Tensor
    window_len: torch.Tensor
    accepted_len: torch.Tensor
    slot_table: torch.Tensor
    seq_pos: Optional[torch.Tensor]
    fused_qkv: Optional[List[torch.Tensor]] = None
    kda: bool = False     # per-channel decay: a [T, HV, K], dt_bias [HV, K]

    @property
    def device(self) -> torch.device:
        return self.pools[0].device

    def row_slots(self, r: int) -> List[int]:
        return [int(x) for x in self.slot_table[r].tolist() if int(x) >= 0]


def sentinel_like(shape, dtype, device) -> torch.Tensor:
    if dtype == F32:
        return torch.full(shape, SENTINEL_F32_BITS, dtype=torch.int32, device=device).view(F32)
    return torch.full(shape, SENTINEL_BF16_BITS, dtype=torch.int16, device=device).view(BF16)


def _uniform(shape, lo, hi, gen, device):
    return torch.rand(shape, generator=gen, device=device, dtype=F32) * (hi - lo) + lo


def _make(name, *, HK, HV, K, V, W, L, windows, accepted, num_slots, slots_for_row,
          seq_pos=None, block_size=0, qkv_dtype, state_dtype, gen, device,
          sentinel, gate_range=None, gaps=None, row_order=None, fused=False, kda=False):
    """Lay out one step and draw its tensors.

    windows/accepted: per-row lists.  slots_for_row: list of per-row tables
    (lists, -1 = null).  gaps: per-row count of unused token rows placed
    before the row.  row_order: order in which rows are placed in the token
    array (default 0..B-1).
    """
    B = len(windows)
    order = list(range(B)) if row_order is None else list(row_order)
    token_start = [0] * B
    pos = 0
    for r in order:
        pos += 0 if gaps is None else int(gaps[r])
        token_start[r] = pos
        pos += int(windows[r])
    T = max(pos, 1)
    stride = max(len(s) for s in slots_for_row)
    table = torch.full((B, stride), -1, dtype=torch.int32)
    for r, s in enumerate(slots_for_row):
        table[r, :len(s)] = torch.tensor(s, dtype=torch.int32)

    # Slots some live row reads as its checkpoint: these carry a random state.
    read_slots = set()
    for r in range(B):
        if windows[r] == 0:
            continue
        if block_size == 0:
            s = slots_for_row[r][0]
        else:
            s = slots_for_row[r][(seq_pos[r] - 1) // block_size]
        if s >= 0:
            read_slots.add(int(s))

    q, k, v, a, b, A_log, dt_bias, pools, fused_list = [], [], [], [], [], [], [], [], []
    width = 2 * HK * K + HV * V
    for _ in range(L):
        if fused:
            buf = torch.randn((T, width), generator=gen, device=device, dtype=F32).to(qkv_dtype)
            fused_list.append(buf)
            q.append(buf[:, :HK * K].unflatten(1, (HK, K)))
            k.append(buf[:, HK * K:2 * HK * K].unflatten(1, (HK, K)))
            v.append(buf[:, 2 * HK * K:].unflatten(1, (HV, V)))
        else:
            q.append(torch.randn((T, HK, K), generator=gen, device=device, dtype=F32).to(qkv_dtype))
            k.append(torch.randn((T, HK, K), generator=gen, device=device, dtype=F32).to(qkv_dtype))
            v.append(torch.randn((T, HV, V), generator=gen, device=device, dtype=F32).to(qkv_dtype))
        ga = (T, HV, K) if kda else (T, HV)       # per-channel gate inputs for KDA
        if gate_range is None:
            a.append(torch.randn(ga, generator=gen, device=device, dtype=F32))
            b.append(torch.randn((T, HV), generator=gen, device=device, dtype=F32))
        else:
            a.append(_uniform(ga, -gate_range, gate_range, gen, device))
            b.append(_uniform((T, HV), -gate_range, gate_range, gen, device))
        A_log.append(_uniform((HV,), 0.0, math.log(16.0), gen, device))
        dt_bias.append(_uniform((HV, K) if kda else (HV,), -1.0, 1.0, gen, device))
        state = (torch.randn((num_slots, HV, V, K), generator=gen, device=device, dtype=F32)
                 * 0.1).to(state_dtype)
        if sentinel:
            keep = torch.zeros(num_slots, dtype=torch.bool)
            keep[sorted(read_slots)] = True
            keep = keep.to(device)
            fill = sentinel_like(state.shape, state_dtype, device)
            state = torch.where(keep.view(-1, 1, 1, 1), state, fill)
        pools.append(state)

    dev = torch.device(device)
    as_i32 = lambda x: torch.tensor(x, dtype=torch.int32).to(dev)
    return SpecBatch(
        name=name, HK=HK, HV=HV, K=K, V=V, W=W, L=L, B=B, T=T, num_slots=num_slots,
        block_size=block_size, qkv_dtype=qkv_dtype, state_dtype=state_dtype,
        q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, pools=pools,
        token_start=as_i32(token_start), window_len=as_i32(list(windows)),
        accepted_len=as_i32(list(accepted)), slot_table=table.to(dev),
        seq_pos=None if seq_pos is None else as_i32(list(seq_pos)),
        fused_qkv=fused_list if fused else None, kda=kda)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _ints(gen, lo, hi, n):
    """n integers uniform in [lo, hi] drawn on the CPU generator stream."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen).tolist()]


# ----------------------------------------------------------------- workloads
def tiny(device="cpu", sentinel=True, seed=0):
    """1 layer, batch 2, HK=HV=2, K=V=16, window 4, accepted [1, 3], fp32."""
    gen = _gen(seed, device)
    return _make("tiny", HK=2, HV=2, K=16, V=16, W=4, L=1, windows=[4, 4], accepted=[1, 3],
                 num_slots=2, slots_for_row=[[0], [1]], qkv_dtype=F32, state_dtype=F32,
                 gen=gen, device=device, sentinel=sentinel)


def layer(device="cpu", sentinel=True, seed=1, batch=16, HK=16, HV=32, KV=128, L=1,
          num_slots=64, window=4, qkv_dtype=BF16, state_dtype=F32):
    """Single GDN layer at serving shape (GQA 2:1, 128x128 fp32 state per value head)."""
    cpu = _gen(seed, "cpu")
    windows = [window] * batch
    accepted = _ints(cpu, 1, window, batch)
    slots = torch.randperm(num_slots, generator=cpu)[:batch].tolist()
    gen = _gen(seed, device)
    return _make("layer", HK=HK, HV=HV, K=KV, V=KV, W=window, L=L, windows=windows,
                 accepted=accepted, num_slots=num_slots, slots_for_row=[[s] for s in slots],
                 qkv_dtype=qkv_dtype, state_dtype=state_dtype, gen=gen, device=device,
                 sentinel=sentinel)


def all_layer(device="cpu", sentinel=True, seed=2, L=36, batch=64, pad_rows=8, HK=16, HV=32,
              KV=128, num_slots=256, window=4, state_dtype=F32, kda=False):
    """All-layer commit workload: live rows then graph-padding rows (slot -1, window 0)."""
    cpu = _gen(seed, "cpu")
    live = batch - pad_rows
    windows = [window] * live + [0] * pad_rows
    accepted = _ints(cpu, 1, window, live) + [0] * pad_rows
    perm = torch.randperm(num_slots, generator=cpu).tolist()
    slots = [[perm[r]] for r in range(live)] + [[-1]] * pad_rows
    gen = _gen(seed, device)
    return _make("kda_all_layer" if kda else "all_layer", HK=HK, HV=HV, K=KV, V=KV, W=window,
                 L=L, windows=windows, accepted=accepted, num_slots=num_slots,
                 slots_for_row=slots, qkv_dtype=BF16, state_dtype=state_dtype, gen=gen,
                 device=device, sentinel=sentinel, kda=kda)


def kda_all_layer(device="cpu", sentinel=True, seed=6, state_dtype=F32, **kw):
    """The all_layer shapes with the per-channel (KDA) decay: gate inputs
    a [T, HV, K] ~ N(0, 1) and dt_bias [HV, K] ~ U(-1, 1)."""
    return all_layer(device=device, sentinel=sentinel, seed=seed, state_dtype=state_dtype,
                     kda=True, **kw)


# Per-position acceptance rates of a five-draft (window 6) run, P(n >= 1 + i)
# for i = 1..5, as measured in the review thread of vLLM PR "[Spec Decode]
# [Qwen4Exp] RecoverSSM for Qwen GDN and the PLE short conv" (the MTP 5 run's
# accept-length note); the mean accepted length they imply is 3.941.
MTP5_ACCEPT = (0.856, 0.694, 0.558, 0.457, 0.376)


def accepted_from_profile(gen, profile, n):
    """n accepted lengths with P(len >= 1 + i) = profile[i - 1]: one uniform
    u per row, len = 1 + #{i : u < profile[i - 1]} (the rates decrease, so
    u < profile[i] implies u < every earlier rate)."""
    u = torch.rand(n, generator=gen, dtype=torch.float64).tolist()
    return [1 + sum(1 for p in profile if x < p) for x in u]


def mtp5(device="cpu", sentinel=True, seed=5, L=36, batch=64, pad_rows=8, HK=16, HV=32,
         KV=128, num_slots=256, state_dtype=F32):
    """The all_layer shapes with window 6 (five drafts) and accepted lengths
    drawn from the measured per-position acceptance rates (MTP5_ACCEPT)."""
    cpu = _gen(seed, "cpu")
    live = batch - pad_rows
    window = 1 + len(MTP5_ACCEPT)
    windows = [window] * live + [0] * pad_rows
    accepted = accepted_from_profile(cpu, MTP5_ACCEPT, live) + [0] * pad_rows
    perm = torch.randperm(num_slots, generator=cpu).tolist()
    slots = [[perm[r]] for r in range(live)] + [[-1]] * pad_rows
    gen = _gen(seed, device)
    return _make("mtp5", HK=HK, HV=HV, K=KV, V=KV, W=window, L=L, windows=windows,
                 accepted=accepted, num_slots=num_slots, slots_for_row=slots,
                 qkv_dtype=BF16, state_dtype=state_dtype, gen=gen, device=device,
                 sentinel=sentinel)


def long_ragged(device="cpu", sentinel=True, seed=30, L=36, batch=256, HK=16, HV=32, KV=128,
                num_slots=512, window=6):
    """Long drafts and ragged windows: half the rows use the full window, the
    rest cycle through 4/1/3 (window-1 rows model decode-only rows); rows sit
    in permuted order with 0-3 unused token rows between them; q/k/v are
    strided views of one fused projection output; gates drawn from U(-20, 20)."""
    cpu = _gen(seed, "cpu")
    ragged = [4, 1, 3]
    windows = [window] * (batch // 2) + [ragged[i % 3] for i in range(batch - batch // 2)]
    windows = [windows[i] for i in torch.randperm(batch, generator=cpu).tolist()]
    accepted = [_ints(cpu, 1, w, 1)[0] for w in windows]
    gaps = _ints(cpu, 0, 3, batch)
    order = torch.randperm(batch, generator=cpu).tolist()
    perm = torch.randperm(num_slots, generator=cpu).tolist()
    slots = [[perm[r]] for r in range(batch)]
    gen = _gen(seed, device)
    return _make("long_ragged", HK=HK, HV=HV, K=KV, V=KV, W=window, L=L, windows=windows,
                 accepted=accepted, num_slots=num_slots, slots_for_row=slots,
                 qkv_dtype=BF16, state_dtype=F32, gen=gen, device=device, sentinel=sentinel,
                 gate_range=20.0, gaps=gaps, row_order=order, fused=True)


def align(device="cpu", sentinel=True, seed=4, L=36, batch=128, HK=16, HV=32, KV=128,
          num_slots=384, window=4, block_size=4, state_dtype=F32, max_blocks=63):
    """Align mode: seq_pos = block*m + r with every (r, accepted) pair equally
    often, so windows end on a boundary, cross one (then the boundary slot is
    the source slot) or stay inside a block.  Each row's block table holds
    distinct slots in the columns the step reads or writes, -1 elsewhere."""
    cpu = _gen(seed, "cpu")
    combos = [(r, n) for r in range(block_size) for n in range(1, window + 1)]
    reps = -(-batch // len(combos))
    pairs = (combos * reps)[:batch]
    pairs = [pairs[i] for i in torch.randperm(batch, generator=cpu).tolist()]
    ms = _ints(cpu, 1, max_blocks, batch)
    seq_pos = [block_size * m + r for m, (r, _) in zip(ms, pairs)]
    accepted = [n for _, n in pairs]
    windows = [window] * batch
    stride = (block_size * max_blocks + block_size - 1 + window - 1) // block_size + 1
    perm = torch.randperm(num_slots, generator=cpu).tolist()
    nxt = 0
    tables = []
    for p0, n in zip(seq_pos, accepted):
        row = [-1] * stride
        # every column the window can touch: checkpoint block to last-token block
        for col in range((p0 - 1) // block_size, (p0 + window - 1) // block_size + 1):
            row[col] = perm[nxt]
            nxt += 1
        tables.append(row)
    assert nxt <= num_slots, "slot pool too small for the block tables"
    gen = _gen(seed, device)
    return _make("align", HK=HK, HV=HV, K=KV, V=KV, W=window, L=L, windows=windows,
                 accepted=accepted, num_slots=num_slots, slots_for_row=tables,
                 seq_pos=seq_pos, block_size=block_size, qkv_dtype=BF16,
                 state_dtype=state_dtype, gen=gen, device=device, sentinel=sentinel)


WORKLOADS = {
    "tiny": tiny,
    "layer": layer,
    "all_layer": all_layer,
    "mtp5": mtp5,
    "long_ragged": long_ragged,
    "align": align,
    "kda_all_layer": kda_all_layer,
}


def custom(device="cpu", sentinel=True, seed=100, *, HK, HV, K, V, W, L, windows, accepted,
           null_rows=(), num_slots=None, block_size=0, seq_pos=None, qkv_dtype=F32,
           state_dtype=F32, gate_range=None, gaps=None, shuffle_rows=False, fused=False,
           kda=False):
    """A small step with explicit per-row windows / accepted lengths, for
    parity cases the oracle runs in full.  Rows listed in null_rows get the
    null slot.  In align mode (block_size > 0) seq_pos must be given and each
    row gets distinct slots for every column its window can touch."""
    cpu = _gen(seed, "cpu")
    B = len(windows)
    if block_size == 0:
        need = B
    else:
        need = sum((p + W - 1) // block_size - (p - 1) // block_size + 1 for p in seq_pos)
    num_slots = num_slots or need + 3
    perm = torch.randperm(num_slots, generator=cpu).tolist()
    tables, nxt = [], 0
    for r in range(B):
        if block_size == 0:
            tables.append([perm[nxt]]); nxt += 1
        else:
            p0 = seq_pos[r]
            row = [-1] * ((p0 + W - 1) // block_size + 1)
            for col in range((p0 - 1) // block_size, (p0 + W - 1) // block_size + 1):
                row[col] = perm[nxt]; nxt += 1
            tables.append(row)
        if r in null_rows:
            tables[-1] = [-1] * len(tables[-1])
    stride = max(len(t) for t in tables)
    tables = [t + [-1] * (stride - len(t)) for t in tables]
    order = torch.randperm(B, generator=cpu).tolist() if shuffle_rows else None
    gen = _gen(seed, device)
    return _make(f"custom{seed}", HK=HK, HV=HV, K=K, V=V, W=W, L=L, windows=list(windows),
                 accepted=list(accepted), num_slots=num_slots, slots_for_row=tables,
                 seq_pos=seq_pos, block_size=block_size, qkv_dtype=qkv_dtype,
                 state_dtype=state_dtype, gen=gen, device=device, sentinel=sentinel,
                 gate_range=gate_range, gaps=gaps, row_order=order, fused=fused, kda=kda)


def conv_state(sb: SpecBatch, state_len: int = 3, dtype=BF16, seed: int = 200):
    """Short-conv states and inputs for every layer of a step: per layer a
    pool [num_slots, C, state_len] ~ N(0, 1) and the convolution inputs of
    every token row, C = 2*HK*K + HV*V channels.  The inputs are the fused
    projection rows when the step has them, else fresh N(0, 1) rows."""
    C = 2 * sb.HK * sb.K + sb.HV * sb.V
    gen = _gen(seed, sb.device)
    pools, inputs = [], []
    for l in range(sb.L):
        pools.append(torch.randn((sb.num_slots, C, state_len), generator=gen, device=sb.device,
                                 dtype=F32).to(dtype))
        if sb.fused_qkv is not None and sb.fused_qkv[l].dtype == dtype:
            inputs.append(sb.fused_qkv[l])
        else:
            inputs.append(torch.randn((sb.T, C), generator=gen, device=sb.device,
                                      dtype=F32).to(dtype))
    return pools, inputs
