"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
a SpecBatch, build the expected pools from the GPU native snapshots (for the
bit-exact checks) and run the fp64 oracle (for the tolerance checks)."""
import random

import numpy as np
import torch

import oracle
from spec_decode_recurrent_gb300 import step
from tests._tol import check_bf16, check_close

NAN = float("nan")


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def cpu64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def row_plan(sb, r):
    """(src, [(slot, ntok), ...]) from the oracle's plan for row r; a
    malformed row plans no writes."""
    sp = int(sb.seq_pos[r]) if sb.seq_pos is not None else 0
    try:
        return oracle.commit_plan(int(sb.window_len[r]), int(sb.accepted_len[r]),
                                  sb.slot_table[r].cpu(), sp, sb.block_size, sb.num_slots, sb.W)
    except ValueError:
        return -1, []


def snapshot_mask(sb):
    """[B, W] bool: True where the native kernel must write the snapshot
    (live rows, positions t < window_len), False where it must not."""
    mask = np.zeros((sb.B, sb.W), dtype=bool)
    win, start = sb.window_len.tolist(), sb.token_start.tolist()
    table = sb.slot_table.cpu()
    for r in range(sb.B):
        sp = int(sb.seq_pos[r]) if sb.seq_pos is not None else 0
        src = oracle.source_slot(win[r], table[r], sp, sb.block_size, sb.num_slots, sb.W)
        if src >= 0 and 0 <= start[r] and start[r] + win[r] <= sb.T:
            mask[r, :win[r]] = True
    return mask


class GpuStep:
    """Runs verify (all layers), native snapshots (all layers) and the
    all-layer commit, keeping what the checks need.

    expected[l] is the pool the commit must produce, built from the native
    kernel's snapshots: the bit-exact reference for the commit.

    Snapshots: with keep_snaps every layer's full snapshot array is kept
    (small steps, compared element by element with the oracle); otherwise
    only the snapshot rows of `units` sampled live (layer, row, head) units
    are kept.  In both cases every layer's snapshot array is checked on the
    device: each (row, position) block is finite where the kernel must write
    it and still the NaN fill where it must not (positions at or past the
    row's window, null and empty rows)."""

    def __init__(self, sb, native=True, keep_snaps=None, units=0, unit_seed=0):
        self.sb = sb
        self.plans = [row_plan(sb, r) for r in range(sb.B)]
        self.unit_list = self._pick_units(units, unit_seed)
        if keep_snaps is None:
            keep_snaps = sb.B * sb.W * sb.HV * sb.V * sb.K * sb.L <= (1 << 24)
        self.snaps = [None] * sb.L
        self.unit_snaps = {}
        self.before = [p.clone() for p in sb.pools]
        self.bufs = step.StepBuffers(sb, fill=NAN)
        step.verify_all(sb, self.bufs)
        self.native_out = []
        self.expected = []
        self.verify_err = None
        self.snapshot_mask_ok = None
        if native:
            want = torch.tensor(snapshot_mask(sb), device=sb.device)
            mask_ok = True
            for l in range(sb.L):
                out, snaps = step.native_buffers(sb, fill=NAN)
                step.native_layer(sb, l, out, snaps)
                self.native_out.append(out)
                flat = snaps.view(sb.B, sb.W, -1)
                written = torch.isfinite(flat).all(-1)
                untouched = torch.isnan(flat).all(-1)
                mask_ok &= bool(torch.equal(written, want)) and bool(torch.equal(untouched, ~want))
                exp = sb.pools[l].clone()
                rows, slots, tok = [], [], []
                for r, (src, writes) in enumerate(self.plans):
                    for slot, ntok in writes:
                        rows.append(r); slots.append(slot); tok.append(ntok - 1)
                if rows:
                    dev = sb.device
                    exp[torch.tensor(slots, device=dev)] = snaps[torch.tensor(rows, device=dev),
                                                                 torch.tensor(tok, device=dev)]
                self.expected.append(exp)
                if keep_snaps:
                    self.snaps[l] = snaps
                for (ul, r, h) in self.unit_list:
                    if ul == l:
                        self.unit_snaps[(l, r, h)] = snaps[r, :, h].clone()
                del flat, written, untouched
                if not keep_snaps:
                    del snaps
            self.snapshot_mask_ok = mask_ok
        torch.cuda.synchronize()
        self.pools_after_verify_equal = all(
            torch.equal(bits(a), bits(b)) for a, b in zip(self.before, sb.pools))
        self.verify_err = int(self.bufs.err.item())
        step.commit(sb, self.bufs)
        torch.cuda.synchronize()
        self.err = int(self.bufs.err.item())

    def check_bitwise(self):
        sb = self.sb
        assert self.pools_after_verify_equal, "verify wrote into the checkpoint pool"
        assert self.snapshot_mask_ok, \
            "native snapshots: a position inside a live window is unwritten or one outside was written"
        for l in range(sb.L):
            a, b = self.bufs.out[l], self.native_out[l]
            assert torch.equal(bits(a), bits(b)), f"layer {l}: verify out != native out"
            assert torch.equal(bits(sb.pools[l]), bits(self.expected[l])), \
                f"layer {l}: committed pool != native snapshots (or a stray write)"

    def _pick_units(self, n, seed):
        """n random live (layer, row, head) units."""
        live = [r for r, (src, _) in enumerate(self.plans) if src >= 0]
        if n <= 0 or not live:
            return []
        rnd = random.Random(seed)
        return [(rnd.randrange(self.sb.L), rnd.choice(live), rnd.randrange(self.sb.HV))
                for _ in range(n)]

    def check_unit_against_oracle(self, l, r, h):
        """The oracle recomputes one (layer, row, head) from the raw inputs:
        outputs, record, every native snapshot of the window and the
        committed states are compared element by element."""
        sb = self.sb
        w = int(sb.window_len[r])
        t0 = int(sb.token_start[r])
        hk = h // (sb.HV // sb.HK)
        src, writes = self.plans[r]
        S0 = cpu64(self.before[l][src, h])
        sl = slice(t0, t0 + w)
        if sb.kda:
            ref = oracle.kda_window(S0, cpu64(sb.q[l][sl, hk]), cpu64(sb.k[l][sl, hk]),
                                    cpu64(sb.v[l][sl, h]), cpu64(sb.a[l][sl, h]),
                                    cpu64(sb.b[l][sl, h]), float(sb.A_log[l][h]),
                                    cpu64(sb.dt_bias[l][h]))
        else:
            ref = oracle.window(S0, cpu64(sb.q[l][sl, hk]), cpu64(sb.k[l][sl, hk]),
                                cpu64(sb.v[l][sl, h]), cpu64(sb.a[l][sl, h]),
                                cpu64(sb.b[l][sl, h]), float(sb.A_log[l][h]),
                                float(sb.dt_bias[l][h]))
        tag = f"layer {l} row {r} head {h}"
        check_close(cpu64(self.bufs.out[l][sl, h]), ref["o"], f"{tag}: out")
        check_close(cpu64(self.bufs.rec_u[l][r, h, :w]), ref["u"], f"{tag}: record u")
        check_close(cpu64(self.bufs.rec_k[l][r, h, :w]), ref["khat"], f"{tag}: record khat")
        check_close(cpu64(self.bufs.rec_g[l][r, h, :w]), ref["alpha"], f"{tag}: record gate")
        check = check_close if sb.state_dtype == torch.float32 else check_bf16
        if (l, r, h) in self.unit_snaps:
            snap = cpu64(self.unit_snaps[(l, r, h)])
            check(snap[:w], ref["states"], f"{tag}: native snapshots")
            assert np.all(np.isnan(snap[w:])), f"{tag}: native snapshot written past the window"
        for slot, ntok in writes:
            check(cpu64(sb.pools[l][slot, h]), ref["states"][ntok - 1],
                  f"{tag}: state after {ntok} tokens")


def oracle_full(sb, pools_before):
    """Run the oracle on the whole (small) step from the checkpoint pools as
    they were before the GPU commit: verify with snapshots per layer, then
    the all-layer commit from the oracle's own records."""
    sp = None if sb.seq_pos is None else sb.seq_pos.cpu()
    layers = []
    verify = oracle.kda_spec_verify if sb.kda else oracle.spec_verify
    for l in range(sb.L):
        layers.append(verify(
            q=sb.q[l].cpu(), k=sb.k[l].cpu(), v=sb.v[l].cpu(), a=sb.a[l].cpu(), b=sb.b[l].cpu(),
            A_log=sb.A_log[l].cpu(), dt_bias=sb.dt_bias[l].cpu(), token_start=sb.token_start.cpu(),
            window_len=sb.window_len.cpu(), pool=pools_before[l].cpu(), slot_table=sb.slot_table.cpu(),
            seq_pos=sp, block_size=sb.block_size, max_window=sb.W, snapshots=True))
    commit = oracle.kda_replay_commit if sb.kda else oracle.replay_commit
    pools, err = commit(
        pools=np.stack([cpu64(p) for p in pools_before]),
        rec_u=np.stack([x["rec_u"] for x in layers]), rec_k=np.stack([x["rec_k"] for x in layers]),
        rec_g=np.stack([x["rec_g"] for x in layers]), window_len=sb.window_len.cpu(),
        accepted_len=sb.accepted_len.cpu(), slot_table=sb.slot_table.cpu(), seq_pos=sp,
        block_size=sb.block_size, max_window=sb.W)
    return layers, pools, err


def compare_full(gs: GpuStep, layers, pools_ref):
    """Element-by-element comparison of every output of a small step.
    Entries the oracle leaves NaN (not written) must be NaN on the GPU
    too (the buffers start as NaN)."""
    sb = gs.sb
    for l in range(sb.L):
        for name, gpu in (("out", gs.bufs.out[l]), ("rec_u", gs.bufs.rec_u[l]),
                          ("rec_k", gs.bufs.rec_k[l]), ("rec_g", gs.bufs.rec_g[l])):
            g, ref = cpu64(gpu), layers[l][name]
            written = ~np.isnan(ref)
            assert np.array_equal(np.isnan(g), ~written), f"layer {l} {name}: write mask differs"
            check_close(g[written], ref[written], f"layer {l} {name}")
        # every native snapshot [row, position] against the oracle's state
        # after that token; positions the oracle leaves unwritten (at or past
        # the window, null and empty rows) must still hold the NaN fill
        assert gs.snaps[l] is not None, "compare_full needs the full snapshots (keep_snaps)"
        g, ref = cpu64(gs.snaps[l]), layers[l]["snaps"]
        written = ~np.isnan(ref)
        assert np.array_equal(np.isnan(g), ~written), f"layer {l} snapshots: write mask differs"
        if sb.state_dtype == torch.float32:
            check_close(g[written], ref[written], f"layer {l} native snapshots")
        else:
            check_bf16(g[written], ref[written], f"layer {l} native bf16 snapshots")
        got = cpu64(sb.pools[l])
        ref = pools_ref[l]
        before = cpu64(gs.before[l])
        changed = ~((ref == before) | (np.isnan(ref) & np.isnan(before)))
        same = ~changed
        assert np.array_equal(bits(sb.pools[l]).cpu().numpy()[same],
                              bits(gs.before[l]).cpu().numpy()[same]), \
            f"layer {l}: an unplanned pool element changed"
        if sb.state_dtype == torch.float32:
            check_close(got[changed], ref[changed], f"layer {l} committed state")
        else:
            check_bf16(got[changed], ref[changed], f"layer {l} committed bf16 state")
