"""Host-side checks of libgdn_spec.so that need no GPU: the library builds,
loads, exports every entry point include/gdn_spec.h declares, and rejects
malformed arguments before launching anything."""
import ctypes
import os
import re

import pytest

from spec_decode_recurrent_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*int\s+(gdn_\w+)\s*\(", text, flags=re.M)
            names += re.findall(r"^int\s+(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(api.ENTRY_POINTS) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def _shape(**kw):
    d = dict(num_k_heads=16, num_v_heads=32, head_k=128, head_v=128, max_window=4,
             qkv_dtype=1, state_dtype=0)
    d.update(kw)
    return api.gdn_shape(**d)


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation


def _verify(lib, shape, **over):
    args = dict(batch=2, T=8, slots=4, q=FAKE, qs=2048, k=FAKE, ks=2048, v=FAKE, vs=4096,
                a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, ts=FAKE, wl=FAKE, pool=FAKE, st=FAKE,
                sts=1, sp=None, bs=0, out=FAKE, os=4096, ru=FAKE, rk=FAKE, rg=FAKE, err=None)
    args.update(over)
    sh = ctypes.byref(shape) if shape is not None else None
    return lib.gdn_spec_verify(sh, *[args[k] for k in (
        "batch", "T", "slots", "q", "qs", "k", "ks", "v", "vs", "a", "b", "A_log", "dt_bias",
        "ts", "wl", "pool", "st", "sts", "sp", "bs", "out", "os", "ru", "rk", "rg", "err")], None)


def test_verify_rejects_before_launch(lib):
    assert _verify(lib, None) == -1
    assert _verify(lib, _shape(), q=None) == -1
    assert _verify(lib, _shape(), ru=None) == -1
    assert _verify(lib, _shape(head_k=96)) == -2
    assert _verify(lib, _shape(head_v=256)) == -2
    assert _verify(lib, _shape(max_window=0)) == -2
    assert _verify(lib, _shape(max_window=17)) == -2
    assert _verify(lib, _shape(num_v_heads=24)) == -2          # HV % HK != 0
    assert _verify(lib, _shape(state_dtype=2)) == -2
    assert _verify(lib, _shape(), qs=1024) == -3               # stride shorter than a row
    assert _verify(lib, _shape(), qs=2050) == -3               # stride not a multiple of 4
    assert _verify(lib, _shape(), bs=-1) == -3
    assert _verify(lib, _shape(), bs=4) == -1                  # align mode needs seq_pos
    assert _verify(lib, _shape(), sts=0) == -3
    assert _verify(lib, _shape(), batch=-1) == -3
    assert _verify(lib, _shape(), q=ctypes.c_void_p((1 << 20) + 4)) == -3   # misaligned
    assert _verify(lib, _shape(), pool=ctypes.c_void_p((1 << 20) + 8)) == -3


def test_commit_rejects_before_launch(lib):
    def commit(shape, **over):
        args = dict(L=36, batch=4, slots=8, pools=FAKE, ru=FAKE, rk=FAKE, rg=FAKE, wl=FAKE,
                    al=FAKE, st=FAKE, sts=1, sp=None, bs=0)
        args.update(over)
        sh = ctypes.byref(shape) if shape is not None else None
        return lib.gdn_replay_commit(sh, *[args[k] for k in (
            "L", "batch", "slots", "pools", "ru", "rk", "rg", "wl", "al", "st", "sts", "sp",
            "bs")], None, None)
    assert commit(None) == -1
    assert commit(_shape(), pools=None) == -1
    assert commit(_shape(), al=None) == -1
    assert commit(_shape(head_k=8)) == -2
    assert commit(_shape(), L=0) == -3
    assert commit(_shape(), bs=3) == -1                     # align mode needs seq_pos
    assert commit(_shape(), bs=-2, sp=FAKE) == -3


def test_native_rejects_before_launch(lib):
    sh = _shape()
    args = [2, 8, 4, FAKE, 2048, FAKE, 2048, FAKE, 4096, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
            FAKE, 1, None, 0, FAKE, 4096]
    assert lib.gdn_native_spec_snapshot(ctypes.byref(sh), *args, None, None, None) == -1
    assert lib.gdn_native_spec_snapshot(ctypes.byref(sh), *args,
                                        ctypes.c_void_p((1 << 20) + 4), None, None) == -3


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        api.load()


def test_conv_commit_rejects_before_launch(lib):
    def conv(**over):
        a = dict(L=2, G=1, lg=None, B=4, T=16, slots=8, C=64, SL=3, dt=1, W=4, pools=FAKE,
                 inputs=FAKE, ins=64, ts=FAKE, wl=FAKE, al=FAKE, st=FAKE, sts=1, gs=4, sp=None,
                 bs=0)
        a.update(over)
        return lib.gdn_conv_state_commit(*[a[k] for k in (
            "L", "G", "lg", "B", "T", "slots", "C", "SL", "dt", "W", "pools", "inputs", "ins",
            "ts", "wl", "al", "st", "sts", "gs", "sp", "bs")], None, None)
    assert conv(SL=9) == -2
    assert conv(SL=0) == -2
    assert conv(dt=5) == -2
    assert conv(W=17) == -2
    assert conv(pools=None) == -1
    assert conv(ts=None) == -1
    assert conv(G=2) == -1                      # groups need layer_group
    assert conv(bs=4) == -1                     # align mode needs seq_pos
    assert conv(ins=32) == -3                   # row stride shorter than C
    assert conv(L=0) == -3


def test_kda_entry_points_reject_before_launch(lib):
    # the per-channel (KDA) calls share the scalar-gate calls' checks and
    # also want the [B][HV][W][K] gate record 16-byte aligned
    def kda_verify(shape, **over):
        args = dict(batch=2, T=8, slots=4, q=FAKE, qs=2048, k=FAKE, ks=2048, v=FAKE, vs=4096,
                    a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, ts=FAKE, wl=FAKE, pool=FAKE, st=FAKE,
                    sts=1, sp=None, bs=0, out=FAKE, os=4096, ru=FAKE, rk=FAKE, rg=FAKE, err=None)
        args.update(over)
        sh = ctypes.byref(shape) if shape is not None else None
        return lib.gdn_kda_spec_verify(sh, *[args[k] for k in (
            "batch", "T", "slots", "q", "qs", "k", "ks", "v", "vs", "a", "b", "A_log", "dt_bias",
            "ts", "wl", "pool", "st", "sts", "sp", "bs", "out", "os", "ru", "rk", "rg", "err")],
            None)
    assert kda_verify(None) == -1
    assert kda_verify(_shape(), rg=None) == -1
    assert kda_verify(_shape(head_k=96)) == -2
    assert kda_verify(_shape(), qs=1024) == -3
    assert kda_verify(_shape(), rg=ctypes.c_void_p((1 << 20) + 4)) == -3   # gate record 4-aligned only

    sh = _shape()
    args = [2, 8, 4, FAKE, 2048, FAKE, 2048, FAKE, 4096, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
            FAKE, 1, None, 0, FAKE, 4096]
    assert lib.gdn_kda_native_spec_snapshot(ctypes.byref(sh), *args, None, None, None) == -1
    assert lib.gdn_kda_native_spec_snapshot(ctypes.byref(sh), *args,
                                            ctypes.c_void_p((1 << 20) + 4), None, None) == -3

    def kda_commit(shape, **over):
        a = dict(L=36, batch=4, slots=8, pools=FAKE, ru=FAKE, rk=FAKE, rg=FAKE, wl=FAKE,
                 al=FAKE, st=FAKE, sts=1, sp=None, bs=0)
        a.update(over)
        sh_ = ctypes.byref(shape) if shape is not None else None
        return lib.gdn_kda_replay_commit(sh_, *[a[k] for k in (
            "L", "batch", "slots", "pools", "ru", "rk", "rg", "wl", "al", "st", "sts", "sp",
            "bs")], None, None)
    assert kda_commit(None) == -1
    assert kda_commit(_shape(), rg=None) == -1
    assert kda_commit(_shape(head_v=48)) == -2
    assert kda_commit(_shape(), L=0) == -3
    assert kda_commit(_shape(), bs=3) == -1
