"""The C-ABI library loads, exports every entry point include/kda.h declares,
and rejects bad arguments on the host before touching the GPU.

These run without a GPU: every call here fails validation before any CUDA
call is made (the library links the CUDA runtime statically and reaches the
driver only when it launches).
"""
import ctypes
import os
import re

import pytest
import torch

import gated_delta_rule_21_gb300 as kda
from gated_delta_rule_21_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kda.lib()


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"KDA_API[^;(]*?\b(kda_\w+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    names = declared_symbols()
    for must in ("kda_chunk_fwd", "kda_chunk_fwd_ex", "kda_chunk_fwd_workspace_size",
                 "kda_short_conv_silu", "kda_read_device_status",
                 "kda_clear_device_status", "kda_status_string", "kda_version",
                 "kda_impl_available", "kda_chunk_fwd_workspace_size_for",
                 "kda_chunk_fwd_workspace_size_packed"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), f"libkda.so does not export {name}"


def test_header_compiles_as_c(tmp_path):
    c = tmp_path / "t.c"
    c.write_text('#include "kda.h"\nint main(void){return kda_version()==0;}\n')
    import subprocess
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", str(c), "-I",
                    os.path.join(ROOT, "include"), "-o", str(tmp_path / "t.o")], check=True)


def test_version_and_status_strings(L):
    assert kda.version() == 100
    for st in range(8):
        assert kda.status_string(st)
    assert kda.status_string(99) == "unknown status"


def test_workspace_size_formula(L):
    # the smallest workspace: the header, plus with segment ids the row
    # offsets (B+1 ints rounded to 256 B) and 8 B per possible run
    assert kda.workspace_size(1, 8192, 32, 128, 128, impl="simt") == 256
    assert kda.workspace_size(2, 1000, 4, 64, 64, has_segment_ids=True, impl="simt") == \
        256 + 256 + 8 * 2000
    s = kda.kda_shape(1, 16, 1, 48, 128, 1)   # unsupported K
    assert L.kda_chunk_fwd_workspace_size(ctypes.byref(s), 0) == 0


@pytest.mark.parametrize("shape,seg", [((1, 8192, 32, 128, 128), False),
                                       ((1, 8192, 32, 128, 128), True),
                                       ((2, 1000, 4, 64, 64), True),
                                       ((1, 128, 2, 128, 128), False)])
def test_default_workspace_size_is_the_fast_path_size(L, shape, seg):
    # The default query returns what AUTO needs for its fastest kernel: for
    # bf16 K = V = 128 the split path's size, so a caller that follows the
    # basic recipe (query, allocate, call) gets the split kernels.
    B, T, H, K, V = shape
    d = kda.workspace_size(B, T, H, K, V, has_segment_ids=seg)
    assert d == kda.workspace_size(B, T, H, K, V, has_segment_ids=seg, impl="auto")
    split = kda.workspace_size(B, T, H, K, V, has_segment_ids=seg, impl="split")
    if K == V == 128:
        assert d == split > kda.workspace_size(B, T, H, K, V, has_segment_ids=seg, impl="simt")
    else:
        assert split == 0
        assert d == kda.workspace_size(B, T, H, K, V, has_segment_ids=seg, impl="simt")


FAKE = 0x10000  # a 256-byte aligned address; never dereferenced


def call_fwd(L, shape=(1, 128, 2, 128, 128, 1), q=FAKE, k=FAKE, v=FAKE, g=FAKE,
             beta=FAKE, chunk=64, s0=None, seg=None, o=FAKE, fs=None, ws=FAKE,
             ws_bytes=1 << 20, impl=0, v_tile=0, scale=0.1):
    s = kda.kda_shape(*shape)
    vp = ctypes.c_void_p
    return L.kda_chunk_fwd_ex(ctypes.byref(s), vp(q), vp(k), vp(v), vp(g), vp(beta),
                              scale, chunk, vp(s0), vp(seg), vp(o), vp(fs), vp(ws),
                              ws_bytes, impl, v_tile, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(beta=None), 1),
    (dict(shape=(0, 128, 2, 128, 128, 1)), 1),
    (dict(shape=(1, 128, 2, 128, 128, 7)), 1),
    (dict(shape=(1, 128, 2, 96, 128, 1)), 2),
    (dict(shape=(1, 128, 2, 128, 16, 1)), 2),
    (dict(chunk=32), 2),
    (dict(q=FAKE + 2), 3), (dict(g=FAKE + 4), 3), (dict(s0=FAKE + 8), 3),
    (dict(ws=None), 4), (dict(ws_bytes=16), 4),
    (dict(seg=FAKE, ws_bytes=300), 4),
    (dict(ws=FAKE + 16), 3),
    (dict(impl=9), 1), (dict(v_tile=-1), 1), (dict(scale=float("nan")), 1),
    (dict(impl=1, v_tile=48), 2),
    (dict(impl=2, shape=(1, 128, 2, 64, 64, 1)), 2),
    (dict(impl=2, shape=(1, 128, 2, 128, 128, 0)), 2),
])
def test_forward_rejects_bad_arguments_without_launching(L, kw, expect):
    assert call_fwd(L, **kw) == expect


def call_noalloc(L, shape=(1, 128, 2, 128, 128, 1), q=FAKE, k=FAKE, v=FAKE, g=FAKE,
                 beta=FAKE, chunk=64, s0=None, seg=None, o=FAKE, fs=None, scale=0.1):
    s = kda.kda_shape(*shape)
    vp = ctypes.c_void_p
    return L.kda_chunk_fwd_noalloc(ctypes.byref(s), vp(q), vp(k), vp(v), vp(g), vp(beta),
                                   scale, chunk, vp(s0), vp(seg), vp(o), vp(fs), None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(beta=None), 1),
    (dict(shape=(0, 128, 2, 128, 128, 1)), 1),
    (dict(shape=(1, 0, 2, 128, 128, 1)), 1),
    (dict(shape=(1, 128, 2, 128, 128, 7)), 1),
    (dict(shape=(1, 128, 2, 96, 128, 1)), 2),
    (dict(chunk=32), 2),
    (dict(q=FAKE + 2), 3), (dict(g=FAKE + 4), 3), (dict(s0=FAKE + 8), 3),
    (dict(scale=float("nan")), 1),
    # the run list of 200000 tokens does not fit the fixed array
    (dict(shape=(1, 200000, 1, 32, 32, 1), seg=FAKE), 4),
])
def test_noalloc_rejects_bad_arguments_like_the_workspace_entry_point(L, kw, expect):
    assert call_noalloc(L, **kw) == expect
    if "shape" not in kw or kw["shape"][1] != 200000:
        # kda_chunk_fwd returns the same code for the same input
        kw2 = {k: v for k, v in kw.items()}
        assert call_fwd(L, **kw2) == expect


def test_noalloc_status_rejects_null(L):
    assert L.kda_chunk_fwd_noalloc_status(None, None) == 1


def test_conv_rejects_bad_arguments(L):
    s = kda.kda_shape(1, 64, 2, 128, 128, 1)
    vp = ctypes.c_void_p
    f = lambda *a: L.kda_short_conv_silu(ctypes.byref(s), *[vp(x) for x in a[:5]], 1,
                                         *[vp(x) for x in a[5:]], None)
    assert f(FAKE, FAKE, FAKE, None, None, FAKE + 256, FAKE + 512, FAKE + 768) == 1
    assert f(FAKE + 2, FAKE, FAKE, FAKE, None, FAKE + 256, FAKE + 512, FAKE + 768) == 3
    assert f(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE + 512, FAKE + 768) == 1  # aliasing


def test_impl_available_query(L):
    assert kda.impl_available("simt", 1, 64, 1, 128, 128)
    assert kda.impl_available("auto", 1, 64, 1, 64, 32, torch.float32)
    assert not kda.impl_available("simt", 1, 64, 1, 128, 128, v_tile=48)
    assert not kda.impl_available("tc", 1, 64, 1, 64, 64)
    assert not kda.impl_available("tc", 1, 64, 1, 128, 128, torch.float32)


def test_workspace_size_for_each_impl(L):
    base = kda.workspace_size(1, 8192, 32, 128, 128, impl="simt")
    split = kda.workspace_size(1, 8192, 32, 128, 128, impl="split")
    assert split == 1024 + 128 * 32 * 74240          # one 72.5 KiB item per chunk-head
    assert kda.workspace_size(1, 8192, 32, 128, 128, impl="auto") == split
    assert kda.workspace_size(1, 8192, 32, 128, 128, impl="tc") == base
    # packed: header + run list + chunk tables, then B*(ceil(T/64) + runs bound) items
    packed = kda.workspace_size(1, 100, 2, 128, 128, has_segment_ids=True, impl="split")
    assert packed == kda.workspace_size_packed(1, 100, 2, 128, 128, 2)
    assert kda.workspace_size_packed(1, 100, 2, 128, 128, 5) - \
        kda.workspace_size_packed(1, 100, 2, 128, 128, 2) == 3 * 2 * 74240
    assert kda.workspace_size_packed(1, 100, 2, 128, 128, 0) == 0
    assert kda.workspace_size_packed(1, 100, 2, 64, 64, 3) == 0
    assert kda.workspace_size(1, 100, 2, 64, 64, impl="split") == 0
    assert kda.workspace_size(1, 100, 2, 128, 128, torch.float32, impl="auto") == \
        kda.workspace_size(1, 100, 2, 128, 128, torch.float32, impl="simt")


def test_split_rejects_small_workspace(L):
    assert call_fwd(L, impl=3, ws_bytes=4096) == 4
    assert call_fwd(L, impl=3, seg=FAKE, ws_bytes=8192) == 4


def test_status_calls_reject_null(L):
    bits = ctypes.c_uint32(0)
    assert L.kda_read_device_status(None, None, ctypes.byref(bits)) == 1
    assert L.kda_clear_device_status(None, None) == 1


def test_backward_workspace_size_and_argument_checks(L):
    # supported: K in {32, 64, 128}, V a multiple of 32
    n = kda.bwd_workspace_size(1, 8192, 32, 128, 128, impl="simt")
    nck, n_vt, nK, nB = 8192 // 8, 4, 8192 * 32 * 128, 8192 * 32
    assert n == 256 + 152 * nck * 128 * 32 * 4 + 3 * n_vt * nK * 4 + n_vt * nB * 4
    # the tensor-core path (AUTO for bf16, K = V = 128, no segment ids): the
    # header, then per (chunk, head) an item of 112.5 KiB and 96 KiB of saves
    tc = kda.bwd_workspace_size(1, 8192, 32, 128, 128, impl="tc")
    assert tc == 1024 + 128 * 32 * (115200 + 98304)
    assert kda.bwd_workspace_size(1, 8192, 32, 128, 128) == tc
    assert kda.bwd_workspace_size(1, 8192, 32, 128, 128, impl="auto") == tc
    assert kda.bwd_workspace_size(1, 100, 2, 128, 128, torch.float32, impl="tc") == 0
    assert kda.bwd_workspace_size(1, 100, 2, 64, 64, impl="tc") == 0
    # with segment ids: the run list and chunk tables, then items and saves for
    # ceil(T/64) chunks per row plus ceil(T/64) runs per row (AUTO's size), or
    # a bound of the caller's choice
    tcs = kda.bwd_workspace_size(1, 100, 2, 128, 128, has_segment_ids=True, impl="tc")
    assert tcs == kda.bwd_workspace_size(1, 100, 2, 128, 128, has_segment_ids=True)
    assert tcs == kda.bwd_workspace_size_packed(1, 100, 2, 128, 128, max_runs_per_row=2)
    per_chunk = 2 * (115200 + 98304)
    assert kda.bwd_workspace_size_packed(1, 100, 2, 128, 128, 5) == tcs + 3 * per_chunk
    assert kda.bwd_workspace_size_packed(1, 100, 2, 128, 128, 0) == 0
    assert kda.bwd_workspace_size_packed(1, 100, 2, 64, 64, 4) == 0
    assert kda.bwd_workspace_size(1, 100, 2, 64, 64, has_segment_ids=True) == \
        kda.bwd_workspace_size(1, 100, 2, 64, 64, has_segment_ids=True, impl="simt")
    assert kda.bwd_workspace_size(1, 100, 2, 64, 64) == \
        kda.bwd_workspace_size(1, 100, 2, 64, 64, impl="simt")
    assert kda.bwd_workspace_size(1, 100, 2, 64, 64, has_segment_ids=True) > \
        kda.bwd_workspace_size(1, 100, 2, 64, 64)
    assert kda.bwd_workspace_size(1, 0, 2, 128, 128) == 0
    s = kda.kda_shape(1, 64, 2, 128, 128, 1)
    nb = kda.bwd_workspace_size(1, 64, 2, 128, 128)
    vp = ctypes.c_void_p

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.1, chunk=64, s0=None,
                 seg=None, d_o=FAKE, d_f=None, dq=FAKE, dk=FAKE, dv=FAKE, dg=FAKE, db=FAKE,
                 di=None, ws=FAKE, nbytes=nb)
        a.update(kw)
        p = lambda x: None if x is None else vp(x)
        return L.kda_chunk_bwd(ctypes.byref(s), p(a["q"]), p(a["k"]), p(a["v"]), p(a["g"]),
                               p(a["beta"]), a["scale"], a["chunk"], p(a["s0"]), p(a["seg"]),
                               p(a["d_o"]), p(a["d_f"]), p(a["dq"]), p(a["dk"]), p(a["dv"]),
                               p(a["dg"]), p(a["db"]), p(a["di"]), p(a["ws"]), a["nbytes"], None)
    assert call(d_o=None) == 1                 # NULL d_o
    assert call(dq=None) == 1                  # NULL output
    assert call(chunk=32) == 2                 # chunk size
    assert call(scale=float("nan")) == 1
    assert call(d_o=FAKE + 4) == 3             # misaligned
    assert call(nbytes=nb - 1) == 4            # small workspace
    assert call(ws=FAKE + 16) == 3          # workspace not 256-byte aligned
    # explicit implementations
    def call_ex(impl, shape=(1, 64, 2, 128, 128, 1), seg=None, nbytes=None):
        s2 = kda.kda_shape(*shape)
        nbx = nb if nbytes is None else nbytes
        return L.kda_chunk_bwd_ex(ctypes.byref(s2), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                  vp(FAKE), 0.1, 64, None, None if seg is None else vp(seg),
                                  vp(FAKE), None, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                  vp(FAKE), None, vp(FAKE), nbx, impl, None)
    assert call_ex(7) == 1                                      # unknown impl
    assert call_ex(2, shape=(1, 64, 2, 64, 64, 1)) == 2          # TC: K, V
    assert call_ex(2, shape=(1, 64, 2, 128, 128, 0)) == 2        # TC: fp32 inputs
    min_seg = kda.bwd_workspace_size_packed(1, 64, 2, 128, 128, 1) - 2 * (115200 + 98304)
    assert call_ex(2, seg=FAKE, nbytes=min_seg - 1) == 4         # TC: room for T's chunks
    assert call_ex(2, nbytes=nb - 1) == 4                        # TC: small workspace
    simt_nb = kda.bwd_workspace_size(1, 64, 2, 128, 128, impl="simt")
    assert call_ex(1, nbytes=simt_nb - 1) == 4                   # SIMT: its own size
    # the training-step pair: the tensor-core backward's workspace and shapes
    assert kda.fwd_save_workspace_size(1, 64, 2, 128, 128) == \
        kda.bwd_workspace_size(1, 64, 2, 128, 128, impl="tc")
    assert kda.fwd_save_workspace_size(1, 64, 2, 64, 64) == 0
    assert kda.fwd_save_workspace_size(1, 64, 2, 128, 128, torch.float32) == 0

    def call_save(shape=(1, 64, 2, 128, 128, 1), o=FAKE, nbytes=None, chunk=64, ws=FAKE):
        s2 = kda.kda_shape(*shape)
        return L.kda_chunk_fwd_save(ctypes.byref(s2), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                    vp(FAKE), 0.1, chunk, None, None, None if o is None else vp(o),
                                    None, None if ws is None else vp(ws),
                                    nb if nbytes is None else nbytes, None)
    assert call_save(o=None) == 1
    assert call_save(chunk=32) == 2
    assert call_save(shape=(1, 64, 2, 64, 64, 1)) == 2
    assert call_save(shape=(1, 64, 2, 128, 128, 0)) == 2
    assert call_save(o=FAKE + 2) == 3
    assert call_save(nbytes=nb - 1) == 4
    assert call_save(ws=None) == 4
    assert call_save(ws=FAKE + 16) == 3

    def call_from_saved(shape=(1, 64, 2, 128, 128, 1), nbytes=None, d_o=FAKE):
        s2 = kda.kda_shape(*shape)
        return L.kda_chunk_bwd_from_saved(ctypes.byref(s2), vp(FAKE), vp(FAKE), vp(FAKE),
                                          vp(FAKE), vp(FAKE), 0.1, 64, None, None,
                                          None if d_o is None else vp(d_o), None, vp(FAKE),
                                          vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None,
                                          vp(FAKE), nb if nbytes is None else nbytes, None)
    assert call_from_saved(d_o=None) == 1
    assert call_from_saved(shape=(1, 64, 2, 64, 64, 1)) == 2
    assert call_from_saved(nbytes=nb - 1) == 4
    s48 = kda.kda_shape(1, 64, 2, 128, 48, 1)
    assert L.kda_chunk_bwd_workspace_size(ctypes.byref(s48), 0) == 0
