"""C-ABI library checks that need no GPU: it loads, it exports every symbol
include/ps.h declares, and host-side validation rejects bad arguments before
any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_symbols():
    text = open(os.path.join(ROOT, "include", "ps.h")).read()
    return sorted(set(re.findall(r"\b(ps_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def test_library_exports_every_declared_symbol(ps):
    syms = _header_symbols()
    assert "ps_decode" in syms and "ps_kv_append" in syms and "ps_prefill" in syms
    raw = ctypes.CDLL(ps._lib.LIB_PATH)
    for s in syms:
        assert hasattr(raw, s), s
    assert set(syms) <= set(ps._lib.EXPORTS) | set()


def test_build_targets_sm_103a_only():
    """The build compiles every kernel for sm_103a and nothing else (the GPU test
    asks the runtime which code it loaded)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_ps_build", os.path.join(ROOT, "prefix_sliding_window_02_b300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_decode_append_host_validation(ps):
    desc = ps.CacheDesc()
    f = ctypes.c_void_p(1 << 20)
    # k / v missing, then an invalid descriptor: refused before any CUDA call
    assert ps.lib.ps_decode_append(ctypes.byref(desc), f, None, f, f, 16, ctypes.c_float(0.1), f, f,
                                   f, 0, None) == 1
    assert ps.lib.ps_decode_append(ctypes.byref(desc), f, f, f, f, 16, ctypes.c_float(0.1), f, f,
                                   f, 0, None) == 1


def test_code_version_query_needs_a_device(ps):
    v = ctypes.c_int32(0)
    assert ps.lib.ps_device_code_version(None) == 1
    import torch
    if not torch.cuda.is_available():
        assert ps.lib.ps_device_code_version(ctypes.byref(v)) == 5  # PS_ERR_CUDA


@pytest.mark.gpu
def test_loaded_kernels_are_sm_103(ps):
    v = ctypes.c_int32(0)
    assert ps.lib.ps_device_code_version(ctypes.byref(v)) == 0
    assert v.value == 103


def test_status_strings(ps):
    for code, name in enumerate(["PS_OK", "PS_ERR_INVALID_ARGUMENT", "PS_ERR_UNSUPPORTED",
                                 "PS_ERR_ALIGNMENT", "PS_ERR_WORKSPACE", "PS_ERR_CUDA",
                                 "PS_ERR_DEVICE"]):
        assert ps.lib.ps_status_string(code).decode() == name


def test_host_validation_rejects_before_launch(ps):
    lib = ps.lib
    nq, nk = ctypes.c_int32(), ctypes.c_int32()
    assert lib.ps_prefill_tile_grid(0, 0, 1, 1, 0, 128, 128, ctypes.byref(nq), ctypes.byref(nk)) == 1
    assert lib.ps_prefill_tile_grid(10, 0, -1, 1, 0, 128, 128, ctypes.byref(nq), ctypes.byref(nk)) == 1
    assert lib.ps_prefill_tile_grid(10, 0, 1, 0, 0, 128, 128, ctypes.byref(nq), ctypes.byref(nk)) == 1
    assert lib.ps_ring_slots(None, None, 0, None, 5, None) == 1           # W < 1
    assert lib.ps_ring_slots(None, None, 4, None, 0, None) == 0           # nothing to do
    assert lib.ps_kv_append(None, None, None, None, 0, None, None, 1, None) == 1
    b = ctypes.c_size_t()
    assert lib.ps_decode_workspace_size(4, 3, 2, 128, ctypes.byref(b)) == 1   # Hq % Hkv
    assert lib.ps_decode_workspace_size(4, 32, 2, 128, ctypes.byref(b)) == 2  # group 16
    assert lib.ps_decode_workspace_size(4, 16, 8, 96, ctypes.byref(b)) == 2   # head_dim
    assert lib.ps_decode_workspace_size(0, 16, 8, 128, ctypes.byref(b)) == 1
    desc = ps.CacheDesc()
    assert lib.ps_decode(ctypes.byref(desc), None, None, 16, ctypes.c_float(0.1), None, None,
                         None, 0, None) == 1
    flags = ctypes.c_int32()
    assert lib.ps_check_device_status(None, ctypes.byref(flags)) == 1


def _bad_desc(ps, **kw):
    d = dict(k_pool=4096, v_pool=8192, slot_base=256, prefix_len=512, status=0, total_slots=100,
             nseq=1, n_kv_heads=1, head_dim=128, window=4, capacity=10, prefix_max=6,
             rope_theta=1e4)
    d.update(kw)
    return ps.CacheDesc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(window=0), 1), (dict(capacity=9), 1), (dict(head_dim=96), 2), (dict(k_pool=4100), 3),
    (dict(rope_theta=0.0), 1), (dict(nseq=0), 1), (dict(total_slots=2**31), 1)])
def test_cache_descriptor_validation(ps, kw, code):
    d = _bad_desc(ps, **kw)
    r = ps.lib.ps_kv_append(ctypes.byref(d), 16, 16, 16, 1, 4096, 4096, 1, None)
    assert r == code


@pytest.mark.parametrize("kw,code", [
    (dict(block_table=1024, block_size=8, blocks_per_seq=2), 1),    # block not a multiple of 16
    (dict(block_table=1024, block_size=16, blocks_per_seq=0), 1),   # too few blocks per sequence
    (dict(block_table=1024, block_size=32, blocks_per_seq=1, capacity=40), 1),  # 32 < capacity
    (dict(slot_base=0), 1),                                          # contiguous needs slot_base
    (dict(pe_mode=2), 1),                                            # unknown position encoding
])
def test_paged_descriptor_validation(ps, kw, code):
    d = _bad_desc(ps, **kw)
    r = ps.lib.ps_kv_append(ctypes.byref(d), 16, 16, 16, 1, 4096, 4096, 1, None)
    assert r == code


def test_tile_grid_matches_oracle_shapes(ps):
    from oracle import tile_classes
    for S, q0, P, W, ring, bm, bn in [(1000, 0, 37, 300, 0, 128, 128), (70, 5, 9, 13, 0, 16, 8),
                                      (50, 600, 40, 100, 1, 16, 16), (50, 30, 40, 100, 1, 8, 8)]:
        nq, nk = ps.prefill_tile_grid(S, q0, P, W, bool(ring), bm, bn)
        if ring:
            n_pre = min(P, q0)
            wlo = max(P, q0 - W)
            kpos = list(range(n_pre)) + list(range(wlo, q0)) + list(range(q0, q0 + S))
        else:
            kpos = list(range(q0, q0 + S))
        c = tile_classes(np.arange(q0, q0 + S), np.array(kpos), P, W, bm, bn)
        assert (nq, nk) == c.shape


def test_backward_host_validation(ps):
    """ps_prefill_backward rejects bad arguments before any CUDA call."""
    lib = ps.lib
    b = ctypes.c_size_t()
    assert lib.ps_prefill_backward_workspace_size(1, 300, 4, 2, 128, ctypes.byref(b)) == 0
    need = b.value
    # rotated Q (1 x 300 x 4 x 128 bf16), rotated K, {LSE, D} pairs over 384 padded rows
    assert need >= 300 * 4 * 128 * 2 + 300 * 2 * 128 * 2 + 4 * 384 * 8
    assert lib.ps_prefill_backward_workspace_size(1, 300, 4, 3, 128, ctypes.byref(b)) == 1  # Hq % Hkv
    assert lib.ps_prefill_backward_workspace_size(1, 300, 4, 2, 96, ctypes.byref(b)) == 2   # head_dim
    assert lib.ps_prefill_backward_workspace_size(1, 300, 4, 2, 64, ctypes.byref(b)) == 0
    assert lib.ps_prefill_backward_workspace_size(1, 300, 4, 2, 128, ctypes.byref(b)) == 0
    assert lib.ps_prefill_backward_workspace_size(0, 300, 4, 2, 128, ctypes.byref(b)) == 1
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first
    odd = ctypes.c_void_p((1 << 20) + 2)
    i32 = ctypes.c_void_p(1 << 21)
    f = ctypes.c_void_p(1 << 22)

    def call(q=fake, W=64, hd=128, ws=fake, ws_bytes=need, dq=f, scale=0.088, fwd=None):
        return lib.ps_prefill_backward(q, fake, fake, fake, f, fake, 1, 300, i32, i32, W, 4, 2, hd,
                                       ctypes.c_float(scale), ctypes.c_double(1e4), fwd, dq, f, f,
                                       ws, ws_bytes, None, None)

    assert call(q=None) == 1          # null pointer
    assert call(W=0) == 1             # window < 1
    assert call(scale=0.0) == 1       # scale must be positive
    assert call(hd=96) == 2           # head_dim 64 or 128 only
    assert call(q=odd) == 3           # 16-byte alignment
    assert call(ws=None) == 4         # no workspace
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == 4  # workspace not 256-byte aligned
    assert call(ws_bytes=need - 1) == 4  # workspace too small
    assert call(fwd=ctypes.c_void_p((1 << 20) + 16)) == 4  # forward workspace not 256-byte aligned


def test_prefill_position_encoding_validation(ps):
    """ps_prefill takes PS_PE_CONTINUE or PS_PE_RESET, and with a ring only the
    ring's own mode; ps_prefill_workspace_size grows by one query array under
    Reset PE.  All refused on the host, before any CUDA call."""
    lib = ps.lib
    b0, b1 = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.ps_prefill_workspace_size(2, 300, 4, 2, 128, 0, 0, ctypes.byref(b0)) == 0
    assert lib.ps_prefill_workspace_size(2, 300, 4, 2, 128, 0, 1, ctypes.byref(b1)) == 0
    assert b1.value - b0.value >= 2 * 300 * 4 * 128 * 2
    assert lib.ps_prefill_workspace_size(2, 300, 4, 2, 128, 0, 2, ctypes.byref(b0)) == 1
    fake = ctypes.c_void_p(1 << 20)
    i32 = ctypes.c_void_p(1 << 21)

    def call(pe_mode, ring=None):
        return lib.ps_prefill(fake, fake, fake, 1, 300, i32, i32, 64, 4, 2, 128,
                              ctypes.c_float(0.088), ctypes.c_double(1e4), pe_mode,
                              ctypes.byref(ring) if ring is not None else None, None, fake,
                              ctypes.c_void_p(1 << 22), None, 0, None, None)
    assert call(2) == 1                                  # unknown position encoding
    assert call(-1) == 1
    ring = _bad_desc(ps, n_kv_heads=2, window=64, capacity=80, prefix_max=16)
    assert call(1, ring) == 1                            # ring is Continue PE
    ring.pe_mode = 1
    assert call(0, ring) == 1                            # ring is Reset PE
    assert call(1, ring) == 4                            # consistent: fails later, on the workspace


def test_prefill_head_dims(ps):
    b = ctypes.c_size_t()
    assert ps.lib.ps_prefill_workspace_size(1, 300, 4, 2, 64, 0, 0, ctypes.byref(b)) == 0
    assert b.value >= 300 * 4 * 64 * 2 + 300 * 2 * 64 * 2
    assert ps.lib.ps_prefill_workspace_size(1, 300, 4, 2, 96, 0, 0, ctypes.byref(b)) == 2
    assert ps.lib.ps_prefill_workspace_size(1, 300, 4, 2, 256, 0, 0, ctypes.byref(b)) == 2


def test_decode_step_layout(ps):
    """Packed step blocks: each view 256-byte aligned, in the documented order, no
    overlap, block sizes rounded up to 256; invalid shapes refused."""
    L = ps.StepLayout()
    for nseq, hq, hkv, D in ((1, 1, 1, 64), (3, 16, 8, 128), (64, 16, 8, 128), (257, 8, 1, 64)):
        assert ps.lib.ps_decode_step_layout_get(nseq, hq, hkv, D, ctypes.byref(L)) == 0
        sizes = [("q_off", nseq * hq * D * 2), ("k_off", nseq * hkv * D * 2),
                 ("v_off", nseq * hkv * D * 2), ("pos_off", nseq * 4)]
        end = 0
        for name, nb in sizes:
            off = getattr(L, name)
            assert off % 256 == 0 and off == end
            end = off + (nb + 255) // 256 * 256
        assert L.in_bytes == end
        assert L.out_off == 0 and L.lse_off == (nseq * hq * D * 2 + 255) // 256 * 256
        assert L.res_bytes == L.lse_off + (nseq * hq * 4 + 255) // 256 * 256
        inp, n_in, res, n_res = ps.decode_step_layout(nseq, hq, hkv, D)
        assert n_in == L.in_bytes and n_res == L.res_bytes and inp["v"] == (L.v_off, nseq * hkv * D * 2)
    for args, code in (((0, 16, 8, 128), 1), ((4, 16, 6, 128), 1), ((4, 0, 8, 128), 1),
                       ((4, 16, 8, 96), 2)):
        assert ps.lib.ps_decode_step_layout_get(*args, ctypes.byref(L)) == code
    assert ps.lib.ps_decode_step_layout_get(4, 16, 8, 128, None) == 1


def test_decode_graph_host_validation(ps):
    """The executor refuses bad arguments before any CUDA call; a null handle is
    refused by step and ignored by destroy."""
    lib, f = ps.lib, ctypes.c_void_p(1 << 20)
    h = ctypes.c_void_p(123)
    desc = _bad_desc(ps, nseq=4, n_kv_heads=8, capacity=10)
    one = ctypes.c_float(0.1)
    assert lib.ps_decode_graph_create(ctypes.byref(desc), 16, one, f, f, f, 1 << 20, None) == 1
    assert lib.ps_decode_graph_create(None, 16, one, f, f, f, 1 << 20, ctypes.byref(h)) == 1
    assert h.value is None  # cleared on every refusal
    assert lib.ps_decode_graph_create(ctypes.byref(desc), 16, one, None, f, f, 1 << 20,
                                      ctypes.byref(h)) == 1
    assert lib.ps_decode_graph_create(ctypes.byref(desc), 16, one, ctypes.c_void_p((1 << 20) + 16),
                                      f, f, 1 << 20, ctypes.byref(h)) == 3
    assert lib.ps_decode_graph_create(ctypes.byref(desc), 12, one, f, f, f, 1 << 20,
                                      ctypes.byref(h)) == 1  # Hq % Hkv
    bad_d = _bad_desc(ps, nseq=4, n_kv_heads=8, head_dim=96)
    assert lib.ps_decode_graph_create(ctypes.byref(bad_d), 16, one, f, f, f, 1 << 20,
                                      ctypes.byref(h)) == 2
    assert h.value is None
    assert lib.ps_decode_graph_step(None, f, f, 1, None) == 1
    assert lib.ps_decode_graph_destroy(None) == 0


def test_boundary_usable_from_plain_c(ps, tmp_path):
    """A C99 program that includes ps.h and links libps.so (no Python, no torch)
    calls host-side entry points and gets the same answers as the binding."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(ps.lib._name)
    src = tmp_path / "boundary.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "ps.h"
int main(void) {
  ps_decode_step_layout L;
  if (ps_decode_step_layout_get(64, 16, 8, 128, &L) != PS_OK) return 1;
  if (ps_decode_step_layout_get(0, 16, 8, 128, &L) != PS_ERR_INVALID_ARGUMENT) return 2;
  if (ps_decode_graph_destroy(NULL) != PS_OK) return 3;
  if (strcmp(ps_status_string(PS_ERR_ALIGNMENT), "PS_ERR_ALIGNMENT") != 0) return 4;
  printf("%zu %zu %zu\n", L.v_off, L.in_bytes, L.res_bytes);
  return 0;
}
''')
    exe = tmp_path / "boundary"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lps",
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    inp, n_in, _, n_res = ps.decode_step_layout(64, 16, 8, 128)
    assert r.stdout.split() == [str(inp["v"][0]), str(n_in), str(n_res)]
