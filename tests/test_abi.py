"""The C-ABI library loads and exports every entry point include/moe.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import edge_moe_serving_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported():
    names = _declared()
    assert len(names) >= 13
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_struct_layouts_match_header():
    assert ctypes.sizeof(moe.moe_pool) == 32
    assert ctypes.sizeof(moe.moe_bind_stats) == 32
    assert ctypes.sizeof(moe.moe_layer) == 40
    assert ctypes.sizeof(moe.moe_layer_buffers) == 56
    assert ctypes.sizeof(moe.moe_cache) == 2 * 32 + 4 * 8 + 16
    assert ctypes.sizeof(moe.moe_bw_profile) == 6 * 8 + 4 * 4
    assert ctypes.sizeof(moe.moe_pool_mxfp4) == 6 * 8 + 2 * 4
    assert ctypes.sizeof(moe.moe_pool_nvfp4) == 7 * 8 + 2 * 4
    assert ctypes.sizeof(moe.moe_cache_fp4) == 2 * 64 + 4 * 8 + 6 * 4


def test_status_strings_and_version():
    assert moe.moe_version() >= 100
    assert moe.moe_status_string(moe.MOE_OK) == "ok"
    assert "workspace" in moe.moe_status_string(moe.MOE_ERR_WORKSPACE)


def test_workspace_sizes_are_host_arithmetic():
    assert moe.moe_route_topk_workspace_size(1, 4096, 256) >= 1024
    assert moe.moe_route_topk_workspace_size(8192, 40, 256) == 0
    # tensor-core router: the 3-way bf16 split of the router weights + fp32 logits
    assert moe.moe_route_topk_workspace_size(8192, 4096, 256) >= 256 * 3 * 4096 * 2 + 8192 * 256 * 4
    assert moe.moe_dispatch_workspace_size(1, 6, 256) == 0
    assert moe.moe_dispatch_workspace_size(8192, 6, 256) >= 48 * 256 * 4
    assert moe.moe_expert_ffn_workspace_size(32, 8, 128, 2048, 768, moe.MOE_FFN_GEMV) >= 256 * 768 * 2


def test_invalid_arguments_rejected_before_launch():
    L = moe.lib()
    # k > E, negative T, null outputs: rejected on the host
    assert L.moe_route_topk(None, 4, 64, None, None, 4, 5, None, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_topk(None, -1, 64, None, None, 8, 2, None, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_topk(None, 0, 64, None, None, 8, 2, None, None, None, None, 0, None, None) == moe.MOE_OK
    assert L.moe_dispatch(None, 4, 2, 8, None, None, None, None, None, 0, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(None, None, 4, 2, 64, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(None, None, 4, 17, 64, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    c = moe.moe_cache()
    assert L.moe_cache_bind_slots(ctypes.byref(c), 0, None, 1, 1, 0, 1, 0, 0, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    # unsupported shape: H not a multiple of 8 (fake non-null pointers: never dereferenced)
    c.cache = moe.moe_pool(16, 16, 16, 4)
    c.slot_table, c.owner, c.stamp, c.clock = 16, 16, 16, 16
    c.n_layers, c.E, c.H, c.I = 1, 4, 12, 8
    assert L.moe_cache_bind_slots(ctypes.byref(c), 0, None, 0, 1, 0, 1, 0, 0, None, None, None, 0, None, None) == moe.MOE_ERR_UNSUPPORTED
    c.H = 16
    # phi > 0 with no staging pool cannot fill
    assert L.moe_cache_bind_slots(ctypes.byref(c), 0, None, 0, 1, 100, 1, 0, 0, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_cache_bind_slots(ctypes.byref(c), 0, None, 0, 1, 0, 1, 0, 0, None, None, None, 0, None, None) == moe.MOE_ERR_WORKSPACE
    # bad policy / phi above 1.0 / layer out of range
    assert L.moe_cache_bind_slots(ctypes.byref(c), 0, None, 0, 1, 0, 1, 7, 0, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_cache_bind_slots(ctypes.byref(c), 0, None, 0, 1, 70000, 1, 0, 0, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_cache_bind_slots(ctypes.byref(c), 1, None, 0, 1, 0, 1, 0, 0, None, None, None, 0, None, None) == moe.MOE_ERR_INVALID_ARG


def test_layer_calls_reject_bad_k_and_oversized_calls():
    L = moe.lib()
    c = moe.moe_cache()
    c.cache = moe.moe_pool(16, 16, 16, 4)
    c.slot_table, c.owner, c.stamp, c.clock = 16, 16, 16, 16
    c.n_layers, c.E, c.H, c.I = 1, 8, 16, 16
    lay = moe.moe_layer(16, None, 0, 8, 2, 16, 16)
    assert L.moe_layer_workspace_size(ctypes.byref(lay), ctypes.byref(c), 4, moe.MOE_FFN_AUTO) > 0
    # k outside [1, min(E, 16)]: no workspace size, rejected before any launch
    for k in (0, -3, 9):
        lay.k = k
        assert L.moe_layer_workspace_size(ctypes.byref(lay), ctypes.byref(c), 4, moe.MOE_FFN_AUTO) == 0
        assert L.moe_layer_forward(ctypes.byref(lay), ctypes.byref(c), None, 4, None, 0, 1, 0, 0, moe.MOE_FFN_AUTO,
                                   None, None, 0, None, None, None) == moe.MOE_ERR_INVALID_ARG
    c.E, lay.E, lay.k = 32, 32, 17
    assert L.moe_layer_forward(ctypes.byref(lay), ctypes.byref(c), None, 4, None, 0, 1, 0, 0, moe.MOE_FFN_AUTO,
                               None, None, 0, None, None, None) == moe.MOE_ERR_INVALID_ARG
    # T * k beyond INT_MAX / 2 routed rows
    lay.k = 2
    assert L.moe_layer_workspace_size(ctypes.byref(lay), ctypes.byref(c), 1 << 30, moe.MOE_FFN_AUTO) == 0
    assert L.moe_layer_forward(ctypes.byref(lay), ctypes.byref(c), None, 1 << 30, None, 0, 1, 0, 0,
                               moe.MOE_FFN_AUTO, None, None, 0, None, None, None) == moe.MOE_ERR_UNSUPPORTED
    # the layer's shape must be the cache's
    lay.H = 24
    assert L.moe_layer_forward(ctypes.byref(lay), ctypes.byref(c), None, 4, None, 0, 1, 0, 0, moe.MOE_FFN_AUTO,
                               None, None, 0, None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_mxfp4_ffn_argument_checks():
    L = moe.lib()
    call = L.moe_expert_ffn_mxfp4
    pool = moe.moe_pool_mxfp4(16, 1, 16, 1, 16, 1, 4, 0)     # fake non-null pointers: never dereferenced
    args = lambda pool, T=4, k=2, E=8, H=64, I=64, ws_bytes=1 << 20, x=16, layer=0: (
        ctypes.byref(pool), None, 16, 1, layer, E, H, I, 16, 16, 16, x, T, k, 16, 16, ws_bytes, None, None)
    assert moe.moe_expert_ffn_mxfp4_workspace_size(4, 2, 64, 64) >= 2 * 4 * 2 * 64 * 2   # the bf16 h and token rows
    assert moe.moe_expert_ffn_mxfp4_workspace_size(4, 2, 64, 16) == 0
    assert call(*args(pool, T=0)) == moe.MOE_OK
    assert call(*args(pool, k=9)) == moe.MOE_ERR_INVALID_ARG          # k > E
    assert call(*args(pool, layer=1)) == moe.MOE_ERR_INVALID_ARG      # layer out of range
    assert call(*args(pool, H=48)) == moe.MOE_ERR_UNSUPPORTED         # not a multiple of 32
    assert call(*args(pool, I=80)) == moe.MOE_ERR_UNSUPPORTED
    assert call(*args(pool, E=2000)) == moe.MOE_ERR_UNSUPPORTED
    assert call(*args(pool, x=24)) == moe.MOE_ERR_UNSUPPORTED         # x not 16-byte aligned
    assert call(*args(pool, ws_bytes=64)) == moe.MOE_ERR_WORKSPACE
    assert call(*args(pool)) == moe.MOE_ERR_UNSUPPORTED               # ws (16) not 256-byte aligned
    bad = moe.moe_pool_mxfp4(24, 1, 16, 1, 16, 1, 4, 0)              # misaligned code bank
    assert call(*args(bad)) == moe.MOE_ERR_UNSUPPORTED
    empty = moe.moe_pool_mxfp4(16, None, 16, 1, 16, 1, 4, 0)         # missing scale bank
    assert call(*args(empty)) == moe.MOE_ERR_INVALID_ARG
    assert call(None, None, 16, 1, 0, 8, 64, 64, 16, 16, 16, 16, 4, 2, 16, 16, 1 << 20, None,
                None) == moe.MOE_ERR_INVALID_ARG


def test_nvfp4_ffn_argument_checks():
    L = moe.lib()
    call = L.moe_expert_ffn_nvfp4
    pool = moe.moe_pool_nvfp4(16, 16, 16, 16, 16, 16, 16, 4, 0)    # fake non-null pointers: never dereferenced
    args = lambda pool, T=4, k=2, E=8, H=64, I=64, ws_bytes=1 << 20, x=16, ws=256: (
        ctypes.byref(pool), None, 16, 1, 0, E, H, I, 16, 16, 16, x, T, k, 16, ws, ws_bytes, None, None)
    assert moe.moe_expert_ffn_nvfp4_workspace_size(4, 2, 64, 64) >= 2 * 4 * 2 * 64 * 2
    assert call(*args(pool, T=0)) == moe.MOE_OK
    assert call(*args(pool, k=9)) == moe.MOE_ERR_INVALID_ARG
    assert call(*args(pool, H=40)) == moe.MOE_ERR_UNSUPPORTED          # not a multiple of 16
    assert call(*args(pool, ws_bytes=64)) == moe.MOE_ERR_WORKSPACE
    assert call(*args(pool, ws=272)) == moe.MOE_ERR_UNSUPPORTED        # ws not 256-byte aligned
    assert call(*args(pool)) == moe.MOE_ERR_UNSUPPORTED                # rows of 64 inputs: not a decode-kernel shape
    no_ts = moe.moe_pool_nvfp4(16, 16, 16, 16, 16, 16, None, 4, 0)
    assert call(*args(no_ts)) == moe.MOE_ERR_INVALID_ARG
    odd_ts = moe.moe_pool_nvfp4(16, 16, 16, 16, 16, 16, 18, 4, 0)
    assert call(*args(odd_ts)) == moe.MOE_ERR_UNSUPPORTED


def test_ffn_argument_checks_and_the_allocation_free_variant():
    """The bf16 expert FFN's host checks, and the allocation-free variant's:
    the same argument checks in the same order, then its scratch limit."""
    L = moe.lib()
    c = moe.moe_cache()
    c.cache = moe.moe_pool(256, 256, 256, 4)                          # fake non-null pointers: never dereferenced
    c.slot_table, c.owner, c.stamp, c.clock = 256, 256, 256, 256
    c.n_layers, c.E, c.H, c.I = 1, 8, 64, 64
    ffn = lambda c, T=4, k=2, mode=moe.MOE_FFN_AUTO, ws=256, ws_bytes=1 << 30, x=256, y=256, layer=0: \
        L.moe_expert_ffn_grouped(ctypes.byref(c), layer, 256, 256, 256, x, None, T, k, None, mode, y, ws, ws_bytes,
                                 None, None)
    na = lambda c, T=4, k=2, mode=moe.MOE_FFN_AUTO, x=256, y=256, layer=0, counts=256: \
        L.moe_expert_ffn_grouped_noalloc(ctypes.byref(c), layer, counts, 256, 256, x, None, T, k, None, mode, y, None,
                                         None)
    for call in (ffn, na):
        assert call(c, T=0) == moe.MOE_OK
        assert call(c, k=9) == moe.MOE_ERR_INVALID_ARG                 # k > E
        assert call(c, layer=1) == moe.MOE_ERR_INVALID_ARG             # layer out of range
        assert call(c, mode=7) == moe.MOE_ERR_INVALID_ARG              # unknown kernel choice
        assert call(c, x=None) == moe.MOE_ERR_INVALID_ARG
        assert call(c, y=264) == moe.MOE_ERR_UNSUPPORTED               # y rows not 16-byte aligned
        assert call(c, mode=moe.MOE_FFN_GEMM) == moe.MOE_ERR_INVALID_ARG   # the GEMM needs the gathered rows
    assert ffn(c, ws_bytes=64) == moe.MOE_ERR_WORKSPACE
    assert ffn(c, ws=272) == moe.MOE_ERR_UNSUPPORTED                  # ws not 256-byte aligned
    # beyond the built-in scratch: the workspace error comes after the argument checks
    big = 1 << 16
    assert moe.moe_expert_ffn_workspace_size(big, 2, 8, 64, 64, moe.MOE_FFN_AUTO) > moe.MOE_NOALLOC_FFN_SCRATCH_BYTES
    assert na(c, T=big) == moe.MOE_ERR_WORKSPACE
    assert na(c, T=big, counts=None) == moe.MOE_ERR_INVALID_ARG
    assert na(c, T=big, k=9) == moe.MOE_ERR_INVALID_ARG
    nopool = moe.moe_cache()
    nopool.n_layers, nopool.E, nopool.H, nopool.I = 1, 8, 64, 64
    assert na(nopool, T=big) == moe.MOE_ERR_INVALID_ARG


def test_fp4_layer_argument_checks():
    """Every check of the FP4 layer call comes before its first launch (the
    bind would update the residency state): fake non-null pointers, never
    dereferenced."""
    L = moe.lib()

    def cache(fmt=moe.MOE_FP4_MXFP4, H=1024, I=1024, ts=256, staging=False, scale=256):
        c = moe.moe_cache_fp4()
        c.cache = moe.moe_pool_nvfp4(256, scale, 256, 256, 256, 256, ts, 4, 0)
        if staging:
            c.staging = moe.moe_pool_nvfp4(256, 256, 256, 256, 256, 256, ts, 7, 0)
        c.slot_table, c.owner, c.stamp, c.clock = 256, 256, 256, 256
        c.n_layers, c.E, c.H, c.I, c.format = 1, 8, H, I, fmt
        return c

    def call(c, T=1, k=2, H=None, I=None, phi=0, policy=0, ws=256, ws_bytes=1 << 30, x=256, router=256):
        lay = moe.moe_layer(router, None, 0, c.E, k, H or c.H, I or c.I)
        return L.moe_layer_forward_fp4(ctypes.byref(lay), ctypes.byref(c), x, T, 256, phi, 1, policy, 0, ws, ws_bytes,
                                       None, None, None)

    mx, nv = cache(), cache(moe.MOE_FP4_NVFP4)
    lay = moe.moe_layer(256, None, 0, 8, 2, 1024, 1024)
    assert moe.moe_layer_fp4_workspace_size(lay, mx, 4) >= 4 * 2 * 1024 * 4     # the fp32 expert rows
    assert call(mx, T=0) == moe.MOE_OK
    assert call(cache(fmt=2)) == moe.MOE_ERR_INVALID_ARG                         # unknown format
    assert call(mx, H=2048) == moe.MOE_ERR_INVALID_ARG                           # layer and cache disagree
    assert call(mx, k=9) == moe.MOE_ERR_INVALID_ARG                              # k > E
    assert call(mx, policy=5) == moe.MOE_ERR_INVALID_ARG
    assert call(mx, phi=16384) == moe.MOE_ERR_INVALID_ARG                        # fills need a staging pool
    assert call(cache(staging=True), phi=16384) == moe.MOE_ERR_INVALID_ARG       # staging smaller than n_layers*E
    assert call(cache(H=1040, I=1040)) == moe.MOE_ERR_UNSUPPORTED                # not a multiple of 32
    assert call(cache(scale=264)) == moe.MOE_ERR_UNSUPPORTED                     # scale bank not 16-byte aligned
    assert call(mx, ws_bytes=64) == moe.MOE_ERR_WORKSPACE
    assert call(mx, ws=272) == moe.MOE_ERR_UNSUPPORTED                           # ws not 256-byte aligned
    assert call(mx, x=264) == moe.MOE_ERR_UNSUPPORTED                            # x not 16-byte aligned
    assert call(mx, router=None) == moe.MOE_ERR_INVALID_ARG                      # no router
    assert call(mx, router=264) == moe.MOE_ERR_UNSUPPORTED                       # router not 16-byte aligned
    wide = cache()
    wide.E = 600                                                                 # beyond the router's 512 experts
    assert call(wide) == moe.MOE_ERR_UNSUPPORTED
    assert call(cache(moe.MOE_FP4_NVFP4, ts=None)) == moe.MOE_ERR_INVALID_ARG    # NVFP4 without tensor scales
    assert call(cache(moe.MOE_FP4_NVFP4, ts=258)) == moe.MOE_ERR_UNSUPPORTED     # tensor scales not 4-byte aligned
    # NVFP4 shapes that fit neither the ring kernel (<= 64 routed rows of 1024, 2048 or 4096 inputs) nor the
    # tensor-core GEMM (I a multiple of 128, H of 256)
    assert call(cache(moe.MOE_FP4_NVFP4, H=1040, I=1040), T=33) == moe.MOE_ERR_UNSUPPORTED
    assert call(cache(moe.MOE_FP4_NVFP4, H=1040, I=1040)) == moe.MOE_ERR_UNSUPPORTED


STRUCTS = ["moe_pool", "moe_cache", "moe_bind_stats", "moe_layer", "moe_layer_buffers", "moe_bw_profile",
           "moe_pool_mxfp4", "moe_pool_nvfp4", "moe_cache_fp4"]


def test_header_is_plain_c_and_matches_the_binding_layouts(tmp_path):
    """include/moe.h compiles as C99 with warnings as errors; every struct's
    size and every field's offset, as the C compiler lays them out, equal the
    ctypes binding's."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "moe.h"', "int main(void) {"]
    for name in STRUCTS:
        lines.append(f'  printf("{name} %zu\\n", sizeof({name}));')
        for field, _ in getattr(moe, name)._fields_:
            lines.append(f'  printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                               text=True).stdout.splitlines())
    for name in STRUCTS:
        ct = getattr(moe, name)
        assert int(out[name]) == ctypes.sizeof(ct), name
        for field, _ in ct._fields_:
            assert int(out[f"{name}.{field}"]) == getattr(ct, field).offset, (name, field)


def test_library_is_usable_from_plain_c(tmp_path):
    """A C99 program linked against libmoe.so (no Python) calls the host-side
    entry points: version, status strings, phi in Q16, the bandwidth
    derivation, workspace sizes and argument rejection before any launch."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "moe.h"
#define CHECK(c) do { if (!(c)) { printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #c); return 1; } } while (0)
int main(void) {
  moe_bw_profile p;
  moe_pool_mxfp4 mx;
  moe_layer lay;
  moe_cache c;
  CHECK(moe_version() >= 100);
  CHECK(strcmp(moe_status_string(MOE_OK), "ok") == 0);
  CHECK(moe_phi_to_q16(0.5) == 32768u && moe_phi_to_q16(2.0) == 65536u && moe_phi_to_q16(-1.0) == 0u);
  memset(&p, 0, sizeof p);
  p.b_p_gbs = 25.1; p.b_h_gbs = 63.2;
  CHECK(moe_bw_derive(&p) == MOE_OK && p.phi_q16 == moe_phi_to_q16(25.1 / 63.2) && p.hybrid_ok == 1);
  CHECK(moe_bw_derive(NULL) == MOE_ERR_INVALID_ARG);
  CHECK(moe_dispatch_workspace_size(1, 6, 256) == 0);
  CHECK(moe_expert_ffn_mxfp4_workspace_size(1, 6, 4096, 2048) >= 6u * (4096u + 2048u) * 2u);
  CHECK(moe_route_topk(NULL, 4, 64, NULL, NULL, 4, 5, NULL, NULL, NULL, NULL, 0, NULL, NULL) == MOE_ERR_INVALID_ARG);
  CHECK(moe_combine(NULL, NULL, 0, 2, 64, NULL, NULL, NULL, NULL) == MOE_OK);
  memset(&mx, 0, sizeof mx);
  CHECK(moe_expert_ffn_mxfp4(&mx, NULL, NULL, 1, 0, 8, 64, 64, NULL, NULL, NULL, NULL, 1, 2, NULL, NULL, 0, NULL,
                             NULL) == MOE_ERR_INVALID_ARG);
  memset(&lay, 0, sizeof lay);
  memset(&c, 0, sizeof c);
  CHECK(moe_layer_forward(&lay, &c, NULL, 1, NULL, 0, 1, 0, 0, MOE_FFN_AUTO, NULL, NULL, 0, NULL, NULL, NULL) ==
        MOE_ERR_INVALID_ARG);
  printf("ok\n");
  return 0;
}
''')
    exe = tmp_path / "use"
    libdir = os.path.dirname(moe.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe), "-L", libdir, "-lmoe", f"-Wl,-rpath,{libdir}"], check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
