"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every function has the C name and argument order.  Pointer arguments accept a
torch tensor (its data pointer is passed), an int address, or None (NULL);
``stream`` accepts a torch.cuda.Stream, an int handle or None (the current
torch stream).  The structs mirror moe.h.  Nothing here computes any step of
the layer: all of it runs in the library's CUDA kernels, and importing this
package fails loudly when the library is missing.
"""
import ctypes
import os

from ctypes import c_double, c_int, c_int32, c_uint32, c_uint64, c_ulonglong, c_size_t, c_void_p, c_char_p, POINTER

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = range(5)
MOE_DEV_ERR_BAD_ID, MOE_DEV_ERR_UNBOUND, MOE_DEV_ERR_BAD_SLOT, MOE_DEV_ERR_TIMEOUT = 1, 2, 4, 8
MOE_FILL_LOWEST_ID, MOE_FILL_RANDOM = 0, 1
MOE_FFN_AUTO, MOE_FFN_GEMV, MOE_FFN_GEMM = 0, 1, 2
MOE_STAGING_TAG = 1 << 30
MOE_SLOT_MASK = (1 << 30) - 1


class moe_pool(ctypes.Structure):
    _fields_ = [("w_gate", c_void_p), ("w_up", c_void_p), ("w_down", c_void_p), ("n_slots", c_int32),
                ("host", c_int32)]


class moe_cache(ctypes.Structure):
    _fields_ = [("cache", moe_pool), ("staging", moe_pool), ("slot_table", c_void_p), ("owner", c_void_p),
                ("stamp", c_void_p), ("clock", c_void_p), ("n_layers", c_int32), ("E", c_int32),
                ("H", c_int32), ("I", c_int32)]


class moe_bind_stats(ctypes.Structure):
    _fields_ = [("n_unique", c_int32), ("n_hit", c_int32), ("n_miss", c_int32), ("q", c_int32),
                ("n_fill", c_int32), ("n_overflow", c_int32), ("n_staged", c_int32), ("clock", c_uint32)]


class moe_layer(ctypes.Structure):
    _fields_ = [("w_router", c_void_p), ("bias", c_void_p), ("layer", c_int32), ("E", c_int32),
                ("k", c_int32), ("H", c_int32), ("I", c_int32)]


class moe_layer_buffers(ctypes.Structure):
    _fields_ = [("topk_ids", c_void_p), ("topk_w", c_void_p), ("counts", c_void_p), ("offsets", c_void_p),
                ("perm", c_void_p), ("inv_perm", c_void_p), ("y_rows", c_void_p)]


class moe_pool_mxfp4(ctypes.Structure):
    _fields_ = [("gate_q", c_void_p), ("gate_s", c_void_p), ("up_q", c_void_p), ("up_s", c_void_p),
                ("down_q", c_void_p), ("down_s", c_void_p), ("n_slots", c_int32), ("reserved", c_int32)]


class moe_pool_nvfp4(ctypes.Structure):
    _fields_ = [("gate_q", c_void_p), ("gate_s", c_void_p), ("up_q", c_void_p), ("up_s", c_void_p),
                ("down_q", c_void_p), ("down_s", c_void_p), ("tensor_scale", c_void_p), ("n_slots", c_int32),
                ("reserved", c_int32)]


MOE_FP4_MXFP4, MOE_FP4_NVFP4 = 0, 1


class moe_cache_fp4(ctypes.Structure):
    _fields_ = [("cache", moe_pool_nvfp4), ("staging", moe_pool_nvfp4), ("slot_table", c_void_p),
                ("owner", c_void_p), ("stamp", c_void_p), ("clock", c_void_p), ("n_layers", c_int32),
                ("E", c_int32), ("H", c_int32), ("I", c_int32), ("format", c_int32), ("reserved", c_int32)]


class moe_bw_profile(ctypes.Structure):
    _fields_ = [("b_p_gbs", c_double), ("b_h_gbs", c_double), ("b_p_contended_gbs", c_double),
                ("b_h_contended_gbs", c_double), ("phi", c_double), ("phi_contended", c_double),
                ("phi_q16", c_uint32), ("phi_contended_q16", c_uint32), ("hybrid_ok", c_int32),
                ("read_checksum", c_uint32)]


BIND_STATS_FIELDS = [f for f, _ in moe_bind_stats._fields_]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: {moe_status_string(status)} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built at {LIB_PATH}; run "
                          "`python edge_moe_serving_gb300/csrc/build.py` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sig = {
        "moe_version": (c_int, []),
        "moe_status_string": (c_char_p, [c_int]),
        "moe_check_bounded_wait": (c_int, [P, P]),
        "moe_kernel_launch_count": (c_ulonglong, []),
        "moe_phi_to_q16": (c_uint32, [c_double]),
        "moe_bw_derive": (c_int, [POINTER(moe_bw_profile)]),
        "moe_bench_bandwidth": (c_int, [P, P, c_size_t, c_int, POINTER(moe_bw_profile), P, P]),
        "moe_route_topk_workspace_size": (c_size_t, [c_int, c_int, c_int]),
        "moe_route_topk": (c_int, [P, c_int, c_int, P, P, c_int, c_int, P, P, P, P, c_size_t, P, P]),
        "moe_dispatch_workspace_size": (c_size_t, [c_int, c_int, c_int]),
        "moe_dispatch": (c_int, [P, c_int, c_int, c_int, P, P, P, P, P, c_int, P, P, c_size_t, P, P]),
        "moe_cache_bind_workspace_size": (c_size_t, [POINTER(moe_cache), c_int, c_int]),
        "moe_cache_bind_slots": (c_int, [POINTER(moe_cache), c_int, P, c_int, c_int, c_uint32, c_int, c_int,
                                         c_uint64, P, P, P, c_size_t, P, P]),
        "moe_expert_ffn_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
        "moe_expert_ffn_grouped": (c_int, [POINTER(moe_cache), c_int, P, P, P, P, P, c_int, c_int, P, c_int,
                                           P, P, c_size_t, P, P]),
        "moe_expert_ffn_grouped_noalloc": (c_int, [POINTER(moe_cache), c_int, P, P, P, P, P, c_int, c_int, P,
                                                   c_int, P, P, P]),
        "moe_expert_ffn_mxfp4_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
        "moe_expert_ffn_mxfp4": (c_int, [POINTER(moe_pool_mxfp4), POINTER(moe_pool_mxfp4), P, c_int, c_int,
                                         c_int, c_int, c_int, P, P, P, P, c_int, c_int, P, P, c_size_t, P, P]),
        "moe_expert_ffn_nvfp4_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
        "moe_expert_ffn_nvfp4": (c_int, [POINTER(moe_pool_nvfp4), POINTER(moe_pool_nvfp4), P, c_int, c_int,
                                         c_int, c_int, c_int, P, P, P, P, c_int, c_int, P, P, c_size_t, P, P]),
        "moe_layer_fp4_workspace_size": (c_size_t, [POINTER(moe_layer), POINTER(moe_cache_fp4), c_int]),
        "moe_layer_forward_fp4": (c_int, [POINTER(moe_layer), POINTER(moe_cache_fp4), P, c_int, P, c_uint32, c_int,
                                          c_int, c_uint64, P, c_size_t, P, P, P]),
        "moe_combine": (c_int, [P, P, c_int, c_int, c_int, P, P, P, P]),
        "moe_prefill_double_buffered": (c_int, [POINTER(moe_layer), c_int, POINTER(moe_pool), POINTER(moe_pool),
                                                POINTER(moe_cache), POINTER(c_void_p), c_int, POINTER(c_void_p),
                                                c_int, c_int, P, c_size_t, P, P, P]),
        "moe_layer_workspace_size": (c_size_t, [POINTER(moe_layer), POINTER(moe_cache), c_int, c_int]),
        "moe_layer_forward": (c_int, [POINTER(moe_layer), POINTER(moe_cache), P, c_int, P, c_uint32, c_int,
                                      c_int, c_uint64, c_int, POINTER(moe_layer_buffers), P, c_size_t, P, P,
                                      P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = ["moe_version", "moe_status_string", "moe_check_bounded_wait", "moe_kernel_launch_count",
            "moe_phi_to_q16", "moe_bw_derive", "moe_bench_bandwidth", "moe_route_topk_workspace_size",
            "moe_route_topk",
            "moe_dispatch_workspace_size", "moe_dispatch", "moe_cache_bind_workspace_size",
            "moe_cache_bind_slots", "moe_expert_ffn_workspace_size", "moe_expert_ffn_grouped",
            "moe_expert_ffn_grouped_noalloc", "moe_expert_ffn_mxfp4_workspace_size", "moe_expert_ffn_mxfp4",
            "moe_expert_ffn_nvfp4_workspace_size", "moe_expert_ffn_nvfp4", "moe_layer_fp4_workspace_size",
            "moe_layer_forward_fp4", "moe_combine",
            "moe_layer_workspace_size", "moe_layer_forward", "moe_prefill_double_buffered"]


def lib():
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != MOE_OK:
        raise MoeError(fn, status)
    return status


def moe_version():
    return _lib.moe_version()


def moe_status_string(status):
    return _lib.moe_status_string(status).decode()


def moe_check_bounded_wait(dev_status, stream=None):
    return _check("moe_check_bounded_wait", _lib.moe_check_bounded_wait(_p(dev_status), _s(stream)))


def moe_kernel_launch_count():
    return int(_lib.moe_kernel_launch_count())


def moe_phi_to_q16(phi):
    return int(_lib.moe_phi_to_q16(float(phi)))


def moe_bw_derive(b_p_gbs, b_h_gbs, b_p_contended_gbs=0.0, b_h_contended_gbs=0.0):
    """moe_bw_derive on a profile holding the four rates; returns the profile."""
    prof = moe_bw_profile(b_p_gbs, b_h_gbs, b_p_contended_gbs, b_h_contended_gbs)
    _check("moe_bw_derive", _lib.moe_bw_derive(ctypes.byref(prof)))
    return prof


def moe_bench_bandwidth(host_src, dev_dst, nbytes, iters, copy_stream, read_stream):
    """host_src: pinned host tensor (or address); returns the measured profile."""
    prof = moe_bw_profile()
    _check("moe_bench_bandwidth", _lib.moe_bench_bandwidth(
        _p(host_src), _p(dev_dst), nbytes, iters, ctypes.byref(prof), _s(copy_stream), _s(read_stream)))
    return prof


def moe_route_topk_workspace_size(T, H, E):
    return _lib.moe_route_topk_workspace_size(T, H, E)


def moe_route_topk(x, T, H, w_router, bias, E, k, topk_ids, topk_w, logits_opt, ws, ws_bytes, dev_status,
                   stream=None):
    return _check("moe_route_topk", _lib.moe_route_topk(
        _p(x), T, H, _p(w_router), _p(bias), E, k, _p(topk_ids), _p(topk_w), _p(logits_opt), _p(ws), ws_bytes,
        _p(dev_status), _s(stream)))


def moe_dispatch_workspace_size(T, k, E):
    return _lib.moe_dispatch_workspace_size(T, k, E)


def moe_dispatch(topk_ids, T, k, E, counts, offsets, perm, inv_perm, x_opt, H, x_perm_opt, ws, ws_bytes,
                 dev_status, stream=None):
    return _check("moe_dispatch", _lib.moe_dispatch(
        _p(topk_ids), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv_perm), _p(x_opt), H, _p(x_perm_opt),
        _p(ws), ws_bytes, _p(dev_status), _s(stream)))


def moe_cache_bind_workspace_size(cache, T, k):
    return _lib.moe_cache_bind_workspace_size(ctypes.byref(cache), T, k)


def moe_cache_bind_slots(cache, layer, topk_ids, T, k, phi_q16, min_fill, fill_policy, seed, stats_dev,
                         fills_opt, ws, ws_bytes, dev_status, stream=None):
    return _check("moe_cache_bind_slots", _lib.moe_cache_bind_slots(
        ctypes.byref(cache), layer, _p(topk_ids), T, k, phi_q16, min_fill, fill_policy, seed, _p(stats_dev),
        _p(fills_opt), _p(ws), ws_bytes, _p(dev_status), _s(stream)))


def moe_expert_ffn_workspace_size(T, k, E, H, I, ffn_mode):
    return _lib.moe_expert_ffn_workspace_size(T, k, E, H, I, ffn_mode)


def moe_expert_ffn_grouped(cache, layer, counts, offsets, perm, x, x_perm_opt, T, k, expert_mask_opt,
                           ffn_mode, y_rows, ws, ws_bytes, dev_status, stream=None):
    return _check("moe_expert_ffn_grouped", _lib.moe_expert_ffn_grouped(
        ctypes.byref(cache), layer, _p(counts), _p(offsets), _p(perm), _p(x), _p(x_perm_opt), T, k,
        _p(expert_mask_opt), ffn_mode, _p(y_rows), _p(ws), ws_bytes, _p(dev_status), _s(stream)))


MOE_NOALLOC_FFN_SCRATCH_BYTES = 4 << 20


def moe_expert_ffn_grouped_noalloc(cache, layer, counts, offsets, perm, x, x_perm_opt, T, k, expert_mask_opt,
                                   ffn_mode, y_rows, dev_status, stream=None):
    """moe_expert_ffn_grouped for callers that cannot allocate device memory:
    the scratch is a static array inside the library (see include/moe.h)."""
    return _check("moe_expert_ffn_grouped_noalloc", _lib.moe_expert_ffn_grouped_noalloc(
        ctypes.byref(cache), layer, _p(counts), _p(offsets), _p(perm), _p(x), _p(x_perm_opt), T, k,
        _p(expert_mask_opt), ffn_mode, _p(y_rows), _p(dev_status), _s(stream)))


def moe_expert_ffn_mxfp4_workspace_size(T, k, H, I):
    return _lib.moe_expert_ffn_mxfp4_workspace_size(T, k, H, I)


def moe_expert_ffn_mxfp4(cache_pool, staging_opt, slot_table, n_layers, layer, E, H, I, counts, offsets, perm, x,
                         T, k, y_rows, ws, ws_bytes, dev_status, stream=None):
    """cache_pool / staging_opt: moe_pool_mxfp4 structs (staging_opt may be None)."""
    return _check("moe_expert_ffn_mxfp4", _lib.moe_expert_ffn_mxfp4(
        ctypes.byref(cache_pool), ctypes.byref(staging_opt) if staging_opt is not None else None,
        _p(slot_table), n_layers, layer, E, H, I, _p(counts), _p(offsets), _p(perm), _p(x), T, k, _p(y_rows),
        _p(ws), ws_bytes, _p(dev_status), _s(stream)))


def moe_expert_ffn_nvfp4_workspace_size(T, k, H, I):
    return _lib.moe_expert_ffn_nvfp4_workspace_size(T, k, H, I)


def moe_expert_ffn_nvfp4(cache_pool, staging_opt, slot_table, n_layers, layer, E, H, I, counts, offsets, perm, x,
                         T, k, y_rows, ws, ws_bytes, dev_status, stream=None):
    """cache_pool / staging_opt: moe_pool_nvfp4 structs (staging_opt may be None)."""
    return _check("moe_expert_ffn_nvfp4", _lib.moe_expert_ffn_nvfp4(
        ctypes.byref(cache_pool), ctypes.byref(staging_opt) if staging_opt is not None else None,
        _p(slot_table), n_layers, layer, E, H, I, _p(counts), _p(offsets), _p(perm), _p(x), T, k, _p(y_rows),
        _p(ws), ws_bytes, _p(dev_status), _s(stream)))


def moe_layer_fp4_workspace_size(layer, cache, T):
    return _lib.moe_layer_fp4_workspace_size(ctypes.byref(layer), ctypes.byref(cache), T)


def moe_layer_forward_fp4(layer, cache, x, T, out, phi_q16, min_fill, fill_policy, seed, ws, ws_bytes, dev_status,
                          stats_dev, stream=None):
    """cache: a moe_cache_fp4 struct (format MOE_FP4_MXFP4 or MOE_FP4_NVFP4)."""
    return _check("moe_layer_forward_fp4", _lib.moe_layer_forward_fp4(
        ctypes.byref(layer), ctypes.byref(cache), _p(x), T, _p(out), phi_q16, min_fill, fill_policy, seed, _p(ws),
        ws_bytes, _p(dev_status), _p(stats_dev), _s(stream)))


def moe_combine(y_rows, topk_w, T, k, H, out, out_f32_opt, dev_status, stream=None):
    return _check("moe_combine", _lib.moe_combine(
        _p(y_rows), _p(topk_w), T, k, H, _p(out), _p(out_f32_opt), _p(dev_status), _s(stream)))


def moe_layer_workspace_size(layer, cache, T, ffn_mode):
    return _lib.moe_layer_workspace_size(ctypes.byref(layer), ctypes.byref(cache), T, ffn_mode)


def moe_layer_forward(layer, cache, x, T, out, phi_q16, min_fill, fill_policy, seed, ffn_mode, bufs_opt, ws,
                      ws_bytes, dev_status, stats_dev, stream=None):
    return _check("moe_layer_forward", _lib.moe_layer_forward(
        ctypes.byref(layer), ctypes.byref(cache), _p(x), T, _p(out), phi_q16, min_fill, fill_policy, seed,
        ffn_mode, ctypes.byref(bufs_opt) if bufs_opt is not None else None, _p(ws), ws_bytes, _p(dev_status),
        _p(stats_dev), _s(stream)))


def moe_prefill_double_buffered(layers, source, layer_buf, state, x, T, out, ffn_mode, overlap, ws, ws_bytes,
                                dev_status, stream, copy_stream):
    """layers: list of moe_layer structs; source: moe_pool; layer_buf: two
    moe_pool structs (the second may be an empty moe_pool()); state: moe_cache
    (its residency arrays); x, out: lists of per-layer tensors or addresses."""
    n = len(layers)
    larr = (moe_layer * n)(*layers)
    barr = (moe_pool * 2)(*layer_buf)
    xs = (c_void_p * n)(*[_p(t) for t in x])
    outs = (c_void_p * n)(*[_p(t) for t in out])
    return _check("moe_prefill_double_buffered", _lib.moe_prefill_double_buffered(
        larr, n, ctypes.byref(source), barr, ctypes.byref(state), xs, T, outs, ffn_mode, overlap, _p(ws), ws_bytes,
        _p(dev_status), _s(stream), _s(copy_stream)))
