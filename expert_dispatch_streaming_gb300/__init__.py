"""Python binding of libmoe (the C ABI in include/moe.h), by ctypes.

Argument marshalling only: every step of the MoE layer runs in the library's CUDA kernels.
Device buffers are passed as integers (``tensor.data_ptr()``) or as torch tensors, streams
as ``torch.cuda.Stream`` / raw handles.  The library is loaded eagerly from this directory;
importing this package without a built ``libmoe.so`` raises ``ImportError`` (there is no
fallback implementation).
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_CUDA = -2
MOE_ERR_CAPACITY = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_CORRUPT = -5
MOE_ERR_UNSUPPORTED = -6
MOE_ERR_NO_MEMORY = -7

MOE_GATING_SOFTMAX_RENORM = 0
MOE_GATING_SOFTMAX = 1
MOE_GATING_SIGMOID_BIAS_RENORM = 2
GATING = {"softmax_renorm": 0, "softmax": 1, "sigmoid_bias_renorm": 2}

MOE_W_BF16 = 0
MOE_W_INT4_G128 = 1
MOE_W_NVFP4 = 2
WDTYPE = {"bf16": 0, "int4_g128": 1, "nvfp4": 2}


class MoEError(RuntimeError):
    def __init__(self, status, fn):
        self.status = status
        cuda = _lib.moe_last_cuda_error() if status == MOE_ERR_CUDA else 0
        super().__init__(f"{fn}: {_lib.moe_status_string(status).decode()}"
                         + (f" (cudaError {cuda})" if cuda else ""))


# ----------------------------------------------------------------------------- structs
class moe_bundle_layout(C.Structure):
    _fields_ = [("total_bytes", C.c_size_t), ("gate_up_offset", C.c_size_t),
                ("down_offset", C.c_size_t), ("gate_up_scale_offset", C.c_size_t),
                ("down_scale_offset", C.c_size_t), ("global_scale_offset", C.c_size_t)]


class moe_host_bundle(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("bytes", C.c_size_t), ("checksum", C.c_uint64)]


class moe_expert_cache_config(C.Structure):
    _fields_ = [("slot_bytes", C.c_size_t), ("capacity_bytes", C.c_size_t),
                ("n_layers", C.c_int), ("n_experts", C.c_int),
                ("bundles", C.POINTER(moe_host_bundle)), ("timeout_ms", C.c_int),
                ("verify_checksums", C.c_int), ("device", C.c_int), ("time_copies", C.c_int),
                ("prefetch_next_layer", C.c_int), ("device_lru", C.c_int),
                ("copy_kernel", C.c_int)]


class moe_cache_event(C.Structure):
    _fields_ = [("request", C.c_int64), ("layer", C.c_int32), ("expert", C.c_int32),
                ("miss", C.c_int32), ("victim_layer", C.c_int32),
                ("victim_expert", C.c_int32), ("slot", C.c_int32), ("prefetch", C.c_int32)]


class moe_cache_stats(C.Structure):
    _fields_ = [("requests", C.c_int64), ("hits", C.c_int64), ("misses", C.c_int64),
                ("evictions", C.c_int64), ("bytes_h2d", C.c_int64), ("n_slots", C.c_int32),
                ("resident", C.c_int32), ("prefetch_requests", C.c_int64),
                ("prefetch_fills", C.c_int64), ("prefetch_used", C.c_int64)]


class moe_layer(C.Structure):
    _fields_ = [("H", C.c_int), ("E", C.c_int), ("k", C.c_int), ("I", C.c_int), ("Is", C.c_int),
                ("gating", C.c_int), ("scale", C.c_float), ("wdtype", C.c_int),
                ("layer_index", C.c_int), ("shared_gate_sigmoid", C.c_int),
                ("w_r", C.c_void_p), ("logit_bias", C.c_void_p), ("sel_bias", C.c_void_p),
                ("w_gate", C.c_void_p), ("shared_bundle", C.c_void_p),
                ("bundles", C.POINTER(C.c_void_p)), ("norm_eps", C.c_float)]


MOE_N_PHASE_EVENTS = 6


class moe_layer_stats(C.Structure):
    _fields_ = [("n_unique", C.c_int32), ("n_missed", C.c_int32), ("n_launches", C.c_int32),
                ("shared_merged", C.c_int32), ("fused_decode", C.c_int32),
                ("phase_events", C.POINTER(C.c_void_p))]


# ----------------------------------------------------------------------------- loading
from . import build as _build  # noqa: E402

if not _build.up_to_date():
    # compile in-tree on first import (nvcc is part of the toolchain on every machine used)
    try:
        _build.build()
    except Exception as exc:  # no fallback path exists: fail loudly
        raise ImportError(f"libmoe.so could not be built ({LIB_PATH}): {exc}") from exc
_lib = C.CDLL(LIB_PATH)

_vp, _i, _f, _sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t
_SIGS = {
    "moe_last_cuda_error": (_i, []),
    "moe_status_string": (C.c_char_p, [_i]),
    "moe_version": (_i, []),
    "moe_set_option": (_i, [_i, _i]),
    "moe_workspace_error": (_i, [_vp, C.POINTER(C.c_int32), _vp]),
    "moe_bundle_layout_of": (_i, [_i, _i, _i, C.POINTER(moe_bundle_layout)]),
    "moe_bundle_bytes": (_sz, [_i, _i, _i]),
    "moe_pack_bundle": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_pack_bundle_nvfp4": (_i, [_i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_checksum64": (C.c_uint64, [_vp, _sz]),
    "moe_route_workspace_size": (_sz, [_i, _i, _i, _i]),
    "moe_route_topk": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f,
                            _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_topk_static": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_route_static_error": (_i, [C.POINTER(C.c_int32), _vp]),
    "moe_permute": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "moe_grouped_swiglu_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "moe_grouped_swiglu": (_i, [_vp, _vp, C.POINTER(_vp), _i, _i, _i, _i, _i, _vp, _vp, _sz,
                                _vp]),
    "moe_combine": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _f, _vp]),
    "moe_expert_cache_create": (_i, [C.POINTER(moe_expert_cache_config), C.POINTER(_vp),
                                     C.POINTER(C.c_int64)]),
    "moe_expert_cache_destroy": (_i, [_vp]),
    "moe_expert_cache_request": (_i, [_vp, _i, _vp, _vp, _i, C.POINTER(_vp),
                                      C.POINTER(C.c_int32)]),
    "moe_expert_cache_prefetch": (_i, [_vp, _i, _vp, C.POINTER(C.c_int32)]),
    "moe_expert_cache_wait_expert": (_i, [_vp, _i, _i, _vp]),
    "moe_expert_cache_release": (_i, [_vp, _i, _vp]),
    "moe_expert_cache_evict": (_i, [_vp, _i, _i]),
    "moe_expert_cache_trace": (_i, [_vp, C.POINTER(moe_cache_event), _sz, C.POINTER(_sz)]),
    "moe_expert_cache_reset_trace": (_i, [_vp]),
    "moe_expert_cache_stats": (_i, [_vp, C.POINTER(moe_cache_stats)]),
    "moe_expert_cache_sync": (_i, [_vp]),
    "moe_expert_cache_copy_time": (_i, [_vp, C.POINTER(C.c_double), C.POINTER(C.c_int64)]),
    "moe_layer_workspace_size": (_sz, [C.POINTER(moe_layer), _i]),
    "moe_layer_forward": (_i, [C.POINTER(moe_layer), _vp, _i, _vp, _vp, _vp, _vp, _vp,
                               C.POINTER(moe_layer_stats), _vp, _vp, _vp, _sz, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


# ----------------------------------------------------------------------------- marshalling
def ptr(x) -> int | None:
    """Device/host address of a tensor / array / int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(type(x))


def stream_handle(s) -> int | None:
    if s is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status, fn):
    if status != MOE_OK:
        raise MoEError(status, fn)
    return status


# ----------------------------------------------------------------------------- API
MOE_OPT_FFN_KERNEL = 1
MOE_OPT_PDL = 2
MOE_OPT_DECODE_KERNEL = 3
FFN_KERNEL = {"auto": 0, "stream": 1, "tcgen05": 2}


def moe_set_option(option, value) -> None:
    _check(_lib.moe_set_option(option, value), "moe_set_option")


def set_ffn_kernel(name: str) -> None:
    """'auto' | 'stream' (mma.sync weight streaming) | 'tcgen05' (tensor-core kernel)."""
    moe_set_option(MOE_OPT_FFN_KERNEL, FFN_KERNEL[name])


DECODE_KERNEL = {"off": 0, "auto": 1, "always": 2}


def set_decode_kernel(mode) -> None:
    """The fused decode kernel for small batches with resident bundles: 'auto' (default; INT4
    weights only up to 4 tokens), 'always', or 'off'.  True / False mean 'auto' / 'off'."""
    if isinstance(mode, bool):
        mode = "auto" if mode else "off"
    moe_set_option(MOE_OPT_DECODE_KERNEL, DECODE_KERNEL[mode])


def set_pdl(on: bool) -> None:
    """Programmatic dependent launch of the layer's kernels (default off)."""
    moe_set_option(MOE_OPT_PDL, 1 if on else 0)


def moe_workspace_error(ws, stream=None) -> int:
    code = C.c_int32(0)
    _check(_lib.moe_workspace_error(ptr(ws), C.byref(code), stream_handle(stream)),
           "moe_workspace_error")
    return code.value


def bundle_layout(H, I, wdtype) -> moe_bundle_layout:
    out = moe_bundle_layout()
    _check(_lib.moe_bundle_layout_of(H, I, WDTYPE.get(wdtype, wdtype), C.byref(out)),
           "moe_bundle_layout_of")
    return out


def moe_bundle_bytes(H, I, wdtype) -> int:
    return _lib.moe_bundle_bytes(H, I, WDTYPE.get(wdtype, wdtype))


def moe_pack_bundle(H, I, wdtype, wg, wu, wd, sg, su, sd, dst) -> None:
    _check(_lib.moe_pack_bundle(H, I, WDTYPE.get(wdtype, wdtype), ptr(wg), ptr(wu), ptr(wd),
                                ptr(sg), ptr(su), ptr(sd), ptr(dst)), "moe_pack_bundle")


def moe_pack_bundle_nvfp4(H, I, wg, wu, wd, sg, su, sd, gs, dst) -> None:
    """wg/wu [H][I], wd [I][H]: uint8 E2M1 codes; sg/su [H/16][I], sd [I/16][H]: uint8 E4M3
    block scales; gs: float32 [3] matrix scales (gate, up, down)."""
    _check(_lib.moe_pack_bundle_nvfp4(H, I, ptr(wg), ptr(wu), ptr(wd), ptr(sg), ptr(su),
                                      ptr(sd), ptr(gs), ptr(dst)), "moe_pack_bundle_nvfp4")


def moe_checksum64(data, nbytes) -> int:
    return _lib.moe_checksum64(ptr(data), nbytes)


def moe_route_workspace_size(T, H, E, k) -> int:
    return _lib.moe_route_workspace_size(T, H, E, k)


def moe_route_topk(x, w_r, logit_bias, sel_bias, w_gate, forced_ids, T, H, E, k, gating, scale,
                   ids, w, counts, offsets, pos, src, logits, shared_gate, tie_flags, ws,
                   ws_bytes, stream=None) -> None:
    _check(_lib.moe_route_topk(ptr(x), ptr(w_r), ptr(logit_bias), ptr(sel_bias), ptr(w_gate),
                               ptr(forced_ids), T, H, E, k, GATING.get(gating, gating),
                               float(scale), ptr(ids), ptr(w), ptr(counts), ptr(offsets),
                               ptr(pos), ptr(src), ptr(logits), ptr(shared_gate),
                               ptr(tie_flags), ptr(ws), ws_bytes, stream_handle(stream)),
           "moe_route_topk")


def moe_route_topk_static(x, w_r, logit_bias, sel_bias, w_gate, forced_ids, T, H, E, k, gating,
                          scale, ids, w, counts, offsets, pos, src, logits, shared_gate,
                          tie_flags, stream=None) -> None:
    """moe_route_topk without a workspace (scratch in a fixed array of the library)."""
    _check(_lib.moe_route_topk_static(ptr(x), ptr(w_r), ptr(logit_bias), ptr(sel_bias),
                                      ptr(w_gate), ptr(forced_ids), T, H, E, k,
                                      GATING.get(gating, gating), float(scale), ptr(ids), ptr(w),
                                      ptr(counts), ptr(offsets), ptr(pos), ptr(src), ptr(logits),
                                      ptr(shared_gate), ptr(tie_flags), stream_handle(stream)),
           "moe_route_topk_static")


def moe_route_static_error(stream=None) -> int:
    """Error word of moe_route_topk_static's fixed scratch on the current device (blocking)."""
    code = C.c_int32(0)
    _check(_lib.moe_route_static_error(C.byref(code), stream_handle(stream)),
           "moe_route_static_error")
    return code.value


def moe_permute(x, src, T, k, H, x_perm, stream=None) -> None:
    _check(_lib.moe_permute(ptr(x), ptr(src), T, k, H, ptr(x_perm), stream_handle(stream)),
           "moe_permute")


def moe_grouped_swiglu_workspace_size(max_rows, E, H, I, wdtype) -> int:
    return _lib.moe_grouped_swiglu_workspace_size(max_rows, E, H, I, WDTYPE.get(wdtype, wdtype))


def moe_grouped_swiglu(x_perm, offsets, bundles, E, H, I, wdtype, max_rows, y_perm, ws, ws_bytes,
                       stream=None) -> None:
    arr = (C.c_void_p * E)(*[ptr(b) for b in bundles])
    _check(_lib.moe_grouped_swiglu(ptr(x_perm), ptr(offsets), arr, E, H, I,
                                   WDTYPE.get(wdtype, wdtype), max_rows, ptr(y_perm), ptr(ws),
                                   ws_bytes, stream_handle(stream)), "moe_grouped_swiglu")


def moe_combine(y_perm, pos, w, T, k, H, shared, shared_gate, residual, out, stream=None,
                out_normed=None, norm_eps=1e-6) -> None:
    _check(_lib.moe_combine(ptr(y_perm), ptr(pos), ptr(w), T, k, H, ptr(shared),
                            ptr(shared_gate), ptr(residual), ptr(out), ptr(out_normed),
                            float(norm_eps), stream_handle(stream)),
           "moe_combine")


def moe_expert_cache_create(cfg: moe_expert_cache_config) -> int:
    h = C.c_void_p()
    bad = C.c_int64(-1)
    st = _lib.moe_expert_cache_create(C.byref(cfg), C.byref(h), C.byref(bad))
    if st != MOE_OK:
        err = MoEError(st, "moe_expert_cache_create")
        err.bad_index = bad.value
        raise err
    return h.value


def moe_expert_cache_destroy(cache) -> None:
    _check(_lib.moe_expert_cache_destroy(cache), "moe_expert_cache_destroy")


def moe_expert_cache_request(cache, layer, used_mask, compute=None, defer_waits=0, E=None):
    """used_mask: host uint8 array [E].  Returns (slot_ptrs list, n_missed)."""
    E = E or len(used_mask)
    slots = (C.c_void_p * E)()
    nm = C.c_int32(0)
    _check(_lib.moe_expert_cache_request(cache, layer, ptr(used_mask), stream_handle(compute),
                                         defer_waits, slots, C.byref(nm)),
           "moe_expert_cache_request")
    return [s for s in slots], nm.value


def moe_expert_cache_prefetch(cache, layer, mask=None) -> int:
    """Prefetch request for `layer` (mask: host uint8 array [E], or None for the layer's
    previous expert set); returns the number of copies issued."""
    n = C.c_int32(0)
    _check(_lib.moe_expert_cache_prefetch(cache, layer, ptr(mask), C.byref(n)),
           "moe_expert_cache_prefetch")
    return n.value


def moe_expert_cache_wait_expert(cache, layer, expert, compute=None) -> None:
    _check(_lib.moe_expert_cache_wait_expert(cache, layer, expert, stream_handle(compute)),
           "moe_expert_cache_wait_expert")


def moe_expert_cache_release(cache, layer, compute=None) -> None:
    _check(_lib.moe_expert_cache_release(cache, layer, stream_handle(compute)),
           "moe_expert_cache_release")


def moe_expert_cache_evict(cache, layer, expert) -> None:
    _check(_lib.moe_expert_cache_evict(cache, layer, expert), "moe_expert_cache_evict")


def moe_expert_cache_trace(cache) -> list[tuple]:
    n = C.c_size_t(0)
    _check(_lib.moe_expert_cache_trace(cache, None, 0, C.byref(n)), "moe_expert_cache_trace")
    buf = (moe_cache_event * max(1, n.value))()
    _check(_lib.moe_expert_cache_trace(cache, buf, n.value, C.byref(n)), "moe_expert_cache_trace")
    return [(e.request, e.layer, e.expert, e.miss, e.victim_layer, e.victim_expert, e.slot,
             e.prefetch) for e in buf[:n.value]]


def moe_expert_cache_reset_trace(cache) -> None:
    _check(_lib.moe_expert_cache_reset_trace(cache), "moe_expert_cache_reset_trace")


def moe_expert_cache_stats(cache) -> dict:
    s = moe_cache_stats()
    _check(_lib.moe_expert_cache_stats(cache, C.byref(s)), "moe_expert_cache_stats")
    return {f: getattr(s, f) for f, _ in s._fields_}


def moe_expert_cache_sync(cache) -> None:
    _check(_lib.moe_expert_cache_sync(cache), "moe_expert_cache_sync")


def moe_expert_cache_copy_time(cache) -> tuple[float, int]:
    ms, n = C.c_double(0), C.c_int64(0)
    _check(_lib.moe_expert_cache_copy_time(cache, C.byref(ms), C.byref(n)),
           "moe_expert_cache_copy_time")
    return ms.value, n.value


def moe_layer_workspace_size(layer: moe_layer, T) -> int:
    return _lib.moe_layer_workspace_size(C.byref(layer), T)


def moe_layer_forward(layer: moe_layer, x, T, forced_ids, residual, out, cache, ws, ws_bytes,
                      stream=None, ids_out=None, w_out=None, phase_events=None,
                      out_normed=None) -> moe_layer_stats:
    """phase_events: None or a list of MOE_N_PHASE_EVENTS torch.cuda.Event (recorded by the
    library on `stream` at phase boundaries).  out_normed: None or a device [T][H] buffer for
    the RMS-normalised output (the next layer's input of a pre-norm stack)."""
    st = moe_layer_stats()
    if phase_events is not None:
        arr = (C.c_void_p * MOE_N_PHASE_EVENTS)(*[ev.cuda_event if ev is not None else None
                                                  for ev in phase_events])
        st.phase_events = arr
    _check(_lib.moe_layer_forward(C.byref(layer), ptr(x), T, ptr(forced_ids), ptr(residual),
                                  ptr(out), ptr(out_normed), cache, C.byref(st), ptr(ids_out),
                                  ptr(w_out),
                                  ptr(ws), ws_bytes, stream_handle(stream)), "moe_layer_forward")
    return st
