"""ctypes binding of the C ABI in include/oscar.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors are passed as
raw pointers (torch owns device memory and streams); a non-zero status raises
OscarError with the library's own message.  There is no fallback: if liboscar.so is
missing the import of this module's functions fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboscar.so")

OSCAR_FORMAT_INT2 = 0
OSCAR_FORMAT_BF16 = 1
OSCAR_FORMAT_INT2_CM = 2  # INT2, channel-major value pages (tcgen05 decode)
OSCAR_FLAG_BAD_PAGE = 0x1
OSCAR_FLAG_TIMEOUT = 0x2
OSCAR_FLAG_BAD_SLOT = 0x4
OSCAR_FAULT_LOST_APPEND_SIGNAL = 0x1

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "OUT_OF_PAGES", 4: "BAD_PAGE", 5: "CUDA",
                6: "TIMEOUT", 7: "STATE"}


class OscarError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"oscar status {status} ({STATUS_NAMES.get(status, '?')}): {message}")
        self.status = status


class oscar_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("format", "head_dim", "n_q_heads", "n_kv_heads", "group", "page", "n_sink",
                                            "window", "n_layers", "max_requests", "max_pages",
                                            "max_pages_per_request")]


class oscar_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("codes", "sz", "sink", "ring", "bf16_pages", "codes_page_bytes",
                                               "sz_page_bytes", "bf16_page_bytes", "sink_bytes_per_head",
                                               "ring_bytes_per_head", "page_table", "total")]


EXPORTS = [
    "oscar_cache_device_bytes", "oscar_cache_create", "oscar_cache_destroy", "oscar_cache_layout",
    "oscar_set_layer_params", "oscar_cache_stats", "oscar_request_alloc", "oscar_request_free", "oscar_request_info",
    "oscar_request_pages", "oscar_request_share_prefix", "oscar_reserve", "oscar_quantize_append",
    "oscar_commit_append", "oscar_plan_decode", "oscar_plan_decode_ex", "oscar_decode_workspace_bytes",
    "oscar_decode_workspace_max_bytes", "oscar_plan_info",
    "oscar_decode_attention", "oscar_append_decode_attention", "oscar_decode_attention_noalloc", "oscar_bf16_append",
    "oscar_bf16_decode_attention", "oscar_calibration_workspace_bytes", "oscar_calibrate_layer",
    "oscar_set_wait_limit", "oscar_inject_fault", "oscar_get_status",
    "oscar_last_error", "oscar_last_launch_count",
]

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(the CUDA library is required; there is no fallback)")
            L = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            IP = ctypes.POINTER(ctypes.c_int)
            CP = ctypes.POINTER(oscar_config)
            sig = {
                "oscar_cache_device_bytes": (S, [CP]),
                "oscar_cache_create": (I, [CP, P, S, ctypes.POINTER(P)]),
                "oscar_cache_destroy": (None, [P]),
                "oscar_cache_layout": (I, [P, ctypes.POINTER(oscar_layout)]),
                "oscar_set_layer_params": (I, [P, I, P, P, P, P, P]),
                "oscar_cache_stats": (I, [P, IP, IP]),
                "oscar_request_alloc": (I, [P, IP]),
                "oscar_request_free": (I, [P, I]),
                "oscar_request_info": (I, [P, I, IP, IP, IP]),
                "oscar_request_pages": (I, [P, I, IP, I]),
                "oscar_request_share_prefix": (I, [P, I, I, I, P]),
                "oscar_reserve": (I, [P, IP, IP, I, P]),
                "oscar_quantize_append": (I, [P, I, P, P, P]),
                "oscar_commit_append": (I, [P]),
                "oscar_plan_decode": (I, [P, IP, I, I, P]),
                "oscar_plan_decode_ex": (I, [P, IP, I, I, ctypes.c_uint32, P]),
                "oscar_decode_workspace_bytes": (S, [P]),
                "oscar_decode_workspace_max_bytes": (S, [P]),
                "oscar_plan_info": (I, [P, IP, IP, IP]),
                "oscar_decode_attention": (I, [P, I, P, P, P, S, P, P]),
                "oscar_append_decode_attention": (I, [P, I, P, P, P, P, P, S, P, P]),
                "oscar_decode_attention_noalloc": (I, [P, I, P, P, P, P]),
                "oscar_bf16_append": (I, [P, I, P, P, P]),
                "oscar_bf16_decode_attention": (I, [P, I, P, P, P, S, P, P]),
                "oscar_calibration_workspace_bytes": (S, [I, I, I]),
                "oscar_calibrate_layer": (I, [P, P, P, I, I, I, ctypes.c_longlong, I, P, P, P, P, P, P, S, P]),
                "oscar_set_wait_limit": (I, [P, ctypes.c_uint32]),
                "oscar_inject_fault": (I, [P, ctypes.c_uint32]),
                "oscar_get_status": (I, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
                "oscar_last_error": (ctypes.c_char_p, []),
                "oscar_last_launch_count": (I, []),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def _check(status: int) -> None:
    if status != 0:
        raise OscarError(status, lib().oscar_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    """Raw address of a tensor (device or host), None for None."""
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ints(values):
    values = [int(v) for v in values]
    return (ctypes.c_int * max(1, len(values)))(*values), len(values)


# ------------------------------------------------------------------ entry points
def oscar_cache_device_bytes(cfg: oscar_config) -> int:
    n = lib().oscar_cache_device_bytes(ctypes.byref(cfg))
    if n == 0:
        raise OscarError(1, lib().oscar_last_error().decode())
    return n


def oscar_cache_create(cfg: oscar_config, device_mem, nbytes: int) -> int:
    h = ctypes.c_void_p()
    _check(lib().oscar_cache_create(ctypes.byref(cfg), _ptr(device_mem), nbytes, ctypes.byref(h)))
    return h.value


def oscar_cache_destroy(handle: int) -> None:
    lib().oscar_cache_destroy(handle)


def oscar_cache_layout(handle: int) -> oscar_layout:
    out = oscar_layout()
    _check(lib().oscar_cache_layout(handle, ctypes.byref(out)))
    return out


def oscar_set_layer_params(handle: int, layer: int, R_K, R_V, clip_K, clip_V, stream=None) -> None:
    """R_K, R_V: host fp32 contiguous [H_kv, d, d]; clip_K, clip_V: host fp32 [H_kv]."""
    for t in (R_K, R_V, clip_K, clip_V):
        assert t.device.type == "cpu" and t.is_contiguous()
    _check(lib().oscar_set_layer_params(handle, layer, _ptr(R_K), _ptr(R_V), _ptr(clip_K), _ptr(clip_V),
                                        _stream(stream)))


def oscar_cache_stats(handle: int):
    """(free pages, free request slots)."""
    p, r = ctypes.c_int(), ctypes.c_int()
    _check(lib().oscar_cache_stats(handle, ctypes.byref(p), ctypes.byref(r)))
    return p.value, r.value


def oscar_request_alloc(handle: int) -> int:
    s = ctypes.c_int()
    _check(lib().oscar_request_alloc(handle, ctypes.byref(s)))
    return s.value


def oscar_request_free(handle: int, slot: int) -> None:
    _check(lib().oscar_request_free(handle, slot))


def oscar_request_info(handle: int, slot: int):
    L, H, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().oscar_request_info(handle, slot, ctypes.byref(L), ctypes.byref(H), ctypes.byref(n)))
    return L.value, H.value, n.value


def oscar_request_pages(handle: int, slot: int, n: int):
    buf = (ctypes.c_int * max(1, n))()
    _check(lib().oscar_request_pages(handle, slot, buf, n))
    return list(buf)[:n]


def oscar_request_share_prefix(handle: int, dst: int, src: int, n_tokens: int, stream=None) -> None:
    _check(lib().oscar_request_share_prefix(handle, dst, src, n_tokens, _stream(stream)))


def oscar_reserve(handle: int, slots, n_new, stream=None) -> None:
    s, n = _ints(slots)
    m, n2 = _ints(n_new)
    assert n == n2
    _check(lib().oscar_reserve(handle, s, m, n, _stream(stream)))


def oscar_quantize_append(handle: int, layer: int, k_new, v_new, stream=None) -> None:
    _check(lib().oscar_quantize_append(handle, layer, _ptr(k_new), _ptr(v_new), _stream(stream)))


def oscar_bf16_append(handle: int, layer: int, k_new, v_new, stream=None) -> None:
    _check(lib().oscar_bf16_append(handle, layer, _ptr(k_new), _ptr(v_new), _stream(stream)))


def oscar_commit_append(handle: int) -> None:
    _check(lib().oscar_commit_append(handle))


def oscar_plan_decode(handle: int, slots, max_split_pages: int = 0, stream=None) -> None:
    s, n = _ints(slots)
    _check(lib().oscar_plan_decode(handle, s, n, max_split_pages, _stream(stream)))


OSCAR_PLAN_NARROW = 0x1
OSCAR_PLAN_FOLDED_ROTATIONS = 0x2  # q arrives rotated (R_K folded into W_q), the output stays rotated


def oscar_plan_decode_ex(handle: int, slots, max_split_pages: int = 0, flags: int = 0, stream=None) -> None:
    s, n = _ints(slots)
    _check(lib().oscar_plan_decode_ex(handle, s, n, max_split_pages, flags, _stream(stream)))


def oscar_decode_workspace_bytes(handle: int) -> int:
    return int(lib().oscar_decode_workspace_bytes(handle))


def oscar_decode_workspace_max_bytes(handle: int) -> int:
    return int(lib().oscar_decode_workspace_max_bytes(handle))


def oscar_plan_info(handle: int):
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().oscar_plan_info(handle, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def oscar_decode_attention(handle: int, layer: int, q, out, workspace, out_f32=None, stream=None) -> None:
    _check(lib().oscar_decode_attention(handle, layer, _ptr(q), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _ptr(out_f32),
                                        _stream(stream)))


def oscar_append_decode_attention(handle: int, layer: int, k_new, v_new, q, out, workspace, out_f32=None,
                                  stream=None) -> None:
    _check(lib().oscar_append_decode_attention(handle, layer, _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out),
                                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                                               _ptr(out_f32), _stream(stream)))


def oscar_decode_attention_noalloc(handle: int, layer: int, q, out, out_f32=None, stream=None) -> None:
    """Decode with the library's fixed device scratch (no caller workspace, no allocation)."""
    _check(lib().oscar_decode_attention_noalloc(handle, layer, _ptr(q), _ptr(out), _ptr(out_f32), _stream(stream)))


def oscar_bf16_decode_attention(handle: int, layer: int, q, out, workspace, out_f32=None, stream=None) -> None:
    _check(lib().oscar_bf16_decode_attention(handle, layer, _ptr(q), _ptr(out), _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _ptr(out_f32),
                                             _stream(stream)))


def oscar_get_status(handle: int, stream=None):
    """(status, flags): status 0 or the error the flags map to; flags are cleared."""
    f = ctypes.c_uint32()
    st = lib().oscar_get_status(handle, _stream(stream), ctypes.byref(f))
    return st, f.value


def oscar_last_launch_count() -> int:
    return int(lib().oscar_last_launch_count())


def oscar_set_wait_limit(handle: int, counter_polls: int) -> None:
    _check(lib().oscar_set_wait_limit(handle, int(counter_polls)))


def oscar_inject_fault(handle: int, faults: int) -> None:
    _check(lib().oscar_inject_fault(handle, int(faults)))


OSCAR_ROTATION_OSCAR = 0
OSCAR_ROTATION_HADAMARD = 1


def oscar_calibration_workspace_bytes(n_tokens: int, n_q_heads: int, n_kv_heads: int) -> int:
    return int(lib().oscar_calibration_workspace_bytes(n_tokens, n_q_heads, n_kv_heads))


def oscar_calibrate_layer(q, k, v, clip_rank: int, rotation: int, R_K, R_V, clip_K, clip_V, workspace,
                          covariances=None, stream=None) -> None:
    """q [N, H_q, d], k and v [N, H_kv, d] bf16 device tensors -> R_K, R_V [H_kv, d, d], clip_K,
    clip_V [H_kv] fp32 device tensors (and optionally the fp64 covariances [2 H_kv, d, d])."""
    n, hq, _ = q.shape
    hkv = k.shape[1]
    _check(lib().oscar_calibrate_layer(_ptr(q), _ptr(k), _ptr(v), n, hq, hkv, int(clip_rank), int(rotation),
                                       _ptr(R_K), _ptr(R_V), _ptr(clip_K), _ptr(clip_V), _ptr(covariances),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))
