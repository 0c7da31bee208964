"""Python binding of libmoe (routed mixture-of-experts FFN on one GB300).

A thin ctypes layer over the C ABI declared in ``include/moe.h``: every
function below has the C entry point's name and only marshals arguments
(torch tensors -> device pointers, streams -> ``cudaStream_t``).  All
arithmetic runs in the library's CUDA kernels; there is no CPU fallback, and
loading fails loudly if ``libmoe.so`` has not been built.
"""

from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe.so")

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_ESTATE, MOE_ETIMEOUT, MOE_EDOMAIN, MOE_EIO = range(8)
MOE_RESIDENT_HBM, MOE_HOST_POOL, MOE_FILE_POOL = 0, 1, 2
MOE_FILE_DIRECT = 1
MOE_STAGING_HOST, MOE_STAGING_DEVICE, MOE_STAGING_FUSED = 0, 1, 2
MOE_CACHE_LRU, MOE_CACHE_LFU = 0, 1
MOE_GELU_ERF, MOE_GELU_TANH = 0, 1
HOOK_FAIL_NEXT_COPY, HOOK_WAIT_LIMIT_US, HOOK_PDL, HOOK_PERSISTENT, HOOK_TIMELINE, HOOK_FREE_BYTES = 1, 2, 3, 4, 5, 6
HOOK_PREFILL_TC = 7
HOOK_CLUSTER = 9
HOOK_SPIN_LIMIT = 10      # bounded waits of the persistent decode kernels: cycles (<= 0: the default)
HOOK_AT_REST = 11         # MOE_OK when the persistent kernels' launch words are back at rest
HOOK_WAIT_DIAG = 12       # the clustered kernel's first wait that ran out (site << 16 | CTA) into a host uint32
HOOK_SMALL_BATCH = 13     # small-batch grouped GEMVs (calls of at most 32 tokens) on / off
HOOK_TOKEN_LOOP = 14      # decode steps of 2 to 4 tokens: one clustered-kernel launch per token on / off


class MoeConfig(C.Structure):
    _fields_ = [("d", C.c_int32), ("f", C.c_int32), ("f_shared", C.c_int32), ("n_experts", C.c_int32),
                ("top_k", C.c_int32), ("group", C.c_int32), ("n_layers", C.c_int32),
                ("gelu_variant", C.c_int32), ("prenorm", C.c_int32), ("max_tokens", C.c_int32),
                ("norm_eps", C.c_float)]


class MoeExpertWeights(C.Structure):
    _fields_ = [("gate_q", C.c_void_p), ("gate_sb", C.c_void_p), ("up_q", C.c_void_p),
                ("up_sb", C.c_void_p), ("down_q", C.c_void_p), ("down_sb", C.c_void_p)]


class MoeTraceRec(C.Structure):
    _fields_ = [("token", C.c_int32), ("layer", C.c_int32), ("k_pos", C.c_int32), ("expert", C.c_int32),
                ("hit", C.c_int32), ("slot", C.c_int32), ("evicted", C.c_int32)]


class MoeStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("steps", "hits", "misses", "staged_bytes", "n_slots",
                                          "expert_bytes", "shared_bytes", "device_bytes",
                                          "host_pool_bytes", "file_read_bytes", "host_tier_hits",
                                          "host_tier_bytes")]


class MoeKernelTime(C.Structure):
    _fields_ = [("launches", C.c_int64), ("total_ms", C.c_double)]


N_KERNEL_KINDS = 8
KERNEL_KINDS = {0: "router_topk_plan", 1: "gateup_gelu_gemv", 2: "down_combine_gemv", 3: "decode_persistent",
                4: "prefill_route_group", 5: "prefill_tcgen05_gemm", 6: "prefill_combine", 7: "small_batch_gemv"}


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


_lib = None

# name -> (restype, argtypes)
_SIGS = {
    "moe_create": (C.c_int, [C.POINTER(MoeConfig), C.c_int, C.POINTER(C.c_void_p)]),
    "moe_init_layer": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.POINTER(MoeExpertWeights),
                                 C.POINTER(MoeExpertWeights), C.c_int]),
    "moe_set_slots": (C.c_int, [C.c_void_p, C.c_int]),
    "moe_set_cache_policy": (C.c_int, [C.c_void_p, C.c_int]),
    "moe_set_expert_file": (C.c_int, [C.c_void_p, C.c_char_p, C.c_int, C.c_uint64, C.c_int]),
    "moe_set_file_cache": (C.c_int, [C.c_void_p, C.c_int]),
    "moe_set_staging": (C.c_int, [C.c_void_p, C.c_int]),
    "moe_pread_parallel": (C.c_int, [C.c_char_p, C.c_uint64, C.c_uint64, C.c_void_p, C.c_int, C.c_uint64]),
    "moe_host_read_rate": (C.c_int, [C.c_void_p, C.c_uint64, C.c_int, C.c_void_p, C.POINTER(C.c_double)]),
    "moe_decode_step": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.POINTER(MoeTraceRec), C.c_int, C.POINTER(C.c_int),
                                  C.c_void_p]),
    "moe_prefill": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                              C.c_void_p, C.c_void_p]),
    "moe_set_debug": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int]),
    "moe_set_debug_logits": (C.c_int, [C.c_void_p, C.c_void_p]),
    "moe_sync": (C.c_int, [C.c_void_p, C.c_void_p]),
    "moe_get_stats": (C.c_int, [C.c_void_p, C.POINTER(MoeStats)]),
    "moe_get_cache_state": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]),
    "moe_reset_cache": (C.c_int, [C.c_void_p]),
    "moe_expert_bytes": (C.c_int64, [C.POINTER(MoeConfig)]),
    "moe_shared_bytes": (C.c_int64, [C.POINTER(MoeConfig)]),
    "moe_test_hook": (C.c_int, [C.c_void_p, C.c_int, C.c_int64]),
    "moe_route_noalloc": (C.c_int, [C.POINTER(MoeConfig), C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_profile": (C.c_int, [C.c_void_p, C.c_int]),
    "moe_get_profile": (C.c_int, [C.c_void_p, C.POINTER(MoeKernelTime), C.c_int]),
    "moe_status_string": (C.c_char_p, [C.c_int]),
    "moe_last_error": (C.c_char_p, [C.c_void_p]),
    "moe_destroy": (None, [C.c_void_p]),
}


def lib():
    """Load libmoe.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmoe.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def status_name(status: int) -> str:
    try:
        return moe_status_string(status)
    except Exception:  # pragma: no cover
        return f"status {status}"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int, ctx=None) -> None:
    """Raise MoeError for a non-OK status, with the context's last message."""
    if status != MOE_OK:
        msg = moe_last_error(ctx) if ctx is not None else ""
        raise MoeError(status, msg)


# ---------------------------------------------------------------- C entry points

def make_config(d, f, f_shared, n_experts, top_k, n_layers=1, group=64, gelu_variant=MOE_GELU_ERF,
                prenorm=0, max_tokens=32, norm_eps=1e-6) -> MoeConfig:
    return MoeConfig(d, f, f_shared, n_experts, top_k, group, n_layers, gelu_variant, prenorm, max_tokens,
                     norm_eps)


def moe_create(cfg: MoeConfig, device: int = 0):
    """Returns (status, ctx handle or None)."""
    h = C.c_void_p()
    st = lib().moe_create(C.byref(cfg), device, C.byref(h))
    return st, (h.value if st == MOE_OK else None)


def expert_weights(d: dict, index=None) -> MoeExpertWeights:
    """Marshal one expert's canonical tensors (``index`` selects from stacked [E, ...] tensors)."""
    def p(name):
        t = d[name] if index is None else d[name][index]
        return _ptr(t)
    return MoeExpertWeights(p("gate_q"), p("gate_sb"), p("up_q"), p("up_sb"), p("down_q"), p("down_sb"))


def moe_init_layer(ctx, layer: int, router_w, experts: dict, shared: dict, residency=MOE_RESIDENT_HBM) -> int:
    """router_w fp16 [E, d]; experts: stacked canonical tensors [E, ...]; shared: canonical tensors."""
    E = router_w.shape[0]
    for t in list(experts.values()) + list(shared.values()) + [router_w]:
        assert t.is_contiguous(), "weights must be contiguous"
    arr = (MoeExpertWeights * E)(*[expert_weights(experts, e) for e in range(E)])
    sw = expert_weights(shared)
    return lib().moe_init_layer(ctx, layer, _ptr(router_w), arr, C.byref(sw), residency)


def moe_set_slots(ctx, n_slots: int) -> int:
    return lib().moe_set_slots(ctx, n_slots)


def moe_set_cache_policy(ctx, policy: int) -> int:
    return lib().moe_set_cache_policy(ctx, policy)


def moe_set_expert_file(ctx, path, n_threads: int = 8, chunk_bytes: int = 0, flags: int = 0) -> int:
    return lib().moe_set_expert_file(ctx, None if path is None else os.fsencode(path), n_threads, chunk_bytes,
                                     flags)


def moe_set_staging(ctx, mode: int) -> int:
    return lib().moe_set_staging(ctx, mode)


def moe_set_file_cache(ctx, n_host: int) -> int:
    return lib().moe_set_file_cache(ctx, n_host)


def moe_host_read_rate(host_buf, nbytes: int, reps: int = 5, stream=None):
    """(status, GB/s): plain-load read rate of pinned host memory from every SM."""
    out = C.c_double(0.0)
    st = lib().moe_host_read_rate(_ptr(host_buf), nbytes, reps, _stream(stream), C.byref(out))
    return st, out.value


def moe_pread_parallel(path, offset: int, nbytes: int, dst, n_threads: int = 8, chunk_bytes: int = 0) -> int:
    """Read [offset, offset + nbytes) of `path` into `dst` (a writable buffer:
    a numpy array or a pinned host tensor)."""
    return lib().moe_pread_parallel(None if path is None else os.fsencode(path), offset, nbytes, _ptr(dst),
                                    n_threads, chunk_bytes)


def moe_decode_step(ctx, h_in, B: int, layer_begin: int, layer_end: int, logit_bias=None, h_out=None,
                    y_last=None, trace=None, stream=None):
    """Returns (status, n_trace).  ``trace`` is a ctypes array of MoeTraceRec or None."""
    n = C.c_int(0)
    cap = len(trace) if trace is not None else 0
    st = lib().moe_decode_step(ctx, _ptr(h_in), B, layer_begin, layer_end, _ptr(logit_bias), _ptr(h_out),
                               _ptr(y_last), trace, cap, C.byref(n), _stream(stream))
    return st, n.value


def moe_prefill(ctx, h, T: int, layer_begin: int, layer_end: int, logit_bias=None, h_out=None, y_last=None,
                stream=None) -> int:
    return lib().moe_prefill(ctx, _ptr(h), T, layer_begin, layer_end, _ptr(logit_bias), _ptr(h_out),
                             _ptr(y_last), _stream(stream))


def moe_set_debug(ctx, x_layers=None, ids=None, gates=None, y_layers=None, max_layers: int = 0) -> int:
    return lib().moe_set_debug(ctx, _ptr(x_layers), _ptr(ids), _ptr(gates), _ptr(y_layers), max_layers)


def moe_set_debug_logits(ctx, logits=None) -> int:
    return lib().moe_set_debug_logits(ctx, _ptr(logits))


def moe_sync(ctx, stream=None) -> int:
    return lib().moe_sync(ctx, _stream(stream))


def moe_get_stats(ctx):
    s = MoeStats()
    st = lib().moe_get_stats(ctx, C.byref(s))
    return st, s


def moe_get_cache_state(ctx, layer: int, n_slots: int):
    import numpy as np
    eos = np.zeros(n_slots, dtype=np.int32)
    lu = np.zeros(n_slots, dtype=np.int64)
    st = lib().moe_get_cache_state(ctx, layer, eos.ctypes.data, lu.ctypes.data)
    return st, eos, lu


def moe_reset_cache(ctx) -> int:
    return lib().moe_reset_cache(ctx)


def moe_expert_bytes(cfg: MoeConfig) -> int:
    return lib().moe_expert_bytes(C.byref(cfg))


def moe_shared_bytes(cfg: MoeConfig) -> int:
    return lib().moe_shared_bytes(C.byref(cfg))


def moe_test_hook(ctx, hook: int, value: int) -> int:
    return lib().moe_test_hook(ctx, hook, value)


ROUTE_NOALLOC_MAX_B = 64


def moe_route_noalloc(cfg: MoeConfig, router_w, h, B: int, logit_bias, ids, gates, stream=None) -> int:
    """Routing without any device allocation (see include/moe.h); every buffer is the caller's."""
    return lib().moe_route_noalloc(C.byref(cfg), _ptr(router_w), _ptr(h), B, _ptr(logit_bias), _ptr(ids),
                                   _ptr(gates), _stream(stream))


def moe_profile(ctx, enable: bool) -> int:
    return lib().moe_profile(ctx, 1 if enable else 0)


def moe_get_profile(ctx):
    """Returns (status, list of (launches, total_ms) per kernel kind); resets the totals."""
    arr = (MoeKernelTime * N_KERNEL_KINDS)()
    st = lib().moe_get_profile(ctx, arr, N_KERNEL_KINDS)
    return st, [(a.launches, a.total_ms) for a in arr]


def moe_last_error(ctx) -> str:
    r = lib().moe_last_error(ctx)
    return r.decode() if r else ""


def moe_destroy(ctx) -> None:
    lib().moe_destroy(ctx)
