"""Python binding of the GB300 routed-expert SwiGLU MoE layer.

Thin ctypes marshalling over the C ABI in ``include/moe.h`` (same function
names): tensors are passed as device pointers, the stream is torch's current
stream.  Every step of the layer runs in the CUDA kernels of
``libmoe_gb300.so``; there is no fallback, and the functions raise if the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

from ._build import LIB, build  # noqa: F401

MOE_OK, MOE_ERR_ARG, MOE_ERR_ALIGN, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_BOUNDS, \
    MOE_ERR_NOMEM = range(8)
MOE_F32, MOE_BF16 = 0, 1
MOE_W_BF16, MOE_W_Q4G64 = 0, 1
MOE_PATH_AUTO, MOE_PATH_GEMV, MOE_PATH_GEMM = 0, 1, 2
MOE_ROUTER_AUTO, MOE_ROUTER_SIMT, MOE_ROUTER_TENSOR = 0, 1, 2
(MOE_K_ROUTER, MOE_K_SELECT, MOE_K_GROUP, MOE_K_GEMV_GATE_UP, MOE_K_GEMV_DOWN, MOE_K_GEMM_GATE_UP, MOE_K_GEMM_DOWN,
 MOE_K_COMBINE, MOE_K_DECODE_FUSED) = range(9)

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {moe_strerror(code)} (code {code})")
        self.code = code


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("d", "n_experts", "inter", "shared_inter", "top_k", "max_tokens",
                                            "x_dtype", "has_router_bias", "has_shared", "bias_select_only",
                                            "shared_gate", "weight_format")]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{os.path.basename(LIB)} is not built: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.moe_init.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(P)]
        L.moe_route.argtypes = [P, P, I, P, P, I, P, P, P, P, P, P]
        L.moe_forward.argtypes = [P, P, I, P, P, P, P, P, I, P, P]
        L.moe_set_path.argtypes = [P, I]
        L.moe_set_router.argtypes = [P, I]
        L.moe_set_spin_limit.argtypes = [P, ctypes.c_longlong]
        L.moe_record_event.argtypes = [P, P]
        L.moe_record_event.restype = I
        L.moe_set_chunk_tokens.argtypes = [P, I]
        L.moe_set_chunk_tokens.restype = I
        L.moe_set_overlap.argtypes = [P, I]
        L.moe_set_overlap.restype = I
        L.moe_set_prefetch.argtypes = [P, P, P]
        L.moe_set_prefetch.restype = I
        L.moe_inject_stall.argtypes = [P, I]
        L.moe_inject_stall.restype = I
        L.moe_time_kernel.argtypes = [P, I, P, P]
        L.moe_time_kernel.restype = I
        L.moe_launch_count.argtypes = [P]
        L.moe_launch_count.restype = ctypes.c_longlong
        L.moe_decode_noalloc.argtypes = [P, I, I, I, I, I, I, P, P, P, P, P, P, P, P]
        L.moe_decode_noalloc.restype = I
        L.moe_last_routing.argtypes = [P, P, P, P, P, P, P, ctypes.POINTER(I), ctypes.POINTER(I), P]
        L.moe_last_routing.restype = I
        L.moe_status.argtypes = [P]
        L.moe_strerror.argtypes = [I]
        L.moe_strerror.restype = ctypes.c_char_p
        L.moe_destroy.argtypes = [P]
        L.moe_destroy.restype = None
        for f in ("moe_init", "moe_route", "moe_forward", "moe_set_path", "moe_set_router", "moe_set_spin_limit",
                  "moe_status"):
            getattr(L, f).restype = I
        del F
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/moe.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def _check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def moe_strerror(code: int) -> str:
    return lib().moe_strerror(code).decode()


def moe_init(d, n_experts, inter, shared_inter, top_k, max_tokens, x_dtype=MOE_BF16, has_router_bias=False,
             has_shared=True, bias_select_only=False, shared_gate=False,
             weight_format=MOE_W_BF16) -> ctypes.c_void_p:
    cfg = moe_config(d, n_experts, inter, shared_inter, top_k, max_tokens, x_dtype, int(has_router_bias),
                     int(has_shared), int(bias_select_only), int(shared_gate), int(weight_format))
    h = ctypes.c_void_p()
    _check(lib().moe_init(ctypes.byref(cfg), ctypes.byref(h)), "moe_init")
    return h


def moe_destroy(ctx) -> None:
    lib().moe_destroy(ctx)


def moe_set_path(ctx, path: int) -> None:
    _check(lib().moe_set_path(ctx, path), "moe_set_path")


def moe_set_router(ctx, router: int) -> None:
    _check(lib().moe_set_router(ctx, router), "moe_set_router")


def moe_set_spin_limit(ctx, limit_ns: int) -> None:
    _check(lib().moe_set_spin_limit(ctx, limit_ns), "moe_set_spin_limit")


def moe_record_event(event, stream=None) -> None:
    """Record a torch.cuda.Event on a stream; timeable also under graph capture."""
    _check(lib().moe_record_event(ctypes.c_void_p(event.cuda_event), _stream(stream)), "moe_record_event")


def moe_set_chunk_tokens(ctx, chunk: int) -> None:
    """Chunked prefill (see moe.h): with chunk > 0 moe_forward accepts any T and runs
    slices of at most `chunk` tokens through the context's bounded workspace."""
    _check(lib().moe_set_chunk_tokens(ctx, int(chunk)), "moe_set_chunk_tokens")


def moe_set_overlap(ctx, on: bool) -> None:
    """Launch the fused small-T kernel with programmatic stream serialization
    (see moe.h); the caller promises the preceding work does not write the weights."""
    _check(lib().moe_set_overlap(ctx, 1 if on else 0), "moe_set_overlap")


def moe_set_prefetch(ctx, next_router_w=None, next_shared_w=None) -> None:
    """Hint: the next small-T forward pulls these next-layer weights into L2."""
    _check(lib().moe_set_prefetch(ctx, _ptr(next_router_w), _ptr(next_shared_w)), "moe_set_prefetch")


def moe_inject_stall(ctx, on: bool) -> None:
    _check(lib().moe_inject_stall(ctx, int(on)), "moe_inject_stall")


def moe_time_kernel(ctx, kernel_id: int, ev_start, ev_stop) -> None:
    """Arm the next call to record torch.cuda.Event pair around kernel `kernel_id`."""
    _check(lib().moe_time_kernel(ctx, kernel_id, ctypes.c_void_p(ev_start.cuda_event),
                                 ctypes.c_void_p(ev_stop.cuda_event)), "moe_time_kernel")


def moe_launch_count(ctx) -> int:
    return lib().moe_launch_count(ctx)


def moe_status(ctx) -> int:
    return lib().moe_status(ctx)


def moe_route(ctx, x, router_w, router_b, top_k, idx=None, w=None, counts=None, offsets=None, perm=None,
              stream=None) -> None:
    import torch

    for name, t, dt in (("x", x, None), ("router_w", router_w, torch.float32), ("router_b", router_b, torch.float32),
                        ("idx", idx, torch.int32), ("w", w, torch.float32), ("counts", counts, torch.int32),
                        ("offsets", offsets, torch.int32), ("perm", perm, torch.int32)):
        _need_cuda(t, name, dt)
    _check(lib().moe_route(ctx, _ptr(x), x.shape[0], _ptr(router_w), _ptr(router_b), top_k, _ptr(idx), _ptr(w),
                           _ptr(counts), _ptr(offsets), _ptr(perm), _stream(stream)), "moe_route")


def moe_forward(ctx, x, router_w, router_b, experts_gate_up, experts_down, shared_w, top_k, y,
                stream=None, packed_weights=False) -> None:
    """``packed_weights``: the expert tensors are 4-bit planes (MOE_W_Q4G64, see
    moe.h), passed as raw byte buffers of any dtype."""
    import torch

    wdt = None if packed_weights else torch.bfloat16
    for name, t, dt in (("x", x, None), ("router_w", router_w, torch.float32), ("router_b", router_b, torch.float32),
                        ("experts_gate_up", experts_gate_up, wdt),
                        ("experts_down", experts_down, wdt), ("shared_w", shared_w, wdt),
                        ("y", y, x.dtype)):
        _need_cuda(t, name, dt)
    _check(lib().moe_forward(ctx, _ptr(x), x.shape[0], _ptr(router_w), _ptr(router_b), _ptr(experts_gate_up),
                             _ptr(experts_down), _ptr(shared_w), top_k, _ptr(y), _stream(stream)), "moe_forward")


def moe_last_routing(ctx, n_experts, stream=None) -> dict:
    """The routing tables the last ``moe_forward`` on ``ctx`` computed and used
    (idx, w, counts, offsets, perm, slot), as device tensors; see moe.h."""
    import torch

    T, k = ctypes.c_int(), ctypes.c_int()
    _check(lib().moe_last_routing(ctx, None, None, None, None, None, None, ctypes.byref(T), ctypes.byref(k), None),
           "moe_last_routing")
    T, k = T.value, k.value
    dev = torch.device("cuda", torch.cuda.current_device())
    out = dict(idx=torch.empty(T, k, dtype=torch.int32, device=dev), w=torch.empty(T, k, dtype=torch.float32, device=dev),
               counts=torch.empty(n_experts, dtype=torch.int32, device=dev),
               offsets=torch.empty(n_experts + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(T * k, dtype=torch.int32, device=dev),
               slot=torch.empty(T, k, dtype=torch.int32, device=dev))
    _check(lib().moe_last_routing(ctx, _ptr(out["idx"]), _ptr(out["w"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                                  _ptr(out["perm"]), _ptr(out["slot"]), None, None, _stream(stream)),
           "moe_last_routing")
    return out


def moe_decode_noalloc(x, router_w, router_b, experts_gate_up, experts_down, shared_w, top_k, y, status=None,
                       stream=None) -> None:
    """The small-T layer without a context, for callers that cannot allocate
    device memory (a plugin whose host owns every device buffer, a serving loop
    that must not risk an allocation's device synchronisation).  Scratch memory
    is a fixed device array inside the library; see moe.h."""
    import torch

    for name, t, dt in (("x", x, None), ("router_w", router_w, torch.float32), ("router_b", router_b, torch.float32),
                        ("experts_gate_up", experts_gate_up, torch.bfloat16),
                        ("experts_down", experts_down, torch.bfloat16), ("shared_w", shared_w, torch.bfloat16),
                        ("y", y, x.dtype), ("status", status, torch.int32)):
        _need_cuda(t, name, dt)
    T, d = x.shape
    E, inter = experts_down.shape[0], experts_down.shape[2]
    x_dtype = MOE_BF16 if x.dtype == torch.bfloat16 else MOE_F32
    _check(lib().moe_decode_noalloc(_ptr(x), T, x_dtype, d, E, inter, top_k, _ptr(router_w), _ptr(router_b),
                                    _ptr(experts_gate_up), _ptr(experts_down), _ptr(shared_w), _ptr(y), _ptr(status),
                                    _stream(stream)), "moe_decode_noalloc")


class MoeLayer:
    """Owns one context; ``forward`` / ``route`` call the C ABI on torch tensors."""

    def __init__(self, d, n_experts, inter, top_k, max_tokens, *, shared_inter=None, x_dtype=MOE_BF16,
                 has_router_bias=False, has_shared=True, bias_select_only=False, shared_gate=False,
                 weight_format=MOE_W_BF16):
        """``shared_gate``: sigmoid-gated shared expert; router_w then holds n_experts + 1
        rows, the last being the gate vector.  ``weight_format``: MOE_W_BF16, or
        MOE_W_Q4G64 for 4-bit experts (planes as in moe.h; see ``pack_q4``)."""
        self.top_k = top_k
        self.d = d
        self.n_experts = n_experts
        self.x_dtype = x_dtype
        self.weight_format = weight_format
        self.ctx = moe_init(d, n_experts, inter, inter if shared_inter is None else shared_inter, top_k,
                            max_tokens, x_dtype, has_router_bias, has_shared, bias_select_only, shared_gate,
                            weight_format)

    def forward(self, x, router_w, router_b, gate_up, down, shared_w, y=None, top_k=None, stream=None):
        import torch

        if y is None:
            y = torch.empty_like(x)
        moe_forward(self.ctx, x, router_w, router_b, gate_up, down, shared_w, top_k or self.top_k, y, stream,
                    packed_weights=self.weight_format == MOE_W_Q4G64)
        return y

    def route(self, x, router_w, router_b, top_k=None, stream=None):
        import torch

        k = top_k or self.top_k
        T = x.shape[0]
        E = self.n_experts
        dev = x.device
        out = dict(idx=torch.empty(T, k, dtype=torch.int32, device=dev),
                   w=torch.empty(T, k, dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   perm=torch.empty(T * k, dtype=torch.int32, device=dev))
        moe_route(self.ctx, x, router_w, router_b, k, stream=stream, **out)
        return out

    def last_routing(self, stream=None) -> dict:
        """Routing tables of the last ``forward`` (device tensors)."""
        return moe_last_routing(self.ctx, self.n_experts, stream)

    def status(self) -> int:
        return moe_status(self.ctx)

    def close(self):
        if self.ctx:
            moe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
