"""Python binding of the GB300 mixture-of-experts layer library (``include/moe.h``).

Argument marshalling only: every function takes torch tensors, checks that
they live on the current CUDA device, and passes raw pointers, sizes and the
current stream to the C ABI of ``libmoe_gb300.so``.  All arithmetic runs in
the library's CUDA kernels.  If the library has not been built the import of
any entry point raises; there is no fallback.

Helpers ``allocate_saved``, ``allocate_grads`` and ``workspace`` size buffers
with ``moe_max_rows`` / ``moe_workspace_size`` and allocate them with torch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_F32 = 0
MOE_BF16 = 1

STATUS = ["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_SHAPE", "MOE_ERR_DTYPE", "MOE_ERR_ALIGNMENT",
          "MOE_ERR_WORKSPACE", "MOE_ERR_CUDA", "MOE_ERR_DEVICE_CHECK", "MOE_ERR_TIMEOUT", "MOE_ERR_UNSUPPORTED"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        name = STATUS[code] if 0 <= code < len(STATUS) else str(code)
        super().__init__(f"{fn} returned {name}")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("capacity", ctypes.c_int32), ("dtype", ctypes.c_int32), ("aux_loss_coeff", ctypes.c_float)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("W_r", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("W1", ctypes.c_void_p),
                ("W3", ctypes.c_void_p), ("W2", ctypes.c_void_p)]


class MoeSaved(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("ids", "gates", "slot", "row_of", "src_token", "counts", "offsets",
                                               "probs", "x_perm", "a", "b", "h", "y_perm")]


class MoeGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dW_r", "dW1", "dW3", "dW2", "aux_loss")]


_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_CFG = ctypes.POINTER(MoeConfig)

# name -> argtypes (all return int status unless listed in _RESTYPES)
_SIGNATURES = {
    "moe_capacity": [_CFG, ctypes.POINTER(ctypes.c_int32)],
    "moe_max_rows": [_CFG, ctypes.POINTER(ctypes.c_int64)],
    "moe_workspace_size": [_CFG, _I, ctypes.POINTER(ctypes.c_size_t)],
    "moe_router_topk": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P],
    "moe_router_topk_noalloc": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_permute": [_CFG, _P, _P, _P, _P, _P, _P],
    "moe_grouped_ffn": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_unpermute_combine": [_CFG, _P, _P, _P, _P, _P],
    "moe_layer_fwd": [_CFG, ctypes.POINTER(MoeWeights), _P, _P, ctypes.POINTER(MoeSaved), _P, _Z, _P],
    "moe_combine_bwd": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_grouped_ffn_bwd": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P],
    "moe_unpermute_dx_router_bwd": [_CFG, _P, _P, _P, _P, _P, _P, _P, _I, _P, _Z, _P],
    "moe_aux_loss": [_CFG, _P, _P, _P, _P, _P, _Z, _P],
    "moe_layer_bwd": [_CFG, ctypes.POINTER(MoeWeights), _P, _P, ctypes.POINTER(MoeSaved), _P,
                      ctypes.POINTER(MoeGrads), _I, _P, _Z, _P],
    "moe_get_device_error": [ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), _I],
    "moe_launch_count": [],
    "moe_selftest_bounded_wait": [ctypes.c_int64, _I, _P],
    "moe_profiler_enable": [_I],
    "moe_kernel_kinds": [],
    "moe_profiler_filter": [ctypes.c_int32],
    "moe_nvtx_enable": [_I],
    "moe_kernel_name": [ctypes.c_int32],
    "moe_profiler_read": [ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)],
    "moe_status_string": [_I],
}
_RESTYPES = {"moe_launch_count": ctypes.c_uint64, "moe_kernel_kinds": ctypes.c_int32,
             "moe_kernel_name": ctypes.c_char_p, "moe_status_string": ctypes.c_char_p}

_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it was not built (no fallback exists)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m routing_permute_grouped_router_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(h, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib_handle = h
    return _lib_handle


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise MoeError(fn, code)


def config(T: int, d_model: int, d_ff: int, E: int, k: int, capacity_factor: float = 0.0, capacity: int = -1,
           dtype: int = MOE_BF16, aux_loss_coeff: float = 0.0) -> MoeConfig:
    return MoeConfig(T, d_model, d_ff, E, k, capacity_factor, capacity, dtype, aux_loss_coeff)


def config_of(shape, T: Optional[int] = None, aux_loss_coeff: float = 0.0) -> MoeConfig:
    """Config for a ``workload.LayerShape``."""
    return config(shape.T if T is None else T, shape.d_model, shape.d_ff, shape.E, shape.k, shape.capacity_factor,
                  shape.capacity, MOE_BF16 if shape.dtype == "bf16" else MOE_F32, aux_loss_coeff)


def _ptr(t) -> int:
    if t is None:
        return None
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if t.numel() > 0 and not t.is_cuda:
        raise ValueError("tensor must be on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ----------------------------- sizes ------------------------------------- #
def moe_capacity(cfg: MoeConfig) -> int:
    c = ctypes.c_int32()
    _check("moe_capacity", lib().moe_capacity(ctypes.byref(cfg), ctypes.byref(c)))
    return c.value


def moe_max_rows(cfg: MoeConfig) -> int:
    r = ctypes.c_int64()
    _check("moe_max_rows", lib().moe_max_rows(ctypes.byref(cfg), ctypes.byref(r)))
    return r.value


def moe_workspace_size(cfg: MoeConfig, training: int) -> int:
    b = ctypes.c_size_t()
    _check("moe_workspace_size", lib().moe_workspace_size(ctypes.byref(cfg), int(training), ctypes.byref(b)))
    return b.value


# ----------------------------- steps ------------------------------------- #
def moe_router_topk(cfg, x, W_r, bias, ids, gates, probs, slot, row_of, src_token, counts, offsets, ws,
                    stream=None) -> None:
    _check("moe_router_topk", lib().moe_router_topk(
        ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(ids), _ptr(gates), _ptr(probs), _ptr(slot),
        _ptr(row_of), _ptr(src_token), _ptr(counts), _ptr(offsets), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_router_topk_noalloc(cfg, x, W_r, bias, ids, gates, probs, slot, row_of, src_token, counts, offsets,
                            stream=None) -> None:
    """moe_router_topk without a workspace, for callers that cannot allocate device memory.

    The library keeps the routing scratch in its own static device array
    (MOE_NOALLOC_SCRATCH_BYTES), shared by every call on a device: do not let
    two of these calls overlap on the GPU.
    """
    _check("moe_router_topk_noalloc", lib().moe_router_topk_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(ids), _ptr(gates), _ptr(probs), _ptr(slot),
        _ptr(row_of), _ptr(src_token), _ptr(counts), _ptr(offsets), _stream(stream)))


def moe_permute(cfg, x, row_of, counts, offsets, x_perm, stream=None) -> None:
    _check("moe_permute", lib().moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(row_of), _ptr(counts),
                                            _ptr(offsets), _ptr(x_perm), _stream(stream)))


def moe_grouped_ffn(cfg, x_perm, counts, offsets, W1, W3, W2, h, y_perm, a=None, b=None, stream=None) -> None:
    _check("moe_grouped_ffn", lib().moe_grouped_ffn(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(counts), _ptr(offsets), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(h),
        _ptr(y_perm), _ptr(a), _ptr(b), _stream(stream)))


def moe_unpermute_combine(cfg, y_perm, row_of, gates, y, stream=None) -> None:
    _check("moe_unpermute_combine", lib().moe_unpermute_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(row_of), _ptr(gates), _ptr(y), _stream(stream)))


def _weights(w: dict) -> MoeWeights:
    return MoeWeights(_ptr(w["W_r"]), _ptr(w.get("bias")), _ptr(w["W1"]), _ptr(w["W3"]), _ptr(w["W2"]))


def _saved(s: dict) -> MoeSaved:
    return MoeSaved(*[_ptr(s[n]) for n, _ in MoeSaved._fields_])


def moe_layer_fwd(cfg, weights: dict, x, y, saved: Optional[dict], ws, stream=None) -> None:
    w = _weights(weights)
    sv = _saved(saved) if saved is not None else None
    _check("moe_layer_fwd", lib().moe_layer_fwd(
        ctypes.byref(cfg), ctypes.byref(w), _ptr(x), _ptr(y), ctypes.byref(sv) if sv is not None else None,
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine_bwd(cfg, dy, y_perm, ids, row_of, gates, probs, counts, offsets, dy_perm, dg, dl,
                    stream=None) -> None:
    _check("moe_combine_bwd", lib().moe_combine_bwd(
        ctypes.byref(cfg), _ptr(dy), _ptr(y_perm), _ptr(ids), _ptr(row_of), _ptr(gates), _ptr(probs),
        _ptr(counts), _ptr(offsets), _ptr(dy_perm), _ptr(dg), _ptr(dl), _stream(stream)))


def moe_grouped_ffn_bwd(cfg, x_perm, a, b, h, dy_perm, counts, offsets, W1, W3, W2, da, db, dx_perm, dW1, dW3,
                        dW2, accumulate: int, stream=None) -> None:
    _check("moe_grouped_ffn_bwd", lib().moe_grouped_ffn_bwd(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(a), _ptr(b), _ptr(h), _ptr(dy_perm), _ptr(counts), _ptr(offsets),
        _ptr(W1), _ptr(W3), _ptr(W2), _ptr(da), _ptr(db), _ptr(dx_perm), _ptr(dW1), _ptr(dW3), _ptr(dW2),
        int(accumulate), _stream(stream)))


def moe_unpermute_dx_router_bwd(cfg, x, dx_perm, row_of, dl, W_r, dx, dW_r, accumulate: int, ws,
                                stream=None) -> None:
    _check("moe_unpermute_dx_router_bwd", lib().moe_unpermute_dx_router_bwd(
        ctypes.byref(cfg), _ptr(x), _ptr(dx_perm), _ptr(row_of), _ptr(dl), _ptr(W_r), _ptr(dx), _ptr(dW_r),
        int(accumulate), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_aux_loss(cfg, probs, ids, loss, dl, ws, stream=None) -> None:
    """Auxiliary load-balancing loss: writes it to ``loss`` (1 fp32, or None) and adds its
    logit gradient to ``dl`` [T, E] in place (cfg.aux_loss_coeff; nothing when 0)."""
    _check("moe_aux_loss", lib().moe_aux_loss(ctypes.byref(cfg), _ptr(probs), _ptr(ids), _ptr(loss), _ptr(dl),
                                              _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_bwd(cfg, weights: dict, x, dy, saved: dict, dx, grads: dict, accumulate: int, ws,
                  stream=None) -> None:
    w = _weights(weights)
    sv = _saved(saved)
    g = MoeGrads(_ptr(grads["dW_r"]), _ptr(grads["dW1"]), _ptr(grads["dW3"]), _ptr(grads["dW2"]),
                 _ptr(grads.get("aux_loss")))
    _check("moe_layer_bwd", lib().moe_layer_bwd(
        ctypes.byref(cfg), ctypes.byref(w), _ptr(x), _ptr(dy), ctypes.byref(sv), _ptr(dx), ctypes.byref(g),
        int(accumulate), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_get_device_error(clear: bool = True):
    """(code, detail) from the device error word; waits for the device."""
    c, d = ctypes.c_int32(), ctypes.c_int32()
    _check("moe_get_device_error", lib().moe_get_device_error(ctypes.byref(c), ctypes.byref(d), int(clear)))
    return c.value, d.value


def moe_selftest_bounded_wait(limit_ns: int, arrive: bool, stream=None) -> None:
    """Run the bounded-wait self-test kernel (see include/moe.h)."""
    _check("moe_selftest_bounded_wait",
           lib().moe_selftest_bounded_wait(int(limit_ns), int(arrive), _stream(stream)))


def moe_launch_count() -> int:
    return int(lib().moe_launch_count())


def moe_profiler_enable(on: bool) -> None:
    _check("moe_profiler_enable", lib().moe_profiler_enable(int(on)))


def moe_profiler_filter(name: Optional[str]) -> None:
    """Profile only the kernel kind called ``name`` (None: every kind)."""
    idx = -1
    if name is not None:
        names = [lib().moe_kernel_name(i).decode() for i in range(lib().moe_kernel_kinds())]
        idx = names.index(name)
    _check("moe_profiler_filter", lib().moe_profiler_filter(idx))


def moe_nvtx_enable(on: bool) -> None:
    """NVTX ranges around every kernel launch and layer call (for nsys/ncu timelines)."""
    _check("moe_nvtx_enable", lib().moe_nvtx_enable(int(bool(on))))


def moe_profiler_read() -> dict:
    """{kernel name: (launches, total ms)} for kernels launched while the profiler was on."""
    out = {}
    for i in range(lib().moe_kernel_kinds()):
        n, ms = ctypes.c_int64(), ctypes.c_double()
        _check("moe_profiler_read", lib().moe_profiler_read(i, ctypes.byref(n), ctypes.byref(ms)))
        if n.value:
            out[lib().moe_kernel_name(i).decode()] = (n.value, ms.value)
    return out


# ----------------------------- allocation helpers ------------------------ #
def _act_dtype(cfg):
    import torch

    return torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32


def allocate_saved(cfg: MoeConfig, device="cuda", recompute: bool = False) -> dict:
    """Caller-owned routing state and activations for ``moe_layer_fwd``/``moe_layer_bwd``.
    recompute: keep neither a, b nor h (the backward recomputes them; workspace(cfg, 2))."""
    import torch

    R, T, k, E, d, f = moe_max_rows(cfg), max(cfg.T, 1), cfg.k, cfg.E, cfg.d_model, cfg.d_ff
    i32, f32, act = torch.int32, torch.float32, _act_dtype(cfg)
    return dict(ids=torch.empty(T, k, dtype=i32, device=device), gates=torch.empty(T, k, dtype=f32, device=device),
                slot=torch.empty(T, k, dtype=i32, device=device), row_of=torch.empty(T, k, dtype=i32, device=device),
                src_token=torch.empty(max(R, 1), dtype=i32, device=device),
                counts=torch.empty(E, dtype=i32, device=device), offsets=torch.empty(E + 1, dtype=i32, device=device),
                probs=torch.empty(T, E, dtype=f32, device=device),
                x_perm=torch.empty(max(R, 1), d, dtype=act, device=device),
                a=torch.empty(max(R, 1), f, dtype=act, device=device),
                b=torch.empty(max(R, 1), f, dtype=act, device=device),
                h=torch.empty(max(R, 1), f, dtype=act, device=device),
                y_perm=torch.empty(max(R, 1), d, dtype=act, device=device)) if not recompute else dict(
                ids=torch.empty(T, k, dtype=i32, device=device), gates=torch.empty(T, k, dtype=f32, device=device),
                slot=torch.empty(T, k, dtype=i32, device=device), row_of=torch.empty(T, k, dtype=i32, device=device),
                src_token=torch.empty(max(R, 1), dtype=i32, device=device),
                counts=torch.empty(E, dtype=i32, device=device), offsets=torch.empty(E + 1, dtype=i32, device=device),
                probs=torch.empty(T, E, dtype=f32, device=device),
                x_perm=torch.empty(max(R, 1), d, dtype=act, device=device), a=None, b=None, h=None,
                y_perm=torch.empty(max(R, 1), d, dtype=act, device=device))


def allocate_grads(cfg: MoeConfig, device="cuda") -> dict:
    import torch

    E, d, f = cfg.E, cfg.d_model, cfg.d_ff
    z = dict(dtype=torch.float32, device=device)
    return dict(dW_r=torch.zeros(d, E, **z), dW1=torch.zeros(E, d, f, **z), dW3=torch.zeros(E, d, f, **z),
                dW2=torch.zeros(E, f, d, **z), aux_loss=torch.zeros(1, **z))


def workspace(cfg: MoeConfig, training: int, device="cuda"):
    import torch

    return torch.empty(moe_workspace_size(cfg, training), dtype=torch.uint8, device=device)
