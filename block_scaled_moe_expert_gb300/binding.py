"""Python binding of the C ABI in include/moe_experts.h (ctypes).

Argument marshalling only: every step of the forward runs in the CUDA
library. torch provides device memory and the current stream. If the library
is missing the calls raise; there is no fallback.

The Python-level refusals follow the transformers pages: a non-bf16 hidden
state raises ValueError (deepgemm excerpt), a static activation scheme
raises NotImplementedError (finegrained_fp8 page: the grouped dispatch only
quantizes activations dynamically), and tensors on another device than the
current one raise RuntimeError (the multi-device refusal).
"""
import ctypes
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbsmoe.so")

MOE_W_FP8 = 0
MOE_W_FP4 = 1
MOE_W_FP4_ACT_FP4 = 2
# format names of the prepared weights: the weight format, and for FP4
# weights used with FP4 activations "fp4_act_fp4"
FMT = {"fp8": MOE_W_FP8, "fp4": MOE_W_FP4, "fp4_act_fp4": MOE_W_FP4_ACT_FP4}

MOE_OK = 0
MOE_DEV_BAD_EXPERT_ID = 0x1
MOE_DEV_TIMEOUT = 0x2

_c = ctypes
_vp, _sz, _int, _f32 = _c.c_void_p, _c.c_size_t, _c.c_int, _c.c_float


class MoeLayout(_c.Structure):
    _fields_ = [("total_bytes", _sz), ("status", _sz), ("counts", _sz), ("offsets", _sz),
                ("padded_offsets", _sz), ("perm", _sz), ("inv", _sz), ("row_slot", _sz), ("tiles", _sz),
                ("xq", _sz), ("xsf", _sz), ("act", _sz), ("asf", _sz), ("y", _sz),
                ("row_capacity", _c.c_int32), ("row_align", _c.c_int32), ("xq_cols", _c.c_int32),
                ("act_cols", _c.c_int32), ("x_blocks", _c.c_int32), ("act_blocks", _c.c_int32)]


_SIGS = {
    "moe_status_string": (_c.c_char_p, [_int]),
    "moe_abi_version": (_int, []),
    "moe_prepared_w13_bytes": (_sz, [_int, _int, _int, _int]),
    "moe_prepared_w2_bytes": (_sz, [_int, _int, _int, _int]),
    "moe_workspace_bytes": (_sz, [_int, _int, _int, _int, _int, _int]),
    "moe_prepare_weights": (_int, [_int, _int, _int, _int, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp]),
    "moe_prepare_weights_transposed": (_int, [_int, _int, _int, _int, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp]),
    "moe_experts_forward": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _vp, _vp, _f32, _vp, _sz,
                                   _vp, _vp]),
    "moe_experts_forward_timed": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _vp, _vp, _f32, _vp,
                                         _sz, _vp, _vp, _c.POINTER(_vp)]),
    "moe_experts_forward_static": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _vp, _vp, _f32,
                                          _vp, _vp]),
    "moe_static_workspace_capacity": (_sz, []),
    "moe_static_get_device_status": (_int, [_vp, _c.POINTER(_c.c_uint32)]),
    "moe_debug_forward_act_f32": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _vp, _vp, _f32, _vp,
                                         _sz, _vp, _vp, _sz, _vp]),
    "moe_get_device_status": (_int, [_vp, _vp, _c.POINTER(_c.c_uint32)]),
    "moe_selftest_wait_timeout": (_int, [_vp, _c.c_size_t, _vp]),
    "moe_query_workspace_layout": (_int, [_int, _int, _int, _int, _int, _int, _c.POINTER(MoeLayout)]),
}

_lib = None


def lib():
    """Load libbsmoe.so (built in tree by build.py). Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with block_scaled_moe_expert_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class MoeError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {lib().moe_status_string(status).decode()}")


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


def _stream():
    return _vp(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return _vp(t.data_ptr())


def _same_device(*ts):
    dev = torch.cuda.current_device()
    for t in ts:
        if t.device.type != "cuda" or t.device.index != dev:
            raise RuntimeError("all tensors must live on the current CUDA device (one device per call)")


def workspace_bytes(fmt, T, H, I, E, K):
    n = lib().moe_workspace_bytes(FMT[fmt], T, H, I, E, K)
    if n == 0:
        raise MoeError(2, "moe_workspace_bytes")
    return n


def workspace_layout(fmt, T, H, I, E, K):
    out = MoeLayout()
    _check(lib().moe_query_workspace_layout(FMT[fmt], T, H, I, E, K, _c.byref(out)), "moe_query_workspace_layout")
    return out


class PreparedWeights:
    """Kernel-layout weights made once by moe_prepare_weights."""

    def __init__(self, fmt, E, H, I, w13_prep, w2_prep):
        self.fmt, self.E, self.H, self.I = fmt, E, H, I
        self.w13_prep, self.w2_prep = w13_prep, w2_prep

    @property
    def act_fmt(self):
        return "fp4" if self.fmt == "fp4_act_fp4" else "fp8"


def prepare_weights(weights, transposed=False, activations="fp8"):
    """weights: dict(fmt, E, H, I, w13, w13_scale, w2, w2_scale) of CUDA tensors,
    K-major ([E, N, K]) or, with transposed=True, N-major ([E, K, N]; see
    moe_prepare_weights_transposed for the exact shapes). activations="fp4"
    (FP4 weights only) selects the FP4 x FP4 variant for every forward with
    these prepared weights: e2m1 activations in 1x32 blocks."""
    fmt, E, H, I = weights["fmt"], weights["E"], weights["H"], weights["I"]
    if activations not in ("fp8", "fp4"):
        raise ValueError(f"activations must be 'fp8' or 'fp4', got {activations!r}")
    if activations == "fp4":
        if fmt != "fp4":
            raise ValueError("FP4 activations are available with FP4 weights only")
        fmt = "fp4_act_fp4"
    ts = [weights[k].contiguous() for k in ("w13", "w13_scale", "w2", "w2_scale")]
    _same_device(*ts)
    L = lib()
    n13 = L.moe_prepared_w13_bytes(FMT[fmt], E, H, I)
    n2 = L.moe_prepared_w2_bytes(FMT[fmt], E, H, I)
    if n13 == 0 or n2 == 0:
        raise MoeError(2, "moe_prepared_*_bytes")
    dev = ts[0].device
    p13 = torch.empty(n13, dtype=torch.uint8, device=dev)
    p2 = torch.empty(n2, dtype=torch.uint8, device=dev)
    fn = "moe_prepare_weights_transposed" if transposed else "moe_prepare_weights"
    _check(getattr(L, fn)(FMT[fmt], E, H, I, *[_ptr(t) for t in ts], _ptr(p13), n13, _ptr(p2), n2, _stream()), fn)
    return PreparedWeights(fmt, E, H, I, p13, p2)


def experts_forward(hidden, topk_idx, topk_w, prepared, swiglu_limit=None, workspace=None, out=None,
                    activation_scheme="dynamic"):
    """bf16 [T, H] experts forward; returns `out` (allocated if None)."""
    if activation_scheme == "static":
        raise NotImplementedError("the grouped experts forward quantizes activations dynamically per block; "
                                  "static activation scales are not supported")
    if hidden.dtype != torch.bfloat16:
        raise ValueError(f"the experts forward requires bfloat16 hidden states, got {hidden.dtype}")
    if topk_idx.dtype != torch.int32 or topk_w.dtype != torch.float32:
        raise ValueError("topk_idx must be int32 and topk_w float32")
    T, H = hidden.shape
    K = topk_idx.shape[1]
    p = prepared
    if H != p.H:
        raise ValueError(f"hidden size {H} does not match the prepared weights ({p.H})")
    hidden, topk_idx, topk_w = hidden.contiguous(), topk_idx.contiguous(), topk_w.contiguous()
    _same_device(hidden, topk_idx, topk_w, p.w13_prep, p.w2_prep)
    need = workspace_bytes(p.fmt, T, H, p.I, p.E, K)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=hidden.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=hidden.device)
    limit = float("nan") if swiglu_limit is None else float(swiglu_limit)
    _check(lib().moe_experts_forward(_ptr(hidden), _ptr(topk_idx), _ptr(topk_w), T, H, p.I, p.E, K, FMT[p.fmt],
                                     _ptr(p.w13_prep), _ptr(p.w2_prep), limit, _ptr(workspace),
                                     workspace.numel(), _ptr(out), _stream()), "moe_experts_forward")
    return out


def experts_forward_timed(hidden, topk_idx, topk_w, prepared, events, swiglu_limit=None, workspace=None,
                          out=None):
    """experts_forward that records 6 torch.cuda.Event objects at the stage
    boundaries (before routing, after routing, quantization, GEMM1, GEMM2,
    combine) on the current stream."""
    T, H = hidden.shape
    K = topk_idx.shape[1]
    p = prepared
    if workspace is None:
        workspace = torch.empty(workspace_bytes(p.fmt, T, H, p.I, p.E, K), dtype=torch.uint8, device=hidden.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=hidden.device)
    ev = (_vp * 6)(*[_vp(e.cuda_event) for e in events])
    limit = float("nan") if swiglu_limit is None else float(swiglu_limit)
    _check(lib().moe_experts_forward_timed(_ptr(hidden), _ptr(topk_idx), _ptr(topk_w), T, H, p.I, p.E, K,
                                           FMT[p.fmt], _ptr(p.w13_prep), _ptr(p.w2_prep), limit, _ptr(workspace),
                                           workspace.numel(), _ptr(out), _stream(), ev), "moe_experts_forward_timed")
    return out


def experts_forward_static(hidden, topk_idx, topk_w, prepared, swiglu_limit=None, out=None):
    """experts_forward without a workspace: the library's fixed device array
    (moe_static_workspace_capacity() bytes) is the scratch memory, for
    callers that cannot allocate. Calls on one device must not overlap."""
    if hidden.dtype != torch.bfloat16:
        raise ValueError(f"the experts forward requires bfloat16 hidden states, got {hidden.dtype}")
    T, H = hidden.shape
    K = topk_idx.shape[1]
    p = prepared
    hidden, topk_idx, topk_w = hidden.contiguous(), topk_idx.contiguous(), topk_w.contiguous()
    _same_device(hidden, topk_idx, topk_w, p.w13_prep, p.w2_prep)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=hidden.device)
    limit = float("nan") if swiglu_limit is None else float(swiglu_limit)
    _check(lib().moe_experts_forward_static(_ptr(hidden), _ptr(topk_idx), _ptr(topk_w), T, H, p.I, p.E, K,
                                            FMT[p.fmt], _ptr(p.w13_prep), _ptr(p.w2_prep), limit, _ptr(out),
                                            _stream()), "moe_experts_forward_static")
    return out


def debug_forward_act_f32(hidden, topk_idx, topk_w, prepared, swiglu_limit=None, workspace=None):
    """Test tap: the forward that also returns GEMM1's fp32 SwiGLU values,
    [row_capacity, act_cols] in padded grouped row order (see
    moe_debug_forward_act_f32). Returns (out, act_f32, workspace)."""
    T, H = hidden.shape
    K = topk_idx.shape[1]
    p = prepared
    lay = workspace_layout(p.fmt, T, H, p.I, p.E, K)
    if workspace is None:
        workspace = torch.empty(lay.total_bytes, dtype=torch.uint8, device=hidden.device)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=hidden.device)
    act = torch.zeros(lay.row_capacity, lay.act_cols, dtype=torch.float32, device=hidden.device)
    limit = float("nan") if swiglu_limit is None else float(swiglu_limit)
    _check(lib().moe_debug_forward_act_f32(_ptr(hidden), _ptr(topk_idx), _ptr(topk_w), T, H, p.I, p.E, K,
                                           FMT[p.fmt], _ptr(p.w13_prep), _ptr(p.w2_prep), limit, _ptr(workspace),
                                           workspace.numel(), _ptr(out), _ptr(act), act.numel() * 4, _stream()),
           "moe_debug_forward_act_f32")
    return out, act, workspace


def static_device_status():
    """Synchronize and return the flags of the most recent static forward."""
    flags = _c.c_uint32(0)
    lib().moe_static_get_device_status(_stream(), _c.byref(flags))
    return int(flags.value)


def device_status(workspace):
    """Synchronize and return the forward's device flags (0 if clean)."""
    flags = _c.c_uint32(0)
    lib().moe_get_device_status(_ptr(workspace), _stream(), _c.byref(flags))
    return int(flags.value)


def selftest_wait_timeout(workspace):
    """Run the bounded-wait self-test (about one second on the GPU) and
    return the device flags it left (MOE_DEV_TIMEOUT when the path works)."""
    _check(lib().moe_selftest_wait_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream()), "moe_selftest_wait_timeout")
    return device_status(workspace)


def header_symbols():
    """Names of the functions declared in include/moe_experts.h."""
    import re
    path = os.path.join(os.path.dirname(HERE), "include", "moe_experts.h")
    src = open(path).read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


__all__ = ["lib", "MoeError", "prepare_weights", "experts_forward", "experts_forward_timed", "experts_forward_static",
           "workspace_bytes", "workspace_layout", "debug_forward_act_f32", "static_device_status",
           "device_status", "selftest_wait_timeout", "PreparedWeights", "header_symbols", "MOE_DEV_BAD_EXPERT_ID", "MOE_DEV_TIMEOUT"]
