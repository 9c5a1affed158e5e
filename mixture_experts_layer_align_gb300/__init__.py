"""GB300 (sm_103a) fused Mixture-of-Experts layer forward.

Thin Python binding over the C ABI in include/moe_gb300.h
(libmoe_gb300.so, built in-tree by `build.py`).  Functions keep the C names
and only marshal arguments: tensors become device pointers, the current torch
stream becomes the cudaStream_t, outputs and workspaces are allocated with
torch.  Every step of the layer runs in the library's CUDA kernels; there is
no fallback path, and a missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_DT_BF16 = 0
MOE_DT_FP8_E4M3 = 1
MOE_DEBUG_FORCE_TIMEOUT = 0x1
MOE_DEBUG_TRACE = 0x2
MOE_FLAG_TOKENS_IN_M = 0x4   # both GEMMs: tokens in the MMA M slot (ablation of the swap)
MOE_FLAG_WEIGHTS_IN_M = 0x8  # both GEMMs: weight rows in the MMA M slot
MOE_FLAG_NO_SM_PAIRS = 0x10  # wide FP8 gate/up tiles on one SM each (ablation of the SM pairs)
MOE_FLAG_ONE_KERNEL = 0x20  # small batches: the whole layer as one cooperative kernel
TRACE_MAX_CTAS = 256
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT",
                6: "MOE_ERR_DEVICE_RANGE"}

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})"
        if status == 4:
            msg += f" [{load().moe_last_error_detail().decode()}]"
        super().__init__(msg)


class MoeFusedArgs(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("router_logits", ctypes.c_void_p),
        ("w13", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("w13_scale", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p),
        ("weight_dtype", ctypes.c_int),
        ("T", ctypes.c_int),
        ("H", ctypes.c_int),
        ("I", ctypes.c_int),
        ("E", ctypes.c_int),
        ("top_k", ctypes.c_int),
        ("renormalize", ctypes.c_int),
        ("out", ctypes.c_void_p),
        ("topk_ids_out", ctypes.c_void_p),
        ("topk_w_out", ctypes.c_void_p),
        ("counts_out", ctypes.c_void_p),
        ("debug_flags", ctypes.c_int),
    ]


def load():
    """Load libmoe_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_layer_align_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_route_topk.argtypes = [P, i, i, i, i, P, P, P]
        L.moe_align_by_expert.argtypes = [P, i, i, i, i, P, P, P, P, P, P]
        L.moe_quantize_scratch_size.argtypes = [i, i]
        L.moe_quantize_scratch_size.restype = sz
        L.moe_quantize_e4m3.argtypes = [P, i, i, P, P, P, sz, P]
        L.moe_quantize_e4m3_noalloc.argtypes = [P, i, i, P, P, P]
        L.moe_inv_rope_scratch_size.argtypes = [i, i, i]
        L.moe_inv_rope_scratch_size.restype = sz
        L.moe_inv_rope_quant_per_head.argtypes = [P, P, P, P, i, i, i, i, P, P, P, sz, P]
        L.moe_quantize_e4m3_noalloc.restype = ctypes.c_int
        L.moe_fused_trace_offset.argtypes = [i, i, i, i, i, i]
        L.moe_fused_trace_offset.restype = sz
        L.moe_fused_workspace_size.argtypes = [i, i, i, i, i, i]
        L.moe_fused_workspace_size.restype = sz
        L.moe_fused_launch_count.argtypes = [i, i, i, i, i, i]
        L.moe_fused_launch_count.restype = i
        L.moe_fused_forward.argtypes = [ctypes.POINTER(MoeFusedArgs), P, sz, P]
        L.moe_fused_forward_timed.argtypes = [ctypes.POINTER(MoeFusedArgs), P, sz, P,
                                               ctypes.POINTER(ctypes.c_void_p), i]
        L.moe_fused_forward_gate_up.argtypes = [ctypes.POINTER(MoeFusedArgs), P, sz, P]
        L.moe_fused_forward_down.argtypes = [ctypes.POINTER(MoeFusedArgs), P, sz, P]
        L.moe_fused_h_amax_offset.argtypes = []
        L.moe_fused_h_amax_offset.restype = sz
        L.moe_check_status.argtypes = [P, P]
        L.moe_status_string.argtypes = [i]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_error_detail.argtypes = []
        L.moe_last_error_detail.restype = ctypes.c_char_p
        for name in ("moe_route_topk", "moe_align_by_expert", "moe_quantize_e4m3",
                     "moe_fused_forward", "moe_fused_forward_timed", "moe_check_status",
                     "moe_fused_forward_gate_up", "moe_fused_forward_down"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
        return _lib


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require(t, dtype, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device and uses its per-device state
        raise ValueError(f"{name} is on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.device(...))")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def moe_route_topk(logits, top_k: int, renormalize: bool, topk_ids=None, topk_w=None, stream=None):
    """Router: softmax + top-k (+ renormalisation).  Returns (ids int32, w fp32), [T, k]."""
    import torch
    _require(logits, torch.float32, "logits")
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty(T, top_k, dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty(T, top_k, dtype=torch.float32, device=logits.device)
    _require(topk_ids, torch.int32, "topk_ids", (T, top_k))
    _require(topk_w, torch.float32, "topk_w", (T, top_k))
    _check(load().moe_route_topk(_ptr(logits), T, E, top_k, int(bool(renormalize)), _ptr(topk_ids),
                                 _ptr(topk_w), _stream(stream)), "moe_route_topk")
    return topk_ids, topk_w


def moe_align_by_expert(topk_ids, E: int, block_m: int, stream=None):
    """Alignment by expert.  Returns dict(counts, offsets, sorted_ids, tile_expert,
    num_padded) as device tensors (sorted_ids / tile_expert at capacity size)."""
    import torch
    _require(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    P = T * k
    cap = P + E * (block_m - 1)
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_ids = torch.full((max(cap, 1),), -1, dtype=torch.int32, device=dev)
    tile_expert = torch.full((max(cap // block_m, 1),), -1, dtype=torch.int32, device=dev)
    num_padded = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(load().moe_align_by_expert(_ptr(topk_ids), T, k, E, block_m, _ptr(counts),
                                      _ptr(offsets), _ptr(sorted_ids), _ptr(tile_expert),
                                      _ptr(num_padded), _stream(stream)), "moe_align_by_expert")
    return dict(counts=counts, offsets=offsets, sorted_ids=sorted_ids, tile_expert=tile_expert,
                num_padded=num_padded)


def moe_quantize_e4m3(x, stream=None):
    """Dynamic per-tensor E4M3 quantisation of bf16 x.  Returns (codes uint8, scale fp32[1])."""
    import torch
    _require(x, torch.bfloat16, "x")
    T, H = x.shape
    L = load()
    xq = torch.empty(T, H, dtype=torch.uint8, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    nscr = L.moe_quantize_scratch_size(T, H)
    scratch = torch.empty(max(nscr, 16), dtype=torch.uint8, device=x.device)
    _check(L.moe_quantize_e4m3(_ptr(x), T, H, _ptr(xq), _ptr(scale), _ptr(scratch), nscr,
                               _stream(stream)), "moe_quantize_e4m3")
    return xq, scale


def moe_quantize_e4m3_noalloc(x, x_q=None, scale=None, stream=None):
    """moe_quantize_e4m3 for callers that cannot allocate device scratch: the
    library's static device array holds the partial maxima (shared by all
    calls on a device; overlapping calls race).  Outputs may be passed in;
    when omitted they are allocated here by torch, outside the C call.
    Returns (codes uint8 [T,H], scale fp32 [1])."""
    import torch
    _require(x, torch.bfloat16, "x")
    T, H = x.shape
    if x_q is None:
        x_q = torch.empty(T, H, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
    _require(x_q, torch.uint8, "x_q", (T, H))
    _require(scale, torch.float32, "scale", (1,))
    _check(load().moe_quantize_e4m3_noalloc(_ptr(x), T, H, _ptr(x_q), _ptr(scale),
                                            _stream(stream)), "moe_quantize_e4m3_noalloc")
    return x_q, scale


def moe_inv_rope_scratch_size(T: int, NH: int, D: int) -> int:
    return int(load().moe_inv_rope_scratch_size(T, NH, D))


def moe_inv_rope_quant_per_head(x, positions, cos_tab, sin_tab, codes=None, scales=None,
                                scratch=None, stream=None):
    """Inverse rotary embedding of each head vector, then one dynamic E4M3
    scale per head.  x: bf16 [T, NH, D]; positions: int32 [T]; cos_tab,
    sin_tab: fp32 [max_pos, D/2].  Returns (codes uint8 [T, NH, D], scales fp32
    [NH]); `scratch` (uint8, moe_inv_rope_scratch_size bytes) may be passed in."""
    import torch
    _require(x, torch.bfloat16, "x")
    T, NH, D = x.shape
    _require(positions, torch.int32, "positions", (T,))
    _require(cos_tab, torch.float32, "cos_tab")
    max_pos = cos_tab.shape[0]
    _require(cos_tab, torch.float32, "cos_tab", (max_pos, D // 2))
    _require(sin_tab, torch.float32, "sin_tab", (max_pos, D // 2))
    if codes is None:
        codes = torch.empty(T, NH, D, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(NH, dtype=torch.float32, device=x.device)
    _require(codes, torch.uint8, "codes", (T, NH, D))
    _require(scales, torch.float32, "scales", (NH,))
    n = moe_inv_rope_scratch_size(T, NH, D)
    if n == 0:
        raise MoeError(1, "moe_inv_rope_scratch_size")
    if scratch is None:
        scratch = torch.empty(n, dtype=torch.uint8, device=x.device)
    _check(load().moe_inv_rope_quant_per_head(_ptr(x), _ptr(positions), _ptr(cos_tab),
                                              _ptr(sin_tab), T, NH, D, max_pos, _ptr(codes),
                                              _ptr(scales), _ptr(scratch), scratch.numel(),
                                              _stream(stream)), "moe_inv_rope_quant_per_head")
    return codes, scales, scratch


def moe_fused_workspace_size(T: int, H: int, I: int, E: int, top_k: int, dtype: int) -> int:
    return int(load().moe_fused_workspace_size(T, H, I, E, top_k, dtype))


def moe_fused_launch_count(T: int, H: int, I: int, E: int, top_k: int, dtype: int) -> int:
    """Kernels one moe_fused_forward call launches (-1: invalid sizes)."""
    return int(load().moe_fused_launch_count(T, H, I, E, top_k, dtype))


def alloc_workspace(T, H, I, E, top_k, dtype, device="cuda"):
    import torch
    n = moe_fused_workspace_size(T, H, I, E, top_k, dtype)
    if n == 0:
        raise MoeError(1, "moe_fused_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _fused_args(x, router_logits, w13, w2, w13_scale, w2_scale, top_k, renormalize, out,
                topk_ids_out, topk_w_out, counts_out, debug_flags):
    import torch
    _require(x, torch.bfloat16, "x")
    _require(router_logits, torch.float32, "router_logits")
    T, H = x.shape
    E = router_logits.shape[1]
    fp8 = w13_scale is not None
    wdt = torch.uint8 if fp8 else torch.bfloat16
    _require(w13, wdt, "w13")
    _require(w2, wdt, "w2")
    I = w13.shape[1] // 2
    if tuple(w13.shape) != (E, 2 * I, H) or tuple(w2.shape) != (E, H, I):
        raise ValueError("w13 must be [E,2I,H] and w2 [E,H,I]")
    if fp8:
        _require(w13_scale, torch.float32, "w13_scale", (E,))
        _require(w2_scale, torch.float32, "w2_scale", (E,))
    dtype = MOE_DT_FP8_E4M3 if fp8 else MOE_DT_BF16
    _require(out, torch.bfloat16, "out", (T, H))
    if topk_ids_out is not None:
        _require(topk_ids_out, torch.int32, "topk_ids_out", (T, top_k))
    if topk_w_out is not None:
        _require(topk_w_out, torch.float32, "topk_w_out", (T, top_k))
    if counts_out is not None:
        _require(counts_out, torch.int32, "counts_out", (E,))
    args = MoeFusedArgs(
        x=x.data_ptr(), router_logits=router_logits.data_ptr(), w13=w13.data_ptr(),
        w2=w2.data_ptr(), w13_scale=w13_scale.data_ptr() if fp8 else None,
        w2_scale=w2_scale.data_ptr() if fp8 else None, weight_dtype=dtype, T=T, H=H, I=I, E=E,
        top_k=top_k, renormalize=int(bool(renormalize)), out=out.data_ptr(),
        topk_ids_out=topk_ids_out.data_ptr() if topk_ids_out is not None else None,
        topk_w_out=topk_w_out.data_ptr() if topk_w_out is not None else None,
        counts_out=counts_out.data_ptr() if counts_out is not None else None,
        debug_flags=int(debug_flags))
    return args, (T, H, I, E, dtype)


def moe_fused_forward(x, router_logits, w13, w2, w13_scale, w2_scale, top_k: int,
                      renormalize: bool = True, out=None, workspace=None, topk_ids_out=None,
                      topk_w_out=None, counts_out=None, debug_flags: int = 0, stream=None,
                      events=None):
    """Fused MoE layer forward (see include/moe_gb300.h).

    x bf16 [T,H]; router_logits fp32 [T,E]; w13 [E,2I,H] and w2 [E,H,I] as uint8
    E4M3 codes (with fp32 [E] scales) or bf16 (scales None).  Returns out bf16 [T,H].
    With a caller `workspace` the call is asynchronous and device-side errors
    are read with moe_check_status(workspace); without one, a workspace is
    allocated for this call and its status is checked before returning (the
    stream is synchronised and a device-side error raises MoeError).
    `events`: optional list of 8 recorded torch.cuda.Event (enable_timing) that
    bracket the seven steps (moe_fused_forward_timed).
    """
    import torch
    if out is None:
        out = torch.empty(x.shape[0], x.shape[1], dtype=torch.bfloat16, device=x.device)
    args, (T, H, I, E, dtype) = _fused_args(x, router_logits, w13, w2, w13_scale, w2_scale,
                                            top_k, renormalize, out, topk_ids_out, topk_w_out,
                                            counts_out, debug_flags)
    own_ws = workspace is None
    if own_ws:
        workspace = alloc_workspace(T, H, I, E, top_k, dtype, x.device)
    L = load()
    if events is None:
        st = L.moe_fused_forward(ctypes.byref(args), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
        _check(st, "moe_fused_forward")
    else:
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        st = L.moe_fused_forward_timed(ctypes.byref(args), _ptr(workspace), workspace.numel(),
                                       _stream(stream), arr, len(events))
        _check(st, "moe_fused_forward_timed")
    if own_ws and T > 0:
        # nobody else can read a throwaway workspace's status word: read it
        # here (this synchronises the stream; pass a workspace to avoid that)
        _check(moe_check_status(workspace, stream), "moe_fused_forward (device status)")
    return out


def moe_fused_forward_gate_up(x, router_logits, w13, w2, w13_scale, w2_scale, top_k: int,
                              renormalize: bool, out, workspace, stream=None):
    """First of the two calls of a tensor-parallel shard (include/moe_gb300.h):
    routing through the gate/up GEMM; this rank's max |h| is left in the
    workspace (see h_amax_view)."""
    args, _ = _fused_args(x, router_logits, w13, w2, w13_scale, w2_scale, top_k, renormalize,
                          out, None, None, None, 0)
    _check(load().moe_fused_forward_gate_up(ctypes.byref(args), _ptr(workspace),
                                            workspace.numel(), _stream(stream)),
           "moe_fused_forward_gate_up")


def moe_fused_forward_down(x, router_logits, w13, w2, w13_scale, w2_scale, top_k: int,
                           renormalize: bool, out, workspace, stream=None):
    """Second call: h codes with the scale from the workspace's max |h| word,
    the down GEMM and the combine into `out` (this rank's partial output)."""
    args, _ = _fused_args(x, router_logits, w13, w2, w13_scale, w2_scale, top_k, renormalize,
                          out, None, None, None, 0)
    _check(load().moe_fused_forward_down(ctypes.byref(args), _ptr(workspace),
                                         workspace.numel(), _stream(stream)),
           "moe_fused_forward_down")
    return out


def h_amax_view(workspace):
    """The workspace's fp32 max |h| word as a one-element tensor view."""
    import torch
    off = int(load().moe_fused_h_amax_offset())
    return workspace[off:off + 4].view(torch.float32)


def make_step_events(n: int = 8):
    """n timing events, each recorded once so that its CUDA handle exists."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    return evs


def read_trace(workspace, T, H, I, E, top_k, dtype):
    """Per-CTA %globaltimer stamps left by a MOE_DEBUG_TRACE call: uint64
    [2 kernels][TRACE_MAX_CTAS][entry, inputs ready, first weights, exit]."""
    import torch
    off = int(load().moe_fused_trace_offset(T, H, I, E, top_k, dtype))
    n = 2 * TRACE_MAX_CTAS * 4 * 8
    raw = workspace[off:off + n].cpu()
    return raw.view(torch.int64).reshape(2, TRACE_MAX_CTAS, 4)


def moe_check_status(workspace, stream=None) -> int:
    """Synchronise and return the status the last call left in the workspace (0 = MOE_OK)."""
    return int(load().moe_check_status(_ptr(workspace), _stream(stream)))


__all__ = ["load", "moe_fused_forward_gate_up", "moe_fused_forward_down", "h_amax_view",
           "moe_route_topk", "moe_align_by_expert", "moe_quantize_e4m3",
           "moe_fused_workspace_size", "moe_fused_launch_count", "moe_inv_rope_scratch_size",
           "moe_inv_rope_quant_per_head", "moe_fused_forward", "moe_check_status", "alloc_workspace",
           "status_string", "MoeError", "make_step_events", "MoeFusedArgs", "MOE_DT_BF16", "MOE_DT_FP8_E4M3",
           "MOE_DEBUG_FORCE_TIMEOUT", "MOE_FLAG_TOKENS_IN_M",
           "MOE_FLAG_WEIGHTS_IN_M", "MOE_FLAG_NO_SM_PAIRS", "MOE_FLAG_ONE_KERNEL", "LIB_PATH"]
