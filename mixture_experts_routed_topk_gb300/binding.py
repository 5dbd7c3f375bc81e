"""ctypes binding of ``libmoe_gb300.so`` (the C ABI in ``include/moe_routed_experts.h``).

Argument marshalling only: every function takes torch tensors, checks that they are what the C
entry point expects (device, dtype, contiguity, shape), passes their device pointers and sizes to
the entry point of the same name, and raises :class:`MoeError` on a non-``MOE_OK`` status. All
computation runs in the library's CUDA kernels; there is no fallback of any kind, and a missing
library raises at the first call.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MOE_OK = 0
MOE_SCORES_F32 = 0
MOE_SCORES_BF16 = 1
MOE_DEV_BAD_EXPERT_ID = 1
MOE_DEV_TIMEOUT = 2

WS_REGIONS = (
    "status", "counts", "offsets", "tiles1", "tiles2", "block_counts", "block_bases",
    "perm", "inv", "xp", "h", "rms", "ready", "y", "total",
)
MOE_WEIGHT_W13 = 0
MOE_WEIGHT_W2 = 1
MXWS_REGIONS = (
    "status", "counts", "offsets", "tiles", "tiles2", "block_counts", "block_bases",
    "perm", "inv", "xq", "xs", "hq", "hs", "y", "total",
)

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIBRARY


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIBRARY
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library {p} is missing; build it with mixture_experts_routed_topk_gb300.build.build()"
            )
        lib = ctypes.CDLL(p)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "moe_workspace_bytes": ([i64, i32, i32, i32, i32], sz),
            "moe_workspace_layout": ([i64, i32, i32, i32, i32, vp], ctypes.c_int),
            "moe_routing_workspace_bytes": ([i64, i32, i32], sz),
            "moe_routing": ([vp, i64, i32, i32, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "moe_routed_experts_fwd": (
                [vp, vp, vp, i32, vp, vp, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_mega_workspace_bytes": ([i64, i32, i32, i32, i32], sz),
            "moe_mega_workspace_layout": ([i64, i32, i32, i32, i32, vp], ctypes.c_int),
            "moe_routed_experts_fwd_mega": (
                [vp, vp, vp, i32, vp, vp, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_fwd_mega_stages": (
                [vp, vp, vp, i32, vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_routed_experts_fwd_rmsnorm": (
                [vp, vp, vp, i32, vp, vp, vp, i64, i32, i32, i32, i32, ctypes.c_float, vp, sz, vp], ctypes.c_int),
            "moe_fwd_dispatch": ([vp, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_fwd_gemm1": ([vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_fwd_gemm2": ([vp, i32, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_fwd_combine": ([vp, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_get_status": ([vp, ctypes.POINTER(ctypes.c_uint32), vp], ctypes.c_int),
            "moe_routing_static_scratch": ([vp, i64, i32, i32, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "moe_selftest_wait_timeout": ([ctypes.c_uint32, vp, vp], ctypes.c_int),
            "moe_bwd_workspace_bytes": ([i64, i32, i32, i32, i32], sz),
            "moe_routed_experts_bwd": (
                [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_bwd_stages": (
                [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, vp, sz, vp],
                ctypes.c_int),
            "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "moe_mxfp8_weight_bytes": ([i32, i32, i32, i32, vp, vp], ctypes.c_int),
            "moe_mxfp8_prepare_weight": ([i32, vp, i32, i32, i32, vp, sz, vp, sz, vp], ctypes.c_int),
            "moe_mxfp8_workspace_bytes": ([i64, i32, i32, i32, i32], sz),
            "moe_mxfp8_workspace_layout": ([i64, i32, i32, i32, i32, vp], ctypes.c_int),
            "moe_routed_experts_fwd_mxfp8": (
                [vp, vp, vp, i32, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
            "moe_nvfp4_weight_bytes": ([i32, i32, i32, i32, vp, vp], ctypes.c_int),
            "moe_nvfp4_prepare_weight": ([i32, vp, i32, i32, i32, vp, sz, vp, sz, vp], ctypes.c_int),
            "moe_nvfp4_workspace_bytes": ([i64, i32, i32, i32, i32], sz),
            "moe_nvfp4_workspace_layout": ([i64, i32, i32, i32, i32, vp], ctypes.c_int),
            "moe_fwd_nvfp4_stages": (
                [vp, vp, vp, i32, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, i64, i32, i32, i32, i32, i32,
                 i32, vp, sz, vp], ctypes.c_int),
            "moe_routed_experts_fwd_nvfp4": (
                [vp, vp, vp, i32, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, i64, i32, i32, i32, i32, vp, sz,
                 vp], ctypes.c_int),
            "moe_fwd_mxfp8_stages": (
                [vp, vp, vp, i32, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, vp, sz, vp], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoeError(fn, status, moe_status_string(status))


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_routing_outputs(counts, offsets, perm, inv, T: int, E: int, K: int):
    """int32 CUDA outputs of the routing calls, large enough for what the kernels write: counts [E],
    offsets [E+1], perm and inv [T*K]."""
    for name, t, n in (("counts", counts, E), ("offsets", offsets, E + 1), ("perm", perm, T * K),
                       ("inv", inv, T * K)):
        _need(t, name, torch.int32)
        if t.numel() < n:
            raise ValueError(f"{name} must hold at least {n} int32, got {t.numel()}")


def _need_status_word(t):
    """A caller-owned device status word: the library clears and ORs one whole uint32."""
    _need(t, "device_status", (torch.int32, torch.uint8))
    if t.numel() * t.element_size() < 4:
        raise ValueError(f"device_status must hold at least 4 bytes, got {t.numel() * t.element_size()}")
    if t.data_ptr() % 4:
        raise ValueError("device_status must be 4-byte aligned")


def _dims(x, topk_ids, w13):
    T, D = x.shape
    E, two, F, D2 = w13.shape
    if two != 2 or D2 != D:
        raise ValueError(f"w13 must be [E,2,F,D] with D={D}, got {tuple(w13.shape)}")
    if topk_ids.shape[0] != T:
        raise ValueError("topk_ids must be [T,K]")
    return T, D, F, E, topk_ids.shape[1]


# ----------------------------------------------------------------------------------- sizes

def moe_workspace_bytes(T: int, D: int, F: int, E: int, K: int) -> int:
    return int(load().moe_workspace_bytes(T, D, F, E, K))


def moe_workspace_layout(T: int, D: int, F: int, E: int, K: int) -> dict:
    arr = (ctypes.c_size_t * len(WS_REGIONS))()
    _check("moe_workspace_layout", load().moe_workspace_layout(T, D, F, E, K, ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(WS_REGIONS, (int(v) for v in arr)))


def moe_mega_workspace_bytes(T: int, D: int, F: int, E: int, K: int) -> int:
    return int(load().moe_mega_workspace_bytes(T, D, F, E, K))


def moe_mega_workspace_layout(T: int, D: int, F: int, E: int, K: int) -> dict:
    arr = (ctypes.c_size_t * len(WS_REGIONS))()
    _check("moe_mega_workspace_layout",
           load().moe_mega_workspace_layout(T, D, F, E, K, ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(WS_REGIONS, (int(v) for v in arr)))


def moe_routing_workspace_bytes(T: int, E: int, K: int) -> int:
    return int(load().moe_routing_workspace_bytes(T, E, K))


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A device byte buffer for the workspace (torch's allocator aligns it to 256 bytes or more)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------------------ entry points

def moe_routing(topk_ids, num_experts: int, counts, offsets, perm, inv, workspace, stream=None) -> None:
    _need(topk_ids, "topk_ids", torch.int32, 2)
    T, K = topk_ids.shape
    _need_routing_outputs(counts, offsets, perm, inv, T, int(num_experts), K)
    _need(workspace, "workspace", torch.uint8)
    _check("moe_routing", load().moe_routing(
        _ptr(topk_ids), T, int(num_experts), K, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
        _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_routed_experts_fwd(x, topk_ids, topk_scores, w13, w2, out, workspace, stream=None) -> None:
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(w13, "w13", torch.bfloat16, 4)
    _need(w2, "w2", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 2)
    _need(workspace, "workspace", torch.uint8)
    T, D, F, E, K = _dims(x, topk_ids, w13)
    if tuple(w2.shape) != (E, D, F) or tuple(out.shape) != (T, D) or tuple(topk_scores.shape) != (T, K):
        raise ValueError("inconsistent shapes among w2 [E,D,F], out [T,D], topk_scores [T,K]")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_routed_experts_fwd", load().moe_routed_experts_fwd(
        _ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13), _ptr(w2), _ptr(out),
        T, D, F, E, K, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_routed_experts_fwd_mega(x, topk_ids, topk_scores, w13, w2, out, workspace, stream=None) -> None:
    """The forward pass with both grouped GEMMs in one fused pipeline; the workspace is
    moe_mega_workspace_bytes(T, D, F, E, K) bytes. Bit-identical to moe_routed_experts_fwd."""
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(w13, "w13", torch.bfloat16, 4)
    _need(w2, "w2", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 2)
    _need(workspace, "workspace", torch.uint8)
    T, D, F, E, K = _dims(x, topk_ids, w13)
    if tuple(w2.shape) != (E, D, F) or tuple(out.shape) != (T, D) or tuple(topk_scores.shape) != (T, K):
        raise ValueError("inconsistent shapes among w2 [E,D,F], out [T,D], topk_scores [T,K]")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_routed_experts_fwd_mega", load().moe_routed_experts_fwd_mega(
        _ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13), _ptr(w2), _ptr(out),
        T, D, F, E, K, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


MEGA_STAGES = 3  # dispatch, both GEMMs in one grid, combine


def moe_fwd_mega_stages(x, topk_ids, topk_scores, w13, w2, out, workspace, stage_begin: int, stage_end: int,
                        stream=None) -> None:
    """Stages [stage_begin, stage_end) of moe_routed_experts_fwd_mega (MEGA_STAGES in all)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(w13, "w13", torch.bfloat16, 4)
    _need(w2, "w2", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 2)
    _need(workspace, "workspace", torch.uint8)
    T, D, F, E, K = _dims(x, topk_ids, w13)
    if tuple(w2.shape) != (E, D, F) or tuple(out.shape) != (T, D) or tuple(topk_scores.shape) != (T, K):
        raise ValueError("inconsistent shapes among w2 [E,D,F], out [T,D], topk_scores [T,K]")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_fwd_mega_stages", load().moe_fwd_mega_stages(
        _ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13), _ptr(w2), _ptr(out),
        T, D, F, E, K, int(stage_begin), int(stage_end), _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_routed_experts_fwd_rmsnorm(x, topk_ids, topk_scores, w13, w2, out, workspace, eps: float = 1e-6,
                                   stream=None) -> None:
    """The forward pass with route-wise RMSNorm of each expert output before the score weighting."""
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(w13, "w13", torch.bfloat16, 4)
    _need(w2, "w2", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 2)
    _need(workspace, "workspace", torch.uint8)
    T, D, F, E, K = _dims(x, topk_ids, w13)
    if tuple(w2.shape) != (E, D, F) or tuple(out.shape) != (T, D) or tuple(topk_scores.shape) != (T, K):
        raise ValueError("inconsistent shapes among w2 [E,D,F], out [T,D], topk_scores [T,K]")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_routed_experts_fwd_rmsnorm", load().moe_routed_experts_fwd_rmsnorm(
        _ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13), _ptr(w2), _ptr(out),
        T, D, F, E, K, float(eps), _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_fwd_dispatch(x, topk_ids, dims, workspace, stream=None) -> None:
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    T, D, F, E, K = dims
    _check("moe_fwd_dispatch", load().moe_fwd_dispatch(
        _ptr(x), _ptr(topk_ids), T, D, F, E, K, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_fwd_gemm1(w13, dims, workspace, stream=None) -> None:
    _need(w13, "w13", torch.bfloat16, 4)
    T, D, F, E, K = dims
    _check("moe_fwd_gemm1", load().moe_fwd_gemm1(
        _ptr(w13), T, D, F, E, K, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_fwd_gemm2(topk_scores, w2, dims, workspace, stream=None) -> None:
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(w2, "w2", torch.bfloat16, 3)
    T, D, F, E, K = dims
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_fwd_gemm2", load().moe_fwd_gemm2(
        _ptr(topk_scores), sd, _ptr(w2), T, D, F, E, K, _ptr(workspace), workspace.numel(),
        _stream_handle(stream)))


def moe_fwd_combine(topk_ids, out, dims, workspace, stream=None) -> None:
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(out, "out", torch.bfloat16, 2)
    T, D, F, E, K = dims
    _check("moe_fwd_combine", load().moe_fwd_combine(
        _ptr(topk_ids), _ptr(out), T, D, F, E, K, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_routing_static_scratch(topk_ids, num_experts: int, counts, offsets, perm, inv, device_status=None,
                               stream=None) -> None:
    """Routing without a workspace: its scratch is a fixed ~2 MiB array inside the library.

    For callers that cannot allocate device memory where they call the layer (an engine whose
    device memory is all owned by another allocator, a host program with no allocator at hand).
    The first call on a device looks up the array's address; make it before any stream capture.
    Calls share the array, so calls whose GPU work overlaps race: order them on one stream.
    """
    _need(topk_ids, "topk_ids", torch.int32, 2)
    T, K = topk_ids.shape
    _need_routing_outputs(counts, offsets, perm, inv, T, int(num_experts), K)
    if device_status is not None:
        _need_status_word(device_status)
    _check("moe_routing_static_scratch", load().moe_routing_static_scratch(
        _ptr(topk_ids), T, int(num_experts), K, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
        _ptr(device_status), _stream_handle(stream)))


def moe_bwd_workspace_bytes(T: int, D: int, F: int, E: int, K: int) -> int:
    return int(load().moe_bwd_workspace_bytes(T, D, F, E, K))


BWD_STAGES = 7  # dispatch, recompute, dgrad down, dgrad gate/up, wgrad down, wgrad gate/up, reduce
BWD_STAGE_NAMES = ("dispatch", "recompute", "dgrad_down", "dgrad_gate_up", "wgrad_down", "wgrad_gate_up", "reduce")


def moe_routed_experts_bwd(x, topk_ids, topk_scores, w13, w2, dout, dx, dscores, dw13, dw2, workspace,
                           stream=None) -> None:
    """Gradients of the layer: dx [T,D] bf16, dscores [T,K] fp32, dw13 [E,2,F,D] and dw2 [E,D,F] bf16."""
    args, dims = _bwd_args(x, topk_ids, topk_scores, w13, w2, dout, dx, dscores, dw13, dw2, workspace)
    _check("moe_routed_experts_bwd", load().moe_routed_experts_bwd(
        *args, *dims, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def moe_bwd_stages(x, topk_ids, topk_scores, w13, w2, dout, dx, dscores, dw13, dw2, workspace, stage_begin: int,
                   stage_end: int, stream=None) -> None:
    """Backward stages stage_begin .. stage_end-1 (BWD_STAGE_NAMES) on one workspace, in order."""
    args, dims = _bwd_args(x, topk_ids, topk_scores, w13, w2, dout, dx, dscores, dw13, dw2, workspace)
    _check("moe_bwd_stages", load().moe_bwd_stages(
        *args, *dims, int(stage_begin), int(stage_end), _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def _bwd_args(x, topk_ids, topk_scores, w13, w2, dout, dx, dscores, dw13, dw2, workspace):
    """Checked pointer arguments and (T, D, F, E, K) of the backward entry points."""
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(w13, "w13", torch.bfloat16, 4)
    _need(w2, "w2", torch.bfloat16, 3)
    _need(dout, "dout", torch.bfloat16, 2)
    _need(dx, "dx", torch.bfloat16, 2)
    _need(dscores, "dscores", torch.float32, 2)
    _need(dw13, "dw13", torch.bfloat16, 4)
    _need(dw2, "dw2", torch.bfloat16, 3)
    _need(workspace, "workspace", torch.uint8)
    T, D, F, E, K = _dims(x, topk_ids, w13)
    for name, t, shape in (("w2", w2, (E, D, F)), ("dout", dout, (T, D)), ("dx", dx, (T, D)),
                           ("dscores", dscores, (T, K)), ("dw13", dw13, (E, 2, F, D)), ("dw2", dw2, (E, D, F)),
                           ("topk_scores", topk_scores, (T, K))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {shape}, got {tuple(t.shape)}")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    return ((_ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13), _ptr(w2), _ptr(dout), _ptr(dx),
             _ptr(dscores), _ptr(dw13), _ptr(dw2)), (T, D, F, E, K))


def moe_selftest_wait_timeout(timeout_us: int, device_status, stream=None) -> None:
    """Runs a kernel whose bounded wait must run out; device_status receives MOE_DEV_TIMEOUT."""
    _need_status_word(device_status)
    _check("moe_selftest_wait_timeout", load().moe_selftest_wait_timeout(
        int(timeout_us), _ptr(device_status), _stream_handle(stream)))


def moe_get_status(workspace, stream=None) -> int:
    """The device status bits of a workspace (synchronises the stream)."""
    _need(workspace, "workspace", torch.uint8)
    bits = ctypes.c_uint32(0)
    _check("moe_get_status", load().moe_get_status(_ptr(workspace), ctypes.byref(bits), _stream_handle(stream)))
    return int(bits.value)


# ------------------------------------------------------------------------------------- MXFP8

def moe_mxfp8_weight_bytes(which: int, D: int, F: int, E: int) -> tuple[int, int]:
    """(data bytes, scale bytes) of a prepared MXFP8 weight (which = MOE_WEIGHT_W13 or _W2)."""
    data, scales = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("moe_mxfp8_weight_bytes", load().moe_mxfp8_weight_bytes(
        int(which), D, F, E, ctypes.byref(data), ctypes.byref(scales)))
    return int(data.value), int(scales.value)


def moe_mxfp8_prepare_weight(which: int, w, data=None, scales=None, stream=None):
    """Quantizes w13 [E,2,F,D] (which = MOE_WEIGHT_W13) or w2 [E,D,F] (MOE_WEIGHT_W2) to MXFP8.

    Returns (data, scales): uint8 device tensors of E4M3 codes (w's element order) and UE8M0
    scales (grouped per GEMM tile); pass them to preallocate.
    """
    _need(w, "w", torch.bfloat16)
    if which == MOE_WEIGHT_W13:
        if w.dim() != 4 or w.shape[1] != 2:
            raise ValueError(f"w13 must be [E,2,F,D], got {tuple(w.shape)}")
        E, _, F, D = w.shape
    elif which == MOE_WEIGHT_W2:
        if w.dim() != 3:
            raise ValueError(f"w2 must be [E,D,F], got {tuple(w.shape)}")
        E, D, F = w.shape
    else:
        raise ValueError("which must be MOE_WEIGHT_W13 or MOE_WEIGHT_W2")
    nd, ns = moe_mxfp8_weight_bytes(which, D, F, E)
    if data is None:
        data = torch.empty(nd, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(ns, dtype=torch.uint8, device=w.device)
    _need(data, "data", torch.uint8)
    _need(scales, "scales", torch.uint8)
    _check("moe_mxfp8_prepare_weight", load().moe_mxfp8_prepare_weight(
        int(which), _ptr(w), D, F, E, _ptr(data), data.numel(), _ptr(scales), scales.numel(),
        _stream_handle(stream)))
    return data, scales


def moe_mxfp8_workspace_bytes(T: int, D: int, F: int, E: int, K: int) -> int:
    return int(load().moe_mxfp8_workspace_bytes(T, D, F, E, K))


def moe_mxfp8_workspace_layout(T: int, D: int, F: int, E: int, K: int) -> dict:
    arr = (ctypes.c_size_t * len(MXWS_REGIONS))()
    _check("moe_mxfp8_workspace_layout",
           load().moe_mxfp8_workspace_layout(T, D, F, E, K, ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(MXWS_REGIONS, (int(v) for v in arr)))


MX_STAGES = 4


def moe_routed_experts_fwd_mxfp8(x, topk_ids, topk_scores, w13_mx, w2_mx, out, workspace, dims_FE=None,
                                 stream=None) -> None:
    """The MXFP8 forward. w13_mx, w2_mx: (data, scales) from moe_mxfp8_prepare_weight.

    dims_FE = (F, E); the prepared weights are flat byte tensors, so F and E come from here.
    """
    moe_fwd_mxfp8_stages(x, topk_ids, topk_scores, w13_mx, w2_mx, out, workspace, dims_FE, 0, MX_STAGES, stream)


def moe_fwd_mxfp8_stages(x, topk_ids, topk_scores, w13_mx, w2_mx, out, workspace, dims_FE, stage_begin: int,
                         stage_end: int, stream=None) -> None:
    """Stages [stage_begin, stage_end) of the MXFP8 forward (0 dispatch, 1 gate/up, 2 down, 3 combine)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(out, "out", torch.bfloat16, 2)
    _need(workspace, "workspace", torch.uint8)
    for name, t in (("w13 data", w13_mx[0]), ("w13 scales", w13_mx[1]), ("w2 data", w2_mx[0]),
                    ("w2 scales", w2_mx[1])):
        _need(t, name, torch.uint8)
    if dims_FE is None:
        raise ValueError("dims_FE = (F, E) is required")
    T, D = x.shape
    K = topk_ids.shape[1]
    F, E = (int(v) for v in dims_FE)
    if tuple(out.shape) != (T, D) or tuple(topk_scores.shape) != (T, K) or topk_ids.shape[0] != T:
        raise ValueError("inconsistent shapes among x [T,D], topk_ids/topk_scores [T,K], out [T,D]")
    for which, (d, sc) in ((MOE_WEIGHT_W13, w13_mx), (MOE_WEIGHT_W2, w2_mx)):
        nd, ns = moe_mxfp8_weight_bytes(which, D, F, E)
        if d.numel() < nd or sc.numel() < ns:
            raise ValueError("prepared weight buffers are smaller than moe_mxfp8_weight_bytes")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_fwd_mxfp8_stages", load().moe_fwd_mxfp8_stages(
        _ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13_mx[0]), _ptr(w13_mx[1]), _ptr(w2_mx[0]),
        _ptr(w2_mx[1]), _ptr(out), T, D, F, E, K, int(stage_begin), int(stage_end), _ptr(workspace),
        workspace.numel(), _stream_handle(stream)))


# ------------------------------------------------------------------------------------- NVFP4

def moe_nvfp4_weight_bytes(which: int, D: int, F: int, E: int) -> tuple[int, int]:
    """(data bytes, scale bytes) of a prepared NVFP4 weight (which = MOE_WEIGHT_W13 or _W2)."""
    data, scales = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("moe_nvfp4_weight_bytes", load().moe_nvfp4_weight_bytes(
        int(which), D, F, E, ctypes.byref(data), ctypes.byref(scales)))
    return int(data.value), int(scales.value)


def moe_nvfp4_prepare_weight(which: int, w, data=None, scales=None, stream=None):
    """Quantizes w13 [E,2,F,D] or w2 [E,D,F] to NVFP4. Returns (data, scales) uint8 device tensors:
    packed E2M1 codes, and a 256-byte header holding the tensor scale followed by the UE4M3 scales."""
    _need(w, "w", torch.bfloat16)
    if which == MOE_WEIGHT_W13:
        if w.dim() != 4 or w.shape[1] != 2:
            raise ValueError(f"w13 must be [E,2,F,D], got {tuple(w.shape)}")
        E, _, F, D = w.shape
    elif which == MOE_WEIGHT_W2:
        if w.dim() != 3:
            raise ValueError(f"w2 must be [E,D,F], got {tuple(w.shape)}")
        E, D, F = w.shape
    else:
        raise ValueError("which must be MOE_WEIGHT_W13 or MOE_WEIGHT_W2")
    nd, ns = moe_nvfp4_weight_bytes(which, D, F, E)
    if data is None:
        data = torch.empty(nd, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(ns, dtype=torch.uint8, device=w.device)
    _need(data, "data", torch.uint8)
    _need(scales, "scales", torch.uint8)
    _check("moe_nvfp4_prepare_weight", load().moe_nvfp4_prepare_weight(
        int(which), _ptr(w), D, F, E, _ptr(data), data.numel(), _ptr(scales), scales.numel(), _stream_handle(stream)))
    return data, scales


def moe_nvfp4_workspace_bytes(T: int, D: int, F: int, E: int, K: int) -> int:
    return int(load().moe_nvfp4_workspace_bytes(T, D, F, E, K))


def moe_nvfp4_workspace_layout(T: int, D: int, F: int, E: int, K: int) -> dict:
    arr = (ctypes.c_size_t * len(MXWS_REGIONS))()
    _check("moe_nvfp4_workspace_layout",
           load().moe_nvfp4_workspace_layout(T, D, F, E, K, ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(MXWS_REGIONS, (int(v) for v in arr)))


def moe_routed_experts_fwd_nvfp4(x, topk_ids, topk_scores, w13_nv, w2_nv, out, workspace, dims_FE, x_scale: float,
                                 h_scale: float, stream=None) -> None:
    """The NVFP4 forward. w13_nv, w2_nv: (data, scales) from moe_nvfp4_prepare_weight; dims_FE = (F, E);
    x_scale, h_scale: the activations' tensor scales (calibration constants)."""
    moe_fwd_nvfp4_stages(x, topk_ids, topk_scores, w13_nv, w2_nv, out, workspace, dims_FE, x_scale, h_scale, 0,
                         MX_STAGES, stream)


def moe_fwd_nvfp4_stages(x, topk_ids, topk_scores, w13_nv, w2_nv, out, workspace, dims_FE, x_scale: float,
                         h_scale: float, stage_begin: int, stage_end: int, stream=None) -> None:
    """Stages [stage_begin, stage_end) of the NVFP4 forward (0 dispatch, 1 gate/up, 2 down, 3 combine)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(topk_scores, "topk_scores", (torch.float32, torch.bfloat16), 2)
    _need(out, "out", torch.bfloat16, 2)
    _need(workspace, "workspace", torch.uint8)
    for name, t in (("w13 data", w13_nv[0]), ("w13 scales", w13_nv[1]), ("w2 data", w2_nv[0]),
                    ("w2 scales", w2_nv[1])):
        _need(t, name, torch.uint8)
    T, D = x.shape
    K = topk_ids.shape[1]
    F, E = (int(v) for v in dims_FE)
    if tuple(out.shape) != (T, D) or tuple(topk_scores.shape) != (T, K) or topk_ids.shape[0] != T:
        raise ValueError("inconsistent shapes among x [T,D], topk_ids/topk_scores [T,K], out [T,D]")
    for which, (d, sc) in ((MOE_WEIGHT_W13, w13_nv), (MOE_WEIGHT_W2, w2_nv)):
        nd, ns = moe_nvfp4_weight_bytes(which, D, F, E)
        if d.numel() < nd or sc.numel() < ns:
            raise ValueError("prepared weight buffers are smaller than moe_nvfp4_weight_bytes")
    sd = MOE_SCORES_BF16 if topk_scores.dtype == torch.bfloat16 else MOE_SCORES_F32
    _check("moe_fwd_nvfp4_stages", load().moe_fwd_nvfp4_stages(
        _ptr(x), _ptr(topk_ids), _ptr(topk_scores), sd, _ptr(w13_nv[0]), _ptr(w13_nv[1]), _ptr(w2_nv[0]),
        _ptr(w2_nv[1]), float(x_scale), float(h_scale), _ptr(out), T, D, F, E, K, int(stage_begin),
        int(stage_end), _ptr(workspace), workspace.numel(), _stream_handle(stream)))
