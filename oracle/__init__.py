"""CPU oracle for the routed top-k expert layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import this package. The product path (the CUDA library and its Python
binding) never imports it, and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (a plain per-token fp32 loop over bf16 inputs and a
stable counting sort); this module compiles it with gcc and marshals numpy arrays to it. bf16
tensors cross this boundary as their raw 16-bit patterns (``numpy.uint16``).

Every function here is pinned by ``tests/test_oracle_pins.py`` against brute force, closed forms
and invariants, and ``tests/test_oracle_mutants.py`` checks that the pins catch planted mistakes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(_BUILD_DIR, "libmoe_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-Wall"]

_lock = threading.Lock()
_lib = None


def compile_oracle(source: str, output: str) -> None:
    """gcc the oracle source into a shared library (also used on patched copies by the tests)."""
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, output)


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its source. Returns the library path."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, LIBRARY)
    return LIBRARY


def load_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    lib.oracle_routing.argtypes = [p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, p, p, p, p]
    lib.oracle_routing.restype = ctypes.c_long
    lib.oracle_routed_experts.argtypes = [
        p, p, p, ctypes.c_int, p, p, p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int, ctypes.c_int,
    ]
    lib.oracle_routed_experts.restype = ctypes.c_int
    lib.oracle_routed_experts_rmsnorm.argtypes = [
        p, p, p, ctypes.c_int, p, p, p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_float, ctypes.c_int,
    ]
    lib.oracle_routed_experts_rmsnorm.restype = ctypes.c_int
    lib.oracle_routed_experts_bwd.argtypes = [
        p, p, p, ctypes.c_int, p, p, p, p, p, p, p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
    ]
    lib.oracle_routed_experts_bwd.restype = ctypes.c_int
    lib.oracle_mx_quantize_rows.argtypes = [p, ctypes.c_int64, ctypes.c_int32, p, p]
    lib.oracle_mx_quantize_rows.restype = ctypes.c_int
    lib.oracle_routed_experts_mxfp8.argtypes = [
        p, p, p, ctypes.c_int, p, p, p, p, p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
    ]
    lib.oracle_routed_experts_mxfp8.restype = ctypes.c_int
    lib.oracle_nvfp4_weight_scale.argtypes = [p, ctypes.c_int64]
    lib.oracle_nvfp4_weight_scale.restype = ctypes.c_float
    lib.oracle_nvfp4_quantize_rows.argtypes = [p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, p, p]
    lib.oracle_nvfp4_quantize_rows.restype = ctypes.c_int
    lib.oracle_routed_experts_nvfp4.argtypes = [
        p, p, p, ctypes.c_int, p, p, ctypes.c_float, p, p, ctypes.c_float, ctypes.c_float, ctypes.c_float, p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
    ]
    lib.oracle_routed_experts_nvfp4.restype = ctypes.c_int
    return lib


def _library(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def routing(topk_ids: np.ndarray, num_experts: int, lib=None) -> dict:
    """Expert counts, offsets and the stable permutation of the T*K (token, k) pairs.

    Returns ``counts[E]``, ``offsets[E+1]``, ``perm[T*K]`` (row -> flat pair t*K+k),
    ``inv[T*K]`` (flat pair -> row), all int32, and ``n_invalid`` (ids outside [0, E)).
    """
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    if ids.ndim != 2:
        raise ValueError("topk_ids must be [T, K]")
    T, K = ids.shape
    E = int(num_experts)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * K, np.int32)
    inv = np.zeros(T * K, np.int32)
    n_invalid = _library(lib).oracle_routing(
        _ptr(ids), T, E, K, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv)
    )
    if n_invalid < 0:
        raise ValueError("oracle_routing rejected its arguments")
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv, "n_invalid": int(n_invalid)}


def routed_experts(x_bits, topk_ids, topk_scores, w13_bits, w2_bits, round_h: bool = False,
                   nthreads: int | None = None, lib=None) -> np.ndarray:
    """The layer's output ``out[T,D]`` in fp32.

    ``x_bits`` [T,D], ``w13_bits`` [E,2,F,D] and ``w2_bits`` [E,D,F] are bf16 bit patterns
    (uint16). ``topk_ids`` [T,K] int32. ``topk_scores`` [T,K] float32, or uint16 bf16 bits.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w13 = np.ascontiguousarray(w13_bits, dtype=np.uint16)
    w2 = np.ascontiguousarray(w2_bits, dtype=np.uint16)
    sc = np.asarray(topk_scores)
    scores_bf16 = 1 if sc.dtype == np.uint16 else 0
    sc = np.ascontiguousarray(sc, dtype=np.uint16 if scores_bf16 else np.float32)
    T, D = x.shape
    E, two, F, D2 = w13.shape
    if two != 2 or D2 != D or w2.shape != (E, D, F) or ids.shape[0] != T or sc.shape != ids.shape:
        raise ValueError("inconsistent shapes")
    K = ids.shape[1]
    out = np.zeros((T, D), np.float32)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _library(lib).oracle_routed_experts(
        _ptr(x), _ptr(ids), _ptr(sc), scores_bf16, _ptr(w13), _ptr(w2), _ptr(out),
        T, D, F, E, K, 1 if round_h else 0, int(nthreads),
    )
    if rc != 0:
        raise RuntimeError("oracle_routed_experts failed")
    return out


def routed_experts_rmsnorm(x_bits, topk_ids, topk_scores, w13_bits, w2_bits, eps: float,
                           nthreads: int | None = None, lib=None) -> np.ndarray:
    """out[T,D] (fp32) with route-wise RMSNorm of each expert output before the score weighting."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w13 = np.ascontiguousarray(w13_bits, dtype=np.uint16)
    w2 = np.ascontiguousarray(w2_bits, dtype=np.uint16)
    sc = np.asarray(topk_scores)
    scores_bf16 = 1 if sc.dtype == np.uint16 else 0
    sc = np.ascontiguousarray(sc, dtype=np.uint16 if scores_bf16 else np.float32)
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    out = np.zeros((T, D), np.float32)
    rc = _library(lib).oracle_routed_experts_rmsnorm(
        _ptr(x), _ptr(ids), _ptr(sc), scores_bf16, _ptr(w13), _ptr(w2), _ptr(out),
        T, D, F, E, K, float(eps), int(nthreads or os.cpu_count() or 1),
    )
    if rc != 0:
        raise RuntimeError("oracle_routed_experts_rmsnorm failed")
    return out


def routed_experts_bwd(x_bits, topk_ids, topk_scores, w13_bits, w2_bits, dout, nthreads: int | None = None,
                       lib=None) -> dict:
    """Gradients of the layer for the upstream gradient ``dout`` [T,D] (float32).

    Returns fp32 ``dx`` [T,D], ``dscores`` [T,K], ``dw13`` [E,2,F,D] and ``dw2`` [E,D,F].
    Inputs as for :func:`routed_experts`.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w13 = np.ascontiguousarray(w13_bits, dtype=np.uint16)
    w2 = np.ascontiguousarray(w2_bits, dtype=np.uint16)
    go = np.ascontiguousarray(dout, dtype=np.float32)
    sc = np.asarray(topk_scores)
    scores_bf16 = 1 if sc.dtype == np.uint16 else 0
    sc = np.ascontiguousarray(sc, dtype=np.uint16 if scores_bf16 else np.float32)
    T, D = x.shape
    E, two, F, _ = w13.shape
    K = ids.shape[1]
    if two != 2 or w2.shape != (E, D, F) or go.shape != (T, D) or sc.shape != ids.shape:
        raise ValueError("inconsistent shapes")
    out = {
        "dx": np.zeros((T, D), np.float32),
        "dscores": np.zeros((T, K), np.float32),
        "dw13": np.zeros((E, 2, F, D), np.float32),
        "dw2": np.zeros((E, D, F), np.float32),
    }
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _library(lib).oracle_routed_experts_bwd(
        _ptr(x), _ptr(ids), _ptr(sc), scores_bf16, _ptr(w13), _ptr(w2), _ptr(go),
        _ptr(out["dx"]), _ptr(out["dscores"]), _ptr(out["dw13"]), _ptr(out["dw2"]),
        T, D, F, E, K, int(nthreads),
    )
    if rc != 0:
        raise RuntimeError("oracle_routed_experts_bwd failed")
    return out


def mx_quantize_rows(bits, lib=None):
    """MX (E4M3 elements, UE8M0 scales, blocks of 32 along the last axis) quantization of bf16 bits.

    ``bits`` is a uint16 array ``[..., cols]`` with ``cols % 32 == 0``. Returns ``(codes, scales)``:
    uint8 E4M3 codes of the same shape and uint8 UE8M0 scale codes ``[..., cols // 32]``.
    """
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    cols = a.shape[-1]
    rows = a.size // cols if cols else 0
    codes = np.zeros(a.shape, np.uint8)
    scales = np.zeros(a.shape[:-1] + (cols // 32,), np.uint8)
    if _library(lib).oracle_mx_quantize_rows(_ptr(a), rows, cols, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle_mx_quantize_rows rejected its arguments")
    return codes, scales


def e4m3_values(codes) -> np.ndarray:
    """float64 values of E4M3 codes (the format's definition; 0x7F / 0xFF, NaN, never occur)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    ex = (c >> 3) & 15
    man = c & 7
    mag = np.where(ex == 0, np.ldexp(man.astype(np.float64), -9),
                   np.ldexp((8 + man).astype(np.float64), ex - 10))
    return sign * mag


def mx_dequantize(codes, scales) -> np.ndarray:
    """float64 values of an MX-quantized array: value(code) * 2^(scale - 127) per block of 32."""
    v = e4m3_values(codes)
    e = np.repeat(np.asarray(scales, dtype=np.int64) - 127, 32, axis=-1)
    return np.ldexp(v, e)


def routed_experts_mxfp8(x_bits, topk_ids, topk_scores, w13_mx, w2_mx, nthreads: int | None = None,
                         lib=None) -> np.ndarray:
    """out[T,D] (fp32) of the MXFP8 forward.

    ``x_bits`` [T,D] bf16 bits (quantized here, per token row); ``w13_mx`` = (codes [E,2,F,D],
    scales [E,2,F,D/32]) and ``w2_mx`` = (codes [E,D,F], scales [E,D,F/32]) as returned by
    :func:`mx_quantize_rows` on the bf16 weights. ids and scores as for :func:`routed_experts`.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w13q, w13s = (np.ascontiguousarray(a, dtype=np.uint8) for a in w13_mx)
    w2q, w2s = (np.ascontiguousarray(a, dtype=np.uint8) for a in w2_mx)
    sc = np.asarray(topk_scores)
    scores_bf16 = 1 if sc.dtype == np.uint16 else 0
    sc = np.ascontiguousarray(sc, dtype=np.uint16 if scores_bf16 else np.float32)
    T, D = x.shape
    E, two, F, D2 = w13q.shape
    K = ids.shape[1]
    if (two != 2 or D2 != D or w13s.shape != (E, 2, F, D // 32) or w2q.shape != (E, D, F)
            or w2s.shape != (E, D, F // 32) or ids.shape[0] != T or sc.shape != ids.shape):
        raise ValueError("inconsistent shapes")
    out = np.zeros((T, D), np.float32)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _library(lib).oracle_routed_experts_mxfp8(
        _ptr(x), _ptr(ids), _ptr(sc), scores_bf16, _ptr(w13q), _ptr(w13s), _ptr(w2q), _ptr(w2s), _ptr(out),
        T, D, F, E, K, int(nthreads),
    )
    if rc != 0:
        raise RuntimeError("oracle_routed_experts_mxfp8 failed")
    return out


def nvfp4_weight_scale(bits, lib=None) -> float:
    """The tensor scale G of a bf16 weight: amax / 2688 in fp32 (1 for an all-zero tensor)."""
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    return float(_library(lib).oracle_nvfp4_weight_scale(_ptr(a), a.size))


def nvfp4_quantize_rows(bits, G: float, lib=None):
    """NVFP4 quantization of bf16 bits ``[..., cols]`` (cols % 16 == 0) with tensor scale G.

    Returns ``(codes, scales)``: uint8 E2M1 codes (one per byte, low 4 bits) of the same shape and
    uint8 UE4M3 scale codes ``[..., cols // 16]``.
    """
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    cols = a.shape[-1]
    rows = a.size // cols if cols else 0
    codes = np.zeros(a.shape, np.uint8)
    scales = np.zeros(a.shape[:-1] + (cols // 16,), np.uint8)
    if _library(lib).oracle_nvfp4_quantize_rows(_ptr(a), rows, cols, float(G), _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle_nvfp4_quantize_rows rejected its arguments")
    return codes, scales


def nvfp4_prepare(bits, lib=None):
    """(codes, scales, G) of a bf16 weight with its own tensor scale."""
    G = nvfp4_weight_scale(bits, lib=lib)
    codes, scales = nvfp4_quantize_rows(bits, G, lib=lib)
    return codes, scales, G


def routed_experts_nvfp4(x_bits, topk_ids, topk_scores, w13_nv, w2_nv, gx: float, gh: float,
                         nthreads: int | None = None, lib=None) -> np.ndarray:
    """out[T,D] (fp32) of the NVFP4 forward. w13_nv = (codes [E,2,F,D], scales [E,2,F,D/16], G),
    w2_nv = (codes [E,D,F], scales [E,D,F/16], G) from :func:`nvfp4_prepare`; gx and gh are the
    activation tensor scales of x and of the SwiGLU output."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w13q, w13s = (np.ascontiguousarray(a, dtype=np.uint8) for a in w13_nv[:2])
    w2q, w2s = (np.ascontiguousarray(a, dtype=np.uint8) for a in w2_nv[:2])
    sc = np.asarray(topk_scores)
    scores_bf16 = 1 if sc.dtype == np.uint16 else 0
    sc = np.ascontiguousarray(sc, dtype=np.uint16 if scores_bf16 else np.float32)
    T, D = x.shape
    E, two, F, D2 = w13q.shape
    K = ids.shape[1]
    if (two != 2 or D2 != D or w13s.shape != (E, 2, F, D // 16) or w2q.shape != (E, D, F)
            or w2s.shape != (E, D, F // 16) or ids.shape[0] != T or sc.shape != ids.shape):
        raise ValueError("inconsistent shapes")
    out = np.zeros((T, D), np.float32)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _library(lib).oracle_routed_experts_nvfp4(
        _ptr(x), _ptr(ids), _ptr(sc), scores_bf16, _ptr(w13q), _ptr(w13s), float(w13_nv[2]), _ptr(w2q), _ptr(w2s),
        float(w2_nv[2]), float(gx), float(gh), _ptr(out), T, D, F, E, K, int(nthreads),
    )
    if rc != 0:
        raise RuntimeError("oracle_routed_experts_nvfp4 failed")
    return out
