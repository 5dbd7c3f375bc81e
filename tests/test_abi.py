"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol, and rejects
bad arguments on the host before touching CUDA. Workspace layout arithmetic."""

import ctypes
import functools
import os
import re

import pytest

from mixture_experts_routed_topk_gb300 import binding, build

HEADER = os.path.join(build.INCLUDE, "moe_routed_experts.h")

OK, INVALID, SHAPE, MISALIGNED, WS_SMALL = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_workspace_bytes", "moe_routed_experts_fwd", "moe_routing", "moe_get_status",
                     "moe_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(7):
        s = binding.moe_status_string(code)
        assert s.startswith("MOE_")
    assert "unknown" in binding.moe_status_string(99)


FAKE = 1 << 20  # a 256-byte-aligned non-null address; never dereferenced (host checks fail first)


def fwd(lib, entry="moe_routed_experts_fwd", **kw):
    a = dict(x=FAKE, ids=FAKE, scores=FAKE, sd=0, w13=FAKE, w2=FAKE, out=FAKE,
             T=16, D=256, F=256, E=8, K=2, ws=FAKE, wsb=1 << 40)
    a.update(kw)
    v = ctypes.c_void_p
    return getattr(lib, entry)(v(a["x"]), v(a["ids"]), v(a["scores"]), a["sd"], v(a["w13"]), v(a["w2"]),
                               v(a["out"]), a["T"], a["D"], a["F"], a["E"], a["K"], v(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("entry", ["moe_routed_experts_fwd", "moe_routed_experts_fwd_mega"])
def test_host_validation_needs_no_gpu(lib, entry):
    fwd = functools.partial(globals()["fwd"], entry=entry)
    assert fwd(lib, T=0) == OK  # nothing to do
    assert fwd(lib, T=-1) == INVALID
    assert fwd(lib, E=0) == INVALID
    assert fwd(lib, K=0) == INVALID
    assert fwd(lib, D=0) == INVALID
    assert fwd(lib, sd=7) == INVALID
    assert fwd(lib, x=0) == INVALID
    assert fwd(lib, out=0) == INVALID
    assert fwd(lib, ws=0) == INVALID
    assert fwd(lib, D=200) == SHAPE
    assert fwd(lib, F=96) == SHAPE
    assert fwd(lib, E=4097) == SHAPE
    assert fwd(lib, T=1 << 29, K=8) == SHAPE
    assert fwd(lib, x=FAKE + 8) == MISALIGNED
    assert fwd(lib, w2=FAKE + 4) == MISALIGNED
    assert fwd(lib, ids=FAKE + 2) == MISALIGNED
    assert fwd(lib, ws=FAKE + 16) == MISALIGNED
    need = (binding.moe_mega_workspace_bytes if entry.endswith("mega") else binding.moe_workspace_bytes)(
        16, 256, 256, 8, 2)
    assert fwd(lib, wsb=need - 1) == WS_SMALL


def test_mega_stage_range_validation(lib):
    v = ctypes.c_void_p
    call = lambda b, e, **kw: lib.moe_fwd_mega_stages(
        v(FAKE), v(FAKE), v(FAKE), 0, v(FAKE), v(FAKE), v(kw.get("out", FAKE)), 16, 256, 256, 8, 2, b, e,
        v(FAKE), kw.get("wsb", 1 << 40), None)
    assert call(-1, 2) == INVALID
    assert call(0, 4) == INVALID
    assert call(2, 1) == INVALID
    assert call(1, 1) == OK  # an empty range does nothing
    assert call(2, 3, out=0) == INVALID  # the combine stage needs out
    assert call(2, 3, out=FAKE + 8) == MISALIGNED
    assert call(0, 3, wsb=binding.moe_workspace_bytes(16, 256, 256, 8, 2)) == WS_SMALL  # the staged size is short


def test_routing_host_validation(lib):
    v = ctypes.c_void_p
    r = lambda **kw: lib.moe_routing(v(kw.get("ids", FAKE)), kw.get("T", 4), kw.get("E", 4), kw.get("K", 2),
                                     v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(kw.get("ws", FAKE)),
                                     kw.get("wsb", 1 << 30), None)
    assert r(T=0) == OK
    assert r(ids=0) == INVALID
    assert r(E=0) == INVALID
    assert r(ids=FAKE + 1) == MISALIGNED
    assert r(wsb=16) == WS_SMALL


@pytest.mark.parametrize("dims", [(16, 256, 256, 8, 2), (4096, 2048, 1408, 64, 6), (64, 7168, 2048, 256, 8),
                                  (16384, 7168, 2048, 256, 8), (1, 64, 64, 1, 1), (3, 64, 128, 4096, 7)])
def test_workspace_layout(lib, dims):
    T, D, F, E, K = dims
    lay = binding.moe_workspace_layout(*dims)
    R = T * K
    sizes = {"status": 4, "counts": 4 * E, "offsets": 4 * (E + 1), "tiles1": 4 * (E + 1), "tiles2": 4 * (E + 1),
             "perm": 4 * R, "inv": 4 * R, "xp": 2 * R * D, "h": 2 * R * F,
             "rms": 4 * R * ((D + 255) // 256)}
    names = list(binding.WS_REGIONS)
    for i, name in enumerate(names[:-1]):
        assert lay[name] % 256 == 0
        nxt = lay[names[i + 1]]
        if name in sizes:
            assert nxt - lay[name] >= sizes[name], name
    assert lay["status"] == 0
    assert lay["total"] == binding.moe_workspace_bytes(*dims)
    assert binding.moe_routing_workspace_bytes(T, E, K) < lay["total"]
    # the staged layout leaves the fused forward's regions empty
    assert lay["ready"] == lay["y"] == lay["total"]


@pytest.mark.parametrize("dims", [(16, 256, 256, 8, 2), (4096, 2048, 1408, 64, 6), (64, 7168, 2048, 256, 8),
                                  (1, 64, 64, 1, 1), (3, 64, 128, 4096, 7)])
def test_mega_workspace_layout(lib, dims):
    T, D, F, E, K = dims
    staged = binding.moe_workspace_layout(*dims)
    lay = binding.moe_mega_workspace_layout(*dims)
    R = T * K
    names = list(binding.WS_REGIONS)
    for name in names[: names.index("ready")]:
        assert lay[name] == staged[name], name  # the staged regions, at the same offsets
    row_tiles = -(-R // 128) + min(R, E)
    assert lay["y"] - lay["ready"] >= 4 * (32 + row_tiles)
    assert lay["total"] - lay["y"] >= 2 * R * D
    assert lay["y"] >= lay["xp"] + 2 * R * D  # Y never overlaps XP
    assert lay["total"] == binding.moe_mega_workspace_bytes(*dims)
    assert binding.moe_mega_workspace_bytes(0, D, F, E, K) == 0


def bwd(lib, **kw):
    a = dict(x=FAKE, ids=FAKE, scores=FAKE, sd=0, w13=FAKE, w2=FAKE, dout=FAKE, dx=FAKE, dsc=FAKE, dw13=FAKE,
             dw2=FAKE, T=16, D=256, F=256, E=8, K=2, ws=FAKE, wsb=1 << 40)
    a.update(kw)
    v = ctypes.c_void_p
    return lib.moe_routed_experts_bwd(v(a["x"]), v(a["ids"]), v(a["scores"]), a["sd"], v(a["w13"]), v(a["w2"]),
                                      v(a["dout"]), v(a["dx"]), v(a["dsc"]), v(a["dw13"]), v(a["dw2"]), a["T"],
                                      a["D"], a["F"], a["E"], a["K"], v(a["ws"]), a["wsb"], None)


def test_bwd_host_validation_needs_no_gpu(lib):
    assert bwd(lib, T=-1) == INVALID
    assert bwd(lib, sd=3) == INVALID
    assert bwd(lib, dw2=0) == INVALID
    assert bwd(lib, dout=0) == INVALID
    assert bwd(lib, ws=0) == INVALID
    assert bwd(lib, D=96) == SHAPE
    assert bwd(lib, E=5000) == SHAPE
    assert bwd(lib, dx=FAKE + 8) == MISALIGNED
    assert bwd(lib, dw13=FAKE + 2) == MISALIGNED
    assert bwd(lib, dsc=FAKE + 2) == MISALIGNED
    need = binding.moe_bwd_workspace_bytes(16, 256, 256, 8, 2)
    assert need > binding.moe_workspace_bytes(16, 256, 256, 8, 2)
    assert bwd(lib, wsb=need - 1) == WS_SMALL
    assert binding.moe_bwd_workspace_bytes(0, 256, 256, 8, 2) == 0


def test_binding_region_list_matches_header():
    text = open(HEADER).read()
    n = int(re.search(r"MOE_WS_REGIONS\s*=\s*(\d+)", text).group(1))
    assert len(binding.WS_REGIONS) == n


def mx_fwd(lib, **kw):
    a = dict(x=FAKE, ids=FAKE, scores=FAKE, sd=0, w13q=FAKE, w13s=FAKE, w2q=FAKE, w2s=FAKE, out=FAKE,
             T=16, D=256, F=256, E=8, K=2, ws=FAKE, wsb=1 << 40)
    a.update(kw)
    v = ctypes.c_void_p
    return lib.moe_routed_experts_fwd_mxfp8(
        v(a["x"]), v(a["ids"]), v(a["scores"]), a["sd"], v(a["w13q"]), v(a["w13s"]), v(a["w2q"]), v(a["w2s"]),
        v(a["out"]), a["T"], a["D"], a["F"], a["E"], a["K"], v(a["ws"]), a["wsb"], None)


def test_mxfp8_host_validation_needs_no_gpu(lib):
    assert mx_fwd(lib, T=0) == OK
    assert mx_fwd(lib, T=-1) == INVALID
    assert mx_fwd(lib, sd=2) == INVALID
    assert mx_fwd(lib, w13s=0) == INVALID
    assert mx_fwd(lib, w2q=0) == INVALID
    assert mx_fwd(lib, D=192) == SHAPE  # a multiple of 64 but not of 128
    assert mx_fwd(lib, F=320) == SHAPE
    assert mx_fwd(lib, E=4097) == SHAPE
    assert mx_fwd(lib, w13s=FAKE + 16) == MISALIGNED  # scales must be 256-byte aligned
    assert mx_fwd(lib, w2q=FAKE + 8) == MISALIGNED
    assert mx_fwd(lib, ws=FAKE + 64) == MISALIGNED
    need = binding.moe_mxfp8_workspace_bytes(16, 256, 256, 8, 2)
    assert mx_fwd(lib, wsb=need - 1) == WS_SMALL
    v = ctypes.c_void_p
    prep = lambda **kw: lib.moe_mxfp8_prepare_weight(
        kw.get("which", 0), v(kw.get("w", FAKE)), kw.get("D", 256), kw.get("F", 256), kw.get("E", 8),
        v(kw.get("data", FAKE)), kw.get("nd", 1 << 40), v(kw.get("sc", FAKE)), kw.get("ns", 1 << 40), None)
    assert prep(which=2) == INVALID
    assert prep(w=0) == INVALID
    assert prep(D=64) == SHAPE
    assert prep(sc=FAKE + 16) == MISALIGNED
    nd, ns = binding.moe_mxfp8_weight_bytes(binding.MOE_WEIGHT_W2, 256, 256, 8)
    assert prep(which=1, nd=nd - 1) == WS_SMALL
    assert prep(which=1, ns=ns - 1) == WS_SMALL


@pytest.mark.parametrize("dims", [(16, 256, 256, 8, 2), (4096, 2048, 1408, 64, 6), (64, 7168, 2048, 256, 8),
                                  (16384, 7168, 2048, 256, 8), (16384, 4096, 1536, 128, 8), (1, 128, 128, 1, 1)])
def test_mxfp8_sizes_and_layout(lib, dims):
    T, D, F, E, K = dims
    R = T * K
    nd, ns = binding.moe_mxfp8_weight_bytes(binding.MOE_WEIGHT_W13, D, F, E)
    assert nd == E * 2 * F * D and ns == E * -(-F // 96) * (D // 128) * 1024
    nd, ns = binding.moe_mxfp8_weight_bytes(binding.MOE_WEIGHT_W2, D, F, E)
    assert nd == E * D * F and ns == E * -(-D // 192) * (F // 128) * 1024
    lay = binding.moe_mxfp8_workspace_layout(*dims)
    rp = 128 * (-(-R // 128) + min(E, R))
    sizes = {"status": 4, "counts": 4 * E, "offsets": 4 * (E + 1), "tiles": 4 * (E + 1), "perm": 4 * R,
             "inv": 4 * R, "xq": rp * D, "xs": rp * D // 32, "hq": rp * F, "hs": rp * F // 32, "y": 2 * R * D}
    names = list(binding.MXWS_REGIONS)
    for i, name in enumerate(names[:-1]):
        assert lay[name] % 256 == 0
        if name in sizes:
            assert lay[names[i + 1]] - lay[name] >= sizes[name], name
    assert lay["status"] == 0
    assert lay["total"] == binding.moe_mxfp8_workspace_bytes(*dims)


def test_binding_mx_region_list_matches_header():
    text = open(HEADER).read()
    n = int(re.search(r"MOE_MXWS_REGIONS\s*=\s*(\d+)", text).group(1))
    assert len(binding.MXWS_REGIONS) == n


def test_mxfp8_stage_range_validation(lib):
    v = ctypes.c_void_p
    st = lambda b, e, **kw: lib.moe_fwd_mxfp8_stages(
        v(FAKE), v(FAKE), v(FAKE), 0, v(FAKE), v(FAKE), v(FAKE), v(FAKE), v(FAKE), kw.get("T", 16), 256, 256, 8, 2,
        b, e, v(FAKE), 1 << 40, None)
    assert st(-1, 2) == INVALID
    assert st(0, 5) == INVALID
    assert st(3, 2) == INVALID
    assert st(2, 2) == OK  # an empty range enqueues nothing
    assert st(0, 4, T=0) == OK


def test_nvfp4_host_validation_and_sizes(lib):
    v = ctypes.c_void_p
    f = ctypes.c_float
    nv = lambda **kw: lib.moe_routed_experts_fwd_nvfp4(
        v(FAKE), v(FAKE), v(FAKE), kw.get("sd", 0), v(kw.get("w13q", FAKE)), v(kw.get("w13s", FAKE)), v(FAKE),
        v(FAKE), f(kw.get("gx", 0.01)), f(kw.get("gh", 0.01)), v(FAKE), kw.get("T", 16), kw.get("D", 256),
        kw.get("F", 256), 8, 2, v(kw.get("ws", FAKE)), kw.get("wsb", 1 << 40), None)
    assert nv(T=0) == OK
    assert nv(gx=0.0) == INVALID
    assert nv(gh=-1.0) == INVALID
    assert nv(gx=float("inf")) == INVALID
    assert nv(gh=float("nan")) == INVALID
    assert nv(sd=5) == INVALID
    assert nv(w13s=0) == INVALID
    assert nv(D=192) == SHAPE
    assert nv(w13s=FAKE + 16) == MISALIGNED
    assert nv(ws=FAKE + 32) == MISALIGNED
    need = binding.moe_nvfp4_workspace_bytes(16, 256, 256, 8, 2)
    assert nv(wsb=need - 1) == WS_SMALL
    for D, F, E in ((2048, 1408, 64), (7168, 2048, 256), (640, 384, 3)):
        nd, ns = binding.moe_nvfp4_weight_bytes(binding.MOE_WEIGHT_W13, D, F, E)
        assert nd == E * 2 * F * D // 2 and ns == 256 + E * -(-F // 64) * (-(-D // 256) * 4) * 512
        nd, ns = binding.moe_nvfp4_weight_bytes(binding.MOE_WEIGHT_W2, D, F, E)
        assert nd == E * D * F // 2 and ns == 256 + E * -(-D // 128) * (-(-F // 256) * 4) * 512
    T, D, F, E, K = 4096, 2048, 1408, 64, 6
    lay = binding.moe_nvfp4_workspace_layout(T, D, F, E, K)
    rp = 128 * (-(-T * K // 128) + E)
    assert lay["xs"] - lay["xq"] >= rp * D // 2 and lay["hs"] - lay["hq"] >= rp * F // 2
    assert lay["hq"] - lay["xs"] >= rp // 128 * (-(-D // 256) * 4) * 512
    assert lay["y"] - lay["hs"] >= rp // 128 * (-(-F // 256) * 4) * 512
    assert lay["total"] == binding.moe_nvfp4_workspace_bytes(T, D, F, E, K)
