"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol,
and its host-only entry points (EPLB map, size queries, argument checks) behave."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from combine_moe_route_03_gb300 import _lib, api, configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from combine_moe_route_03_gb300 import build
    build.build()
    return _lib.load()


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "moe.h")).read()
    return set(re.findall(r"^(?:int|size_t|int64_t)\s+\**(\w+)\(", hdr, re.M))


def test_exports_every_declared_symbol(L):
    decl = declared_symbols()
    assert decl == set(_lib.SIGNATURES)
    for name in decl:
        assert getattr(L, name) is not None


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "moe.h"\nint main(void){moe_route_cfg c; (void)c; return 0;}\n')
    import subprocess
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", str(tmp_path / "t")])


STRUCTS = {"RouteCfg": "moe_route_cfg", "DispatchCfg": "moe_dispatch_cfg",
           "EplbCfg": "moe_eplb_cfg", "GemmArgs": "moe_gemm_args",
           "CombineCfg": "moe_combine_cfg", "Layer": "moe_layer",
           "FusedCombine": "moe_fused_combine"}


def test_binding_structs_match_the_c_layout(tmp_path):
    """Every ctypes structure of the binding has the C struct's size, and each of its
    fields the C field's offset and size (gcc, printed by a program including moe.h)."""
    import subprocess
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "moe.h"', 'int main(void){']
    for py, c in STRUCTS.items():
        lines.append(f'printf("{py} . %zu %zu\\n", sizeof({c}), (size_t)0);')
        for f, _ in getattr(_lib, py)._fields_:
            lines.append(f'printf("{py} {f} %zu %zu\\n", offsetof({c}, {f}), '
                         f'sizeof((({c} *)0)->{f}));')
    lines.append("return 0;}")
    (tmp_path / "l.c").write_text("\n".join(lines) + "\n")
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(tmp_path / "l.c"), "-o", str(tmp_path / "l")])
    out = subprocess.check_output([str(tmp_path / "l")], text=True).split("\n")
    n = 0
    for line in filter(None, out):
        py, f, a, b = line.split()
        cls = getattr(_lib, py)
        if f == ".":
            assert ctypes.sizeof(cls) == int(a), py
        else:
            fd = getattr(cls, f)
            assert (fd.offset, fd.size) == (int(a), int(b)), (py, f)
            n += 1
    assert n == sum(len(getattr(_lib, py)._fields_) for py in STRUCTS)


def _kind(c_type: str) -> str:
    c_type = c_type.strip()
    if "*" in c_type:
        return "ptr"
    base = c_type.replace("const", "").split()[0]
    return {"int": "int", "size_t": "size", "int64_t": "i64", "float": "f32",
            "double": "f64"}[base]


def _ctypes_kind(t) -> str:
    if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int: "int", ctypes.c_size_t: "size", ctypes.c_int64: "i64",
            ctypes.c_float: "f32", ctypes.c_double: "f64"}[t]


def test_binding_signatures_match_the_header():
    """Each declared entry point's return type and parameter list (count, and pointer
    or integer width of each) equals the binding's ctypes signature."""
    hdr = open(os.path.join(ROOT, "include", "moe.h")).read()
    hdr = re.sub(r"/\*.*?\*/", " ", hdr, flags=re.S)
    hdr = re.sub(r"//[^\n]*", " ", hdr)
    decls = re.findall(r"^(int|size_t|int64_t)\s+(\w+)\s*\(([^;{]*?)\)\s*;", hdr, re.M | re.S)
    assert {d[1] for d in decls} == set(_lib.SIGNATURES)
    for ret, name, params in decls:
        res, args = _lib.SIGNATURES[name]
        assert _kind(ret) == _ctypes_kind(res), name
        ps = [] if params.strip() in ("", "void") else params.split(",")
        assert [_kind(" ".join(p.split()[:-1]) + (" *" if "*" in p else "")) for p in ps] == \
            [_ctypes_kind(a) for a in args], name

@pytest.mark.parametrize("seed", range(6))
def test_eplb_map_matches_oracle(L, seed):
    rng = np.random.default_rng(seed)
    N = [8, 32, 256][seed % 3]
    counts = rng.integers(0, 6, N) * rng.integers(1, 4)        # many ties
    for extra in (0, 1, N // 8, N):
        got = api.eplb_build_map(counts, N, N + extra)
        ref = oracle.eplb_build_map(counts, N, N + extra)
        for g, r in zip(got, ref):
            assert np.array_equal(g, r)


def test_eplb_map_rejects_bad_sizes(L):
    with pytest.raises(_lib.MoEError):
        api.eplb_build_map(np.zeros(8), 8, 7)
    with pytest.raises(_lib.MoEError):
        api.eplb_build_map(np.zeros(8), 8, 17)


@pytest.mark.parametrize("name", list(configs.ALL))
def test_dispatch_size_queries(L, name):
    cfg = configs.ALL[name]
    sz = api.dispatch_sizes(cfg)
    if cfg.layout == configs.CONTIG:
        assert sz["rows"] == oracle.contig_rows_alloc(cfg.B, cfg.K, cfg.N_phys)
    else:
        assert sz["rows"] == cfg.N_phys * cfg.cap
    assert sz["max_tiles"] * 128 == sz["rows"] and sz["ws"] > 0


def test_host_argument_checks_return_before_launch(L):
    bad = _lib.RouteCfg(4, 100, 8, 2, 1, 1, 0, 0, 1.0)           # H % 32 != 0
    assert L.moe_route(ctypes.byref(bad), None, None, None, None, None, None, None, 0, None) == -2
    bad = _lib.RouteCfg(4, 128, 8, 9, 1, 1, 0, 0, 1.0)            # K > N
    assert L.moe_route(ctypes.byref(bad), None, None, None, None, None, None, None, 0, None) == -2
    bad = _lib.RouteCfg(4, 128, 16, 8, 4, 1, 1, 1, 1.0)           # K > experts in kept groups
    assert L.moe_route(ctypes.byref(bad), None, None, None, None, None, None, None, 0, None) == -2
    ok = _lib.RouteCfg(4, 128, 8, 2, 1, 1, 0, 0, 1.0)
    assert L.moe_route(ctypes.byref(ok), None, None, None, None, None, None, None, 0, None) == -1
    dc = _lib.DispatchCfg(4, 100, 2, 8, 8, 0, 0, 0)               # H % 128 != 0
    assert L.moe_dispatch_rows(ctypes.byref(dc)) == 0
    dc = _lib.DispatchCfg(4, 128, 2, 8, 8, 1, 100, 0)             # cap % 128 != 0
    assert L.moe_dispatch(ctypes.byref(dc), *([None] * 14), 0, None, None) == -2
    g = _lib.GemmArgs(0, 300, 128, 128, 1, 1, *([None] * 7), 0, 0, None, None, None, 64, 0, 0, 0,
                      None)
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -2
    g = _lib.GemmArgs(0, 256, 128, 128, 1, 1, *([None] * 7), 0, 0, None, None, None, 64, 0, 0, 0,
                      None)
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    g = _lib.GemmArgs(0, 256, 128, 128, 1, 1, *([None] * 7), 0, 0, None, None, None, 64, 0, 1, 1,
                      None)                                     # binary32 scales: one CTA only
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -2
    g = _lib.GemmArgs(0, 256, 128, 128, 1, 1, *([None] * 7), 0, 0, None, None, None, 64, 0, 0, 2,
                      None)                                     # no such scale format
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    p = [ctypes.c_void_p(16)] * 4
    fc = _lib.FusedCombine(4, 2, 16, 16, 16, 128, 16, -1, 16)
    g = _lib.GemmArgs(0, 256, 128, 128, 1, 1, *p, None, 16, None, 0, 0, 16, 16, None, 64, 0, 0,
                      0, None, ctypes.pointer(fc))                # fused combine on gate/up
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    for bad in (_lib.FusedCombine(4, 17, 16, 16, 16, 128, 16, -1, 16),     # K > 16
                _lib.FusedCombine(4, 2, 16, 16, 16, 128, 16, -1, 8),       # out unaligned
                _lib.FusedCombine(4, 2, 16, 16, None, 128, 16, -1, 16),    # no src_of
                _lib.FusedCombine(4, 2, 16, 16, 16, 128, 16, 126, 16)):    # shared rows past rows
        g = _lib.GemmArgs(1, 256, 128, 128, 1, 1, *p, None, 16, None, 0, 0, 16, None, None, 64,
                          0, 0, 0, None, ctypes.pointer(bad))
        assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    g = _lib.GemmArgs(1, 256, 128, 128, 1, 1, *p, None, 16, None, 0, 0, 16, None, 16, 64, 0, 0,
                      0, None, ctypes.pointer(fc))                # with SBO signals
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    for op, tile_n in ((1, 100), (0, 224)):                      # no such width; gate/up
        g = _lib.GemmArgs(op, 1792, 256, 128, 1, 1, *p, None, 16, None, 0, 0, 16, 16, None, 64,
                          0, 0, 0, None, None, tile_n)
        assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    g = _lib.GemmArgs(1, 1536, 256, 128, 1, 1, *p, None, 16, None, 0, 0, 16, None, None, 64, 0,
                      0, 0, None, None, 224)                   # n % 224 != 0
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -2
    g = _lib.GemmArgs(1, 1792, 256, 128, 1, 1, *p, None, 16, None, 0, 0, 16, None, None, 64, 0,
                      2, 0, None, None, 0)                     # pair_tiles 2 is no mode
    assert L.moe_grouped_gemm_fp8(ctypes.byref(g), None) == -1
    assert L.moe_tiled_scale_bytes(2, 1792, 640, 224) == 2 * 8 * 2 * 1024
    assert L.moe_tiled_scale_bytes(2, 1792, 640, 100) == 0 and L.moe_tiled_scale_bytes(2, 1536, 640, 224) == 0
    assert L.moe_fused_combine_prep(None, 256, None) == -1
    assert L.moe_fused_combine_prep(ctypes.byref(_lib.FusedCombine(4, 0, 16, 16, 16, 128, 16,
                                                                   -1, 16)), 256, None) == -1
    assert L.moe_fused_combine_prep(ctypes.byref(_lib.FusedCombine(4, 17, 16, 16, 16, 128, 16,
                                                                   -1, 16)), 256, None) == -2
    assert L.moe_fused_combine_prep(ctypes.byref(fc), 384, None) == -2      # n % 256
    assert L.moe_fused_combine_prep(ctypes.byref(_lib.FusedCombine(0, 2, None, None, None, 0,
                                                                   None, -1, None)), 256, None) == 0
    cc = _lib.CombineCfg(4, 100, 2, None, 0, 64, 0, 0, 0)          # H % 128 != 0
    assert L.moe_combine(ctypes.byref(cc), *([None] * 7)) == -2
    assert L.moe_packed_scale_bytes(2, 256, 384) == 2 * 2 * 1 * 512   # 3 blocks: one group
    assert L.moe_packed_scale_bytes(2, 256, 640) == 2 * 2 * 2 * 512   # 5 blocks: two groups
    assert L.moe_scale_bytes(384, 7168, 0) == 3 * 14 * 512
    assert L.moe_scale_bytes(384, 7168, 2) == 384 * 56 * 4           # binary32 scales
    assert L.moe_scale_bytes(100, 7168, 0) == 0 and L.moe_scale_bytes(128, 100, 0) == 0
    assert L.moe_scale_bytes(128, 128, 1) == 0                         # bf16 rows: none
    h = ctypes.c_void_p()
    lay = _lib.Layer()
    assert L.moe_layer_graph_create(None, None, None, None, ctypes.byref(h)) == -1
    assert L.moe_layer_graph_create(ctypes.byref(lay), None, None, None, ctypes.byref(h)) == -1
    assert L.moe_layer_graph_create(ctypes.byref(lay), ctypes.c_void_p(16), None,
                                    ctypes.c_void_p(16), ctypes.byref(h)) == -1  # one host buffer
    assert L.moe_layer_graph_launch(None, None) == -1
    assert L.moe_layer_graph_destroy(None) == 0
    hx = (ctypes.c_void_p * 2)(16, 16)
    s1, s2 = ctypes.c_void_p(32), ctypes.c_void_p(48)
    f = L.moe_layer_forward_host_pipelined
    assert f(None, s1, s1, hx, hx, 2, s1, s2) == -1                          # no layer
    assert f(ctypes.byref(lay), s1, s1, hx, hx, 0, s1, s2) == -1             # no steps
    assert f(ctypes.byref(lay), s1, s1, hx, hx, 2, s1, s1) == -1             # one stream
    assert f(ctypes.byref(lay), None, s1, hx, hx, 2, s1, s2) == -1           # no 2nd buffer
    assert f(ctypes.byref(lay), s1, s1, (ctypes.c_void_p * 2)(16, None), hx, 2, s1, s2) == -1


def test_binding_calls_pass_every_parameter():
    """ctypes passes arguments beyond argtypes by default conversion (a pointer would go
    as a C int), so every call of an entry point in the binding, whether through
    load() or a local L = load(), passes exactly its declared parameters."""
    import ast
    src = open(os.path.join(ROOT, "combine_moe_route_03_gb300", "api.py")).read()
    calls = 0
    for node in ast.walk(ast.parse(src)):
        if not (isinstance(node, ast.Call) and isinstance(node.func, ast.Attribute)
                and node.func.attr in _lib.SIGNATURES):
            continue
        recv = node.func.value
        if not ((isinstance(recv, ast.Name) and recv.id == "L") or
                (isinstance(recv, ast.Call) and getattr(recv.func, "id", "") == "load")):
            continue
        assert not any(isinstance(a, ast.Starred) for a in node.args)
        assert len(node.args) == len(_lib.SIGNATURES[node.func.attr][1]), \
            (node.func.attr, node.lineno)
        calls += 1
    assert calls >= 18


def test_oracle_binding_matches_its_c_definitions():
    """The oracle's ctypes table against the C definitions in oracle/moe_oracle.c:
    return type and each parameter's kind (pointer, or integer / float width)."""
    src = open(os.path.join(ROOT, "oracle", "moe_oracle.c")).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    defs = re.findall(r"^(int|void|float|uint8_t|uint16_t)\s+(oracle_\w+)\s*\(([^;{]*?)\)\s*\{",
                      src, re.M | re.S)
    kinds = {"int": "int", "int64_t": "i64", "float": "f32", "uint8_t": "u8", "uint16_t": "u16",
             "void": None}
    ct = {ctypes.c_int: "int", ctypes.c_int64: "i64", ctypes.c_float: "f32",
          ctypes.c_uint8: "u8", ctypes.c_uint16: "u16", None: None}

    def ckind(t):
        if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
            return "ptr"
        if getattr(t, "__name__", "").startswith("ndpointer_"):    # numpy array pointers
            return "ptr"
        return ct[t]
    L = oracle.lib()
    checked = 0
    for ret, name, params in defs:
        fn = getattr(L, name)
        if fn.argtypes is None:          # helpers the binding never calls
            continue
        ps = [] if params.strip() in ("", "void") else params.split(",")
        want = ["ptr" if "*" in p else kinds[p.replace("const", "").split()[0]] for p in ps]
        assert [ckind(a) for a in fn.argtypes] == want, name
        assert ckind(fn.restype) == kinds[ret], name
        checked += 1
    assert checked >= 12


def test_binding_rejects_host_tensors_for_device_parameters(L):
    """A CPU tensor where the library expects device memory is refused in the binding,
    before any call: a kernel would otherwise dereference a host address."""
    import torch
    cfg = configs.TINY
    x = torch.zeros((cfg.B, cfg.H), dtype=torch.bfloat16)
    idx = torch.zeros((cfg.B, cfg.K), dtype=torch.int32)
    u8 = torch.zeros((256, 128), dtype=torch.uint8)
    calls = [
        lambda: api.route(cfg, x, torch.zeros((cfg.N, cfg.H)), None),
        lambda: api.dispatch(cfg, x, idx),
        lambda: api.combine(torch.zeros((4, 128), dtype=torch.bfloat16),
                            torch.zeros((2, 1), dtype=torch.int32), torch.ones((2, 1))),
        lambda: api.pack_weight_scales(torch.zeros((1, 1, 1), dtype=torch.uint8)),
        lambda: api.grouped_gemm_fp8(api.GEMM_DOWN, u8, u8, u8[None, :128], u8, idx, 1),
        lambda: api.read_status(torch.zeros(1, dtype=torch.int32)),
    ]
    for c in calls:
        with pytest.raises(ValueError, match="device parameter"):
            c()
    with pytest.raises(ValueError, match="contiguous"):
        _lib.ptr(torch.zeros((4, 4)).t(), host=True)
    assert _lib.ptr(torch.zeros(4), host=True) is not None and _lib.ptr(None) is None


def test_binding_checks_shapes_and_dtypes_against_the_config(L):
    """Arguments whose shape or dtype disagrees with the configuration are refused
    before any pointer is taken (a kernel would read past the smaller buffer)."""
    import torch
    cfg = configs.SMALL_CONTIG
    B, H, N, K = 10, cfg.H, cfg.N, cfg.K
    x = torch.zeros((B, H), dtype=torch.bfloat16)
    W = torch.zeros((N, H))
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)  # noqa: E731
    bad = [
        lambda: api.route(cfg, x[:, :128].contiguous(), W, None),           # H
        lambda: api.route(cfg, x, W[:-1].contiguous(), None),                # N rows of W
        lambda: api.route(cfg, x, W.double(), None),                          # W dtype
        lambda: api.route(cfg, x, W, torch.zeros(N + 1)),                     # bias length
        lambda: api.route(cfg, x.float(), W, None),                           # x dtype
        lambda: api.dispatch(cfg, x, i32(B, K + 1)),                          # K
        lambda: api.dispatch(cfg, x, i32(B, K).long()),                       # index dtype
        lambda: api.dispatch(cfg, x, i32(B, K), i32(N, 2), None),             # map half given
        lambda: api.dispatch(cfg, x, i32(B, K), i32(N - 1, 2), i32(N)),       # map rows
        lambda: api.combine(torch.zeros((40, H), dtype=torch.bfloat16), i32(B, K),
                            torch.zeros((B, K + 1))),                         # weights shape
        lambda: api.combine(torch.zeros((40, H), dtype=torch.bfloat16), i32(B, K),
                            torch.zeros((B, K)), shared=torch.zeros((B, H + 128),
                                                                    dtype=torch.bfloat16)),
    ]
    for i, c in enumerate(bad):
        with pytest.raises(ValueError, match="expected|together"):
            c()


def test_layer_rejects_row_buffers_smaller_than_dispatch_writes(L):
    """moe_layer_forward checks, before anything is launched, that the layer's row count
    and tile capacity hold what its dispatch writes."""
    lay = _lib.Layer()
    lay.route = _lib.RouteCfg(4, 128, 2, 4, 1, 1, 0, 0, 1.0)   # K > N: the router refuses (-2)
    lay.N_phys, lay.layout = 2, 0
    need = L.moe_dispatch_rows(ctypes.byref(_lib.DispatchCfg(4, 128, 4, 2, 2, 0, 0, 0)))
    assert need == 384
    lay.rows, lay.max_tiles = need, need // 128
    assert L.moe_layer_forward(ctypes.byref(lay), None) == -2  # sizes fine: on to the router
    lay.rows = need - 128
    assert L.moe_layer_forward(ctypes.byref(lay), None) == -1  # too few rows
    lay.rows, lay.max_tiles = need, need // 128 - 1
    assert L.moe_layer_forward(ctypes.byref(lay), None) == -1  # too few tiles
