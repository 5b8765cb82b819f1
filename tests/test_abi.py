"""C-ABI checks that need no GPU: the library loads, exports every function that
include/gda.h declares, and its host-side validation answers before any CUDA call."""
import ctypes
import os
import re

import pytest

import gated_gqa_attention_gb300 as gda
from gated_gqa_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gda.h")

OK, ERR_NULL, ERR_ALIGN, ERR_SHAPE, ERR_UNSUPPORTED, ERR_SPLITS, ERR_WORKSPACE = 0, -1, -2, -3, -4, -5, -6
ERR_ARG = -10


@pytest.fixture(scope="module")
def lib():
    build.build()  # nvcc cross-compiles without a GPU
    return gda.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**(gda_[A-Za-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gda_decode", "gda_decode_ex", "gda_workspace_bytes", "gda_reserve", "gda_gate",
                     "gda_status_str", "gda_read_error", "gda_workspace_init", "gda_version"):
        assert required in names, names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(-10, 1):
        s = gda.status_str(code)
        assert s.startswith("GDA_"), s
    assert "unknown" in gda.status_str(-100)
    assert gda.version() >= 100


def test_workspace_bytes(lib):
    G, D = 8, 256
    piece = G * D * 4 + G * 4
    # explicit splits: B * Hkv * S pieces (+ header, 256-byte rounding)
    b = gda.workspace_bytes(64, 16, 2, 256, 8)
    assert b >= 256 + 64 * 2 * 8 * piece and b % 256 == 0
    assert b - (256 + 64 * 2 * 8 * piece) < 1024
    # automatic mode: bounded by the stage-1 grid cap + B * Hkv pieces
    a = gda.workspace_bytes(64, 16, 2, 256, 0)
    assert a >= 256 + (1024 + 128) * piece
    # invalid or unsupported sizes -> 0
    assert gda.workspace_bytes(-1, 16, 2, 256, 0) == 0
    assert gda.workspace_bytes(4, 16, 3, 256, 0) == 0      # Hq % Hkv
    assert gda.workspace_bytes(4, 16, 2, 128, 0) == 0      # D unsupported
    assert gda.workspace_bytes(4, 16, 4, 256, 0) > 0       # any group size (here 4)
    # G = 16 makes two passes (virtual heads of 8): twice the pieces of G = 8 at the same Hkv
    assert gda.workspace_bytes(4, 32, 2, 256, 8) > 1.9 * gda.workspace_bytes(4, 16, 2, 256, 8)
    assert gda.workspace_bytes(4, 16, 2, 256, 257) == 0    # too many splits


def test_workspace_holds_every_team_layout(lib):
    # G > 8: the BF16 MMA kernel serves the groups of 8 in teams (pairs for 2 or 4
    # groups, threes otherwise), the FP8 kernel in pairs (not for 3 groups), the other
    # kernels one group per piece; a team piece holds t partials at piece * t + group.
    # The caller-sized workspace holds the largest of these layouts.
    G8, D = 8, 256
    piece = G8 * D * 4 + G8 * 4

    def pieces(B, vheads, S):
        return B * vheads * S if S > 0 else 1024 + B * vheads

    def teams(npass):
        bf16 = 1 if npass <= 1 else 2 if npass in (2, 4) else 3
        fp8 = 1 if npass in (1, 3) else 2
        return {1, bf16, fp8}

    for B in (1, 7, 64, 224):
        for Hkv in (1, 2, 4):
            for G in (1, 8, 9, 16, 20, 24, 32, 40, 56, 64):
                npass = -(-G // 8)
                for S in (0, 1, 3, 8):
                    need = max(t * pieces(B, Hkv * -(-npass // t), S) for t in teams(npass)) * piece
                    assert gda.workspace_bytes(B, G * Hkv, Hkv, D, S) >= 256 + need, (B, Hkv, G, S)


def _decode(lib, ptrs=None, B=1, Hq=16, Hkv=2, D=256, scale=0.0625, splits=0):
    p = dict(q=16, gate=16, k=16, v=16, indptr=16, indices=16, out=16)
    if ptrs:
        p.update(ptrs)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return lib.gda_decode(vp(p["q"]), vp(p["gate"]), vp(p["k"]), vp(p["v"]), vp(p["indptr"]),
                          vp(p["indices"]), vp(p["out"]), B, Hq, Hkv, D, scale, splits, None)


def test_decode_host_validation(lib):
    # every case below is rejected before any CUDA call (no GPU needed)
    assert _decode(lib, {"q": 0}) == ERR_NULL
    assert _decode(lib, {"gate": 0}) == ERR_NULL
    assert _decode(lib, {"indices": 0}) == ERR_NULL
    assert _decode(lib, {"out": 0}) == ERR_NULL
    assert _decode(lib, {"q": 24}) == ERR_ALIGN
    assert _decode(lib, {"k": 8}) == ERR_ALIGN
    assert _decode(lib, {"indptr": 2}) == ERR_ALIGN
    assert _decode(lib, B=-1) == ERR_SHAPE
    assert _decode(lib, Hq=16, Hkv=3) == ERR_SHAPE
    assert _decode(lib, Hkv=0) == ERR_SHAPE
    assert _decode(lib, D=128) == ERR_UNSUPPORTED
    assert _decode(lib, splits=300) == ERR_SPLITS
    # B == 0 is a valid empty call: nothing to do, no pointer needed
    assert _decode(lib, {"q": 0, "gate": 0, "k": 0, "v": 0, "indptr": 0, "indices": 0, "out": 0}, B=0) == OK


def test_decode_ex_host_validation(lib):
    args = gda._Args(q=16, gate=16, k_pool=16, v_pool=16, kv_indptr=16, kv_indices=16, out=16, lse=None,
                     num_slots=10, B=2, Hq=16, Hkv=2, D=256, scale=0.0625, num_splits=0, fuse_gate=1,
                     check_indices=0, variant=0, min_chunk=0, window=0, sinks=None)
    call = lambda a, ws=256, nbytes=1 << 30: lib.gda_decode_ex(ctypes.byref(a), ctypes.c_void_p(ws) if ws else None,
                                                               nbytes, None)
    assert lib.gda_decode_ex(None, None, 0, None) == ERR_NULL
    assert call(args, ws=0) == ERR_WORKSPACE
    assert call(args, ws=128) == ERR_WORKSPACE                       # not 256-aligned
    assert call(args, nbytes=1024) == ERR_WORKSPACE                  # too small
    a2 = gda._Args.from_buffer_copy(args)
    a2.variant = 7
    assert call(a2) == ERR_UNSUPPORTED
    a3 = gda._Args.from_buffer_copy(args)
    a3.gate = None
    assert call(a3) == ERR_NULL                                       # gate needed when fused
    a3.fuse_gate = 0
    a3.q = 8
    assert call(a3) == ERR_ALIGN                                      # gate may be absent unfused
    a4 = gda._Args.from_buffer_copy(args)
    a4.check_indices, a4.num_slots = 1, -1
    assert call(a4) == ERR_SHAPE
    a5 = gda._Args.from_buffer_copy(args)
    a5.lse = 2
    assert call(a5) == ERR_ALIGN
    a6 = gda._Args.from_buffer_copy(args)
    a6.window = -1
    assert call(a6) == ERR_SHAPE
    a7 = gda._Args.from_buffer_copy(args)
    a7.sinks = 6
    assert call(a7) == ERR_ALIGN
    a7 = gda._Args.from_buffer_copy(args)
    a7.total_len = -1
    assert call(a7) == ERR_SHAPE
    # e4m3 pools: the MMA kernel only, finite descales, a known element type
    a8 = gda._Args.from_buffer_copy(args)
    a8.kv_dtype = 2
    assert call(a8) == ERR_UNSUPPORTED
    a8.kv_dtype = gda.KV_E4M3
    a8.variant = gda.VARIANT_SIMT
    assert call(a8) == ERR_UNSUPPORTED
    a8.variant = gda.VARIANT_TMA
    assert call(a8) == ERR_UNSUPPORTED
    a8.variant = gda.VARIANT_MMA
    a8.k_descale, a8.v_descale = float("nan"), 1.0
    assert call(a8) == ERR_ARG
    a8.k_descale, a8.v_descale = 1.0, float("inf")
    assert call(a8) == ERR_ARG
    a8.v_descale = 1.0
    a8.v_pool = 8
    assert call(a8) == ERR_ALIGN
    # the descales of a bf16 call are not used (left zero by the struct's initialiser)
    a9 = gda._Args.from_buffer_copy(args)
    a9.k_descale = float("nan")
    a9.B = 0
    assert call(a9) == OK


def _decode_e4m3(lib, ptrs=None, B=1, Hq=16, Hkv=2, D=256, scale=0.0625, kd=1.0, vd=1.0, splits=0):
    p = dict(q=16, gate=16, k=16, v=16, indptr=16, indices=16, out=16)
    if ptrs:
        p.update(ptrs)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return lib.gda_decode_e4m3(vp(p["q"]), vp(p["gate"]), vp(p["k"]), vp(p["v"]), vp(p["indptr"]),
                               vp(p["indices"]), vp(p["out"]), B, Hq, Hkv, D, scale, kd, vd, splits, None)


def test_decode_e4m3_host_validation(lib):
    assert _decode_e4m3(lib, {"k": 0}) == ERR_NULL
    assert _decode_e4m3(lib, {"v": 24}) == ERR_ALIGN
    assert _decode_e4m3(lib, kd=float("nan")) == ERR_ARG
    assert _decode_e4m3(lib, vd=float("-inf")) == ERR_ARG
    assert _decode_e4m3(lib, D=128) == ERR_UNSUPPORTED
    assert _decode_e4m3(lib, Hq=16, Hkv=3) == ERR_SHAPE
    assert _decode_e4m3(lib, splits=257) == ERR_SPLITS
    assert _decode_e4m3(lib, {"q": 0, "gate": 0, "k": 0, "v": 0, "indptr": 0, "indices": 0, "out": 0}, B=0) == OK


def test_gate_and_misc_host_validation(lib):
    vp = ctypes.c_void_p
    assert lib.gda_gate(vp(16), vp(16), vp(16), -1, None) == ERR_SHAPE
    assert lib.gda_gate(None, None, None, 0, None) == OK              # empty
    assert lib.gda_gate(None, vp(16), vp(16), 8, None) == ERR_NULL
    assert lib.gda_gate(vp(16), vp(18), vp(16), 8, None) == ERR_ALIGN
    assert lib.gda_reserve(4, 16, 2, 128, 0) == ERR_UNSUPPORTED
    assert lib.gda_workspace_init(None, 1024, None) == ERR_NULL
    assert lib.gda_workspace_init(vp(128), 1024, None) == ERR_ALIGN
    assert lib.gda_workspace_init(vp(256), 16, None) == ERR_WORKSPACE
    w = ctypes.c_uint32()
    assert lib.gda_read_error(None, None, 0, None) == ERR_NULL


def test_product_path_has_no_cpu_fallback():
    # the binding refuses to run without the library rather than computing elsewhere
    import importlib
    pkg = os.path.join(ROOT, "gated_gqa_attention_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            src = open(os.path.join(pkg, name)).read()
            assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), name
    for name in os.listdir(os.path.join(pkg, "csrc")):
        src = open(os.path.join(pkg, "csrc", name)).read()
        assert not re.search(r"#include\s+[<\"].*oracle", src), name
    mod = importlib.import_module("gated_gqa_attention_gb300")
    with pytest.raises(RuntimeError):
        mod._lib_saved = mod._lib
        try:
            mod._lib = None
            mod.load(os.path.join(ROOT, "does-not-exist", "libgda.so"))
        finally:
            mod._lib = mod._lib_saved


def test_prefill_host_validation(lib):
    vp = lambda x: ctypes.c_void_p(x) if x else None

    def call(q=16, gate=16, k=16, v=16, lens=0, out=16, lse=0, B=1, Sq=8, Skv=8, Hq=4, Hkv=2, D=256,
             scale=0.0625, causal=1, err=0):
        return lib.gda_prefill(vp(q), vp(gate), vp(k), vp(v), vp(lens), vp(out), vp(lse), B, Sq, Skv, Hq, Hkv, D,
                               scale, causal, vp(err), None)
    assert call(q=0) == ERR_NULL
    assert call(out=0) == ERR_NULL
    assert call(k=0) == ERR_NULL
    assert call(q=24) == ERR_ALIGN
    assert call(lse=2) == ERR_ALIGN
    assert call(Hq=4, Hkv=3) == ERR_SHAPE
    assert call(Sq=-1) == ERR_SHAPE
    assert call(D=128) == ERR_UNSUPPORTED
    assert call(scale=0.0) == ERR_ARG
    assert call(scale=-0.5) == ERR_ARG
    assert call(scale=float("inf")) == ERR_ARG
    assert call(B=0, q=0, k=0, v=0, out=0) == OK
    assert call(Sq=0, q=0, k=0, v=0, out=0) == OK
    assert lib.gda_prefill_read_error(None, 0, None) == ERR_NULL


def test_step_host_layout_and_validation(lib):
    # gda_step_layout: 256-byte aligned parts q | gate | kv_indptr | kv_indices
    lib.gda_step_layout.restype = ctypes.c_size_t
    lib.gda_step_layout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                    ctypes.POINTER(ctypes.c_size_t)]
    off = (ctypes.c_size_t * 4)()
    total = lib.gda_step_layout(3, 4, 256, 10, off)
    qg = 3 * 4 * 256 * 2
    assert list(off) == [0, qg, 2 * qg, 2 * qg + 256] and total == 2 * qg + 512
    assert all(o % 256 == 0 for o in off) and total % 256 == 0
    assert lib.gda_step_layout(0, 4, 256, 10, off) == 0
    assert lib.gda_step_layout(3, 4, 256, -1, off) == 0
    assert lib.gda_step_layout(3, 4, 256, 10, None) == 0
    # gda_decode_step_host: every host-side check before any CUDA call
    vp = ctypes.c_void_p
    f = lib.gda_decode_step_host
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, ctypes.c_size_t, vp, vp, ctypes.c_int, ctypes.c_float, ctypes.c_float, vp, vp, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, vp]
    B, Hq, Hkv, D, nnz = 3, 4, 2, 256, 10
    total = lib.gda_step_layout(B, Hq, D, nnz, off)

    def call(host_in=4096, dev_in=4096, nbytes=total, k=4096, v=4096, dout=4096, hout=4096, B=B, Hq=Hq, Hkv=Hkv,
             D=D, nnz=nnz, splits=0, flags=0, kv=0, kd=1.0):
        return f(vp(host_in) if host_in else None, vp(dev_in) if dev_in else None, nbytes, vp(k) if k else None,
                 vp(v) if v else None, kv, kd, 1.0, vp(dout) if dout else None, vp(hout) if hout else None, B, Hq,
                 Hkv, D, nnz, 0.0625, splits, flags, 1, None)

    assert call(B=0) == OK
    assert call(B=-1) == ERR_SHAPE
    assert call(nbytes=total - 256) == ERR_SHAPE
    assert call(nnz=-2) == ERR_SHAPE
    assert call(host_in=0) == ERR_NULL
    assert call(hout=0) == ERR_NULL
    assert call(dev_in=4096 + 128) == ERR_ALIGN
    assert call(k=0) == ERR_NULL
    assert call(v=4096 + 8) == ERR_ALIGN
    assert call(dout=4096 + 2) == ERR_ALIGN
    assert call(D=128, nbytes=lib.gda_step_layout(B, Hq, 128, nnz, off)) == ERR_UNSUPPORTED
    assert call(Hkv=3) == ERR_SHAPE
    assert call(splits=300) == ERR_SPLITS
    assert call(flags=4) == ERR_ARG                       # an unknown flag
    assert call(dev_in=0) == ERR_NULL and call(dout=0) == ERR_NULL
    assert call(host_in=4096 + 16, flags=1) == ERR_ALIGN  # a mapped block starts on 256 bytes
    assert call(kv=7) == ERR_UNSUPPORTED                  # an unknown cache type
    assert call(kv=1, kd=float("nan")) == ERR_ARG         # e4m3 with a non-finite descale

    # kv_indptr is read from the host block before anything is enqueued: a first entry
    # other than 0, a last entry other than nnz, or a decreasing pair is refused (the
    # kernels would read kv_indices past the end of the block)
    import numpy as np
    raw = np.zeros(total + 256, dtype=np.uint8)
    base = raw.ctypes.data
    shift = (-base) % 256
    block = raw[shift:shift + total]
    ip = block[off[2]:off[2] + 4 * (B + 1)].view(np.int32)
    for bad in ([1, 4, 7, 10], [0, 4, 7, 9], [0, 4, 7, 11], [0, 6, 4, 10], [0, -1, 4, 10]):
        ip[:] = bad
        assert call(host_in=base + shift) == ERR_SHAPE, bad
    assert call(host_in=base + shift, nbytes=total - 256) == ERR_SHAPE


def test_auto_splits_matches_the_plan_model(lib):
    # gda_auto_splits (host) restates the device rule; the CPU plan model restates
    # both: they agree on random batches, and invalid arguments give -1
    import random
    import test_plan_model as plan
    rng = random.Random(21)
    for _ in range(3000):
        B = rng.randint(0, 200)
        lens = [rng.choice([0, 1, 16, 65, 300, 512, 2048, 3000, 8192, 32768]) for _ in range(B)]
        if rng.random() < 0.5:
            lens = [lens[0] if B else 0] * B
        indptr = [0]
        for L in lens:
            indptr.append(indptr[-1] + L)
        heads, grid, mc = rng.choice([1, 2, 4, 8]), rng.choice([7, 148, 152]), rng.choice([16, 64])
        lmax = max(lens + [0])
        assert gda.auto_splits(B, heads, grid, lmax, indptr[-1], mc) == plan.uniform_splits(indptr, heads, grid, mc)
    assert gda.auto_splits(-1, 2, 152, 10, 10) == -1
    assert gda.auto_splits(4, 0, 152, 10, 10) == -1
    assert gda.auto_splits(4, 2, 152, 10, -5) == -1
    # the bench workloads: stream for b64_l4096 and b8_l131072, 8 splits for B4 ragged
    assert gda.auto_splits(64, 2, 152, 4096, 64 * 4096) == 0
    assert gda.auto_splits(8, 2, 152, 131072, 8 * 131072) == 0
    assert gda.auto_splits(4, 2, 152, 512, 1946) == 8
