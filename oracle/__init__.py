"""FP64 CPU oracle for gated split-KV GQA decode attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The CUDA library neither
imports nor links anything here, and nothing here imports the CUDA library.

The arithmetic lives in ``gda_oracle.c`` (plain C, IEEE double, no FMA
contraction); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  BF16 tensors travel as their uint16 bit patterns.

Definition followed (FreeToken PR #781 "Fuse the BF16 attention output sigmoid
gate into the existing Triton decode stage2", Summary and Automatic dispatch;
cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stages (4)-(5)):

    O   = softmax(scale * q K^T) V   over the CSR rows of sequence b, KV head h // G
    out = RNE_bf16( RNE_bf16(O) * RNE_bf16(sigmoid(gate)) )

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against brute force, closed forms, a library SDPA
and an independent 50-digit evaluation of the sigmoid.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK = 0
ORACLE_ERR_SHAPE = -1
ORACLE_ERR_INDEX = -2
ORACLE_ERR_NOMEM = -3


def build(force: bool = False) -> str:
    """Compile gda_oracle.c into liboracle.so next to it (gcc, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared",
           "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.oracle_double_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_double_from_bf16.restype = ctypes.c_double
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_double_from_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_double_from_e4m3.restype = ctypes.c_double
        lib.oracle_sigmoid_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_sigmoid_bf16.restype = ctypes.c_uint16
        lib.oracle_gate.argtypes = [u16p, u16p, u16p, ctypes.c_int64]
        lib.oracle_gate.restype = None
        lib.oracle_decode.argtypes = [
            u16p, u16p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            i32p, i32p, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            ctypes.c_int, f64p, i32p, ctypes.c_int64, f64p, u16p, u16p, f64p, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_qk_norm_rope_kv_write.argtypes = [
            u16p, ctypes.c_int64, u16p, u16p, ctypes.c_double, u16p, u16p, ctypes.c_int, i32p,
            u16p, u16p, u16p, u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_qk_norm_rope_kv_write.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [
            u16p, u16p, u16p, u16p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, ctypes.c_int, i32p, ctypes.c_int64, f64p, u16p, u16p, f64p, ctypes.c_int]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    """Accept a numpy uint16 array or a torch bfloat16 / int16 tensor (CPU)."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16, a.dtype
        return np.ascontiguousarray(a)
    import torch  # local: only when a tensor is passed
    t = a.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    assert t.dtype == torch.int16, t.dtype
    return t.numpy().view(np.uint16)


def _kv(a):
    """A K or V pool: (uint16 BF16 bits, False) or (uint8 e4m3 codes, True).
    Accepts numpy uint16 / uint8 arrays or torch bfloat16 / float8_e4m3fn / uint8
    tensors (CPU)."""
    if isinstance(a, np.ndarray):
        if a.dtype == np.uint8:
            return np.ascontiguousarray(a), True
        return _u16(a), False
    import torch  # local: only when a tensor is passed
    t = a.detach().cpu().contiguous()
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return t.view(torch.uint8).numpy(), True
    return _u16(t), False


def _i32(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a, dtype=np.int32)
    return np.ascontiguousarray(a.detach().cpu().numpy(), dtype=np.int32)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def double_from_bf16(bits) -> np.ndarray:
    """Exact widening of BF16 bit patterns (vectorised: a BF16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_double(x) -> np.ndarray:
    """RNE rounding of doubles to BF16 bit patterns, one element at a time through the C oracle."""
    lib = _load()
    xs = np.asarray(x, dtype=np.float64)
    flat = xs.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = lib.oracle_bf16_from_double(float(v))
    return out.reshape(xs.shape)


def double_from_e4m3(codes) -> np.ndarray:
    """Values of e4m3 codes (uint8), one element at a time through the C oracle."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    flat = c.reshape(-1)
    out = np.empty(flat.shape, dtype=np.float64)
    for i, v in enumerate(flat):
        out[i] = lib.oracle_double_from_e4m3(int(v))
    return out.reshape(c.shape)


def sigmoid_bf16(g_bits) -> np.ndarray:
    """RNE_bf16(sigmoid(g)) for BF16 bit patterns g."""
    lib = _load()
    g = np.asarray(g_bits, dtype=np.uint16)
    flat = g.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = lib.oracle_sigmoid_bf16(int(v))
    return out.reshape(g.shape)


def gate(o_bits, gate_bits) -> np.ndarray:
    """out = RNE_bf16(o * RNE_bf16(sigmoid(gate))) on BF16 bit patterns."""
    o = _u16(o_bits)
    g = _u16(gate_bits)
    assert o.shape == g.shape
    out = np.empty(o.shape, dtype=np.uint16)
    _load().oracle_gate(_ptr(o, ctypes.c_uint16), _ptr(g, ctypes.c_uint16),
                        _ptr(out, ctypes.c_uint16), o.size)
    return out


class DecodeResult:
    """Oracle outputs; each field is None when it was not requested."""

    def __init__(self, o_f64, o_bf16, out, lse):
        self.o_f64 = o_f64
        self.o_bf16 = o_bf16
        self.out = out
        self.lse = lse


def decode(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, scale: float,
           num_splits: int = 0, pairs=None, want=("o_f64", "o_bf16", "out", "lse"),
           nthreads: int = 0, window: int = 0, sinks=None, k_descale: float = 1.0,
           v_descale: float = 1.0) -> DecodeResult:
    """Gated GQA decode attention in FP64.

    q, gate_t: [B, Hq, D] BF16 (uint16 bits or torch bf16); k_pool, v_pool:
    [num_slots, Hkv, D] BF16; kv_indptr [B+1], kv_indices [nnz] int32.
    ``num_splits > 0`` evaluates O through the split-merge formulation.
    ``pairs``: optional int array [n, 2] of (b, h) to evaluate; other rows of the
    outputs are left as zeros (NaN for o_f64 / lse).
    ``window > 0`` attends to the last ``window`` positions of each sequence only;
    ``sinks`` ([Hq] floats) adds a per-head sink logit to every softmax denominator.
    FP8 pools (uint8 / float8_e4m3fn e4m3 codes) take the values
    ``k_descale * e4m3(code)`` and ``v_descale * e4m3(code)``; with BF16 pools the
    descales are not used.
    """
    lib = _load()
    qa, ga = _u16(q), (None if gate_t is None else _u16(gate_t))
    (ka, kfp8), (va, vfp8) = _kv(k_pool), _kv(v_pool)
    assert kfp8 == vfp8, "K and V pools must have the same element type"
    ip, ix = _i32(kv_indptr), _i32(kv_indices)
    B, Hq, D = qa.shape
    num_slots, Hkv, Dk = ka.shape
    assert Dk == D and va.shape == ka.shape and ip.shape == (B + 1,)
    pr = None
    n_pairs = 0
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        n_pairs = pr.shape[0]
    o_f64 = np.full((B, Hq, D), np.nan) if "o_f64" in want else None
    o_bf = np.zeros((B, Hq, D), np.uint16) if "o_bf16" in want else None
    out = np.zeros((B, Hq, D), np.uint16) if ("out" in want and ga is not None) else None
    lse = np.full((B, Hq), np.nan) if "lse" in want else None
    sk = None
    if sinks is not None:
        sk = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64).reshape(-1))
        assert sk.shape == (Hq,)
    rc = lib.oracle_decode(
        _ptr(qa, ctypes.c_uint16), _ptr(ga, ctypes.c_uint16), ka.ctypes.data_as(ctypes.c_void_p),
        va.ctypes.data_as(ctypes.c_void_p), int(kfp8), float(k_descale), float(v_descale), _ptr(ip, ctypes.c_int32), _ptr(ix, ctypes.c_int32),
        int(num_slots), int(B), int(Hq), int(Hkv), int(D), float(scale), int(num_splits),
        int(window), _ptr(sk, ctypes.c_double), _ptr(pr, ctypes.c_int32), int(n_pairs), _ptr(o_f64, ctypes.c_double),
        _ptr(o_bf, ctypes.c_uint16), _ptr(out, ctypes.c_uint16), _ptr(lse, ctypes.c_double),
        int(nthreads))
    if rc != ORACLE_OK:
        raise ValueError("oracle_decode rejected its inputs (status %d)" % rc)
    return DecodeResult(o_f64, o_bf, out, lse)


def qk_norm_rope_kv_write(qgkv, w_q, w_k, eps: float, cos_t, sin_t, rope_dim: int, slots, k_pool, v_pool,
                          Hq: int, Hkv: int, D: int):
    """The step before attention, in FP64 with one BF16 rounding per output.

    qgkv: [B, (2 Hq + 2 Hkv) * D] BF16 rows [q | gate | k | v]; w_q / w_k: [D] BF16 or
    None (no norm); cos_t / sin_t: [B, rope_dim] BF16; slots: [B] int32.  Returns
    (q_out [B, Hq, D], gate_out [B, Hq, D], k_pool, v_pool) as uint16 bit arrays; the
    pools are copies of the given ones with the new rows written."""
    lib = _load()
    x = _u16(qgkv)
    B = x.shape[0]
    x = x.reshape(B, -1)
    wq = None if w_q is None else _u16(w_q)
    wk = None if w_k is None else _u16(w_k)
    cs = _u16(cos_t).reshape(B, -1) if rope_dim else np.zeros((B, 0), np.uint16)
    sn = _u16(sin_t).reshape(B, -1) if rope_dim else np.zeros((B, 0), np.uint16)
    sl = _i32(slots)
    kp = _u16(k_pool).copy()
    vp = _u16(v_pool).copy()
    qo = np.zeros((B, Hq, D), np.uint16)
    go = np.zeros((B, Hq, D), np.uint16)
    rc = lib.oracle_qk_norm_rope_kv_write(
        _ptr(x, ctypes.c_uint16), int(x.shape[1]), _ptr(wq, ctypes.c_uint16), _ptr(wk, ctypes.c_uint16),
        float(eps), _ptr(cs, ctypes.c_uint16), _ptr(sn, ctypes.c_uint16), int(rope_dim),
        _ptr(sl, ctypes.c_int32), _ptr(qo, ctypes.c_uint16), _ptr(go, ctypes.c_uint16),
        _ptr(kp, ctypes.c_uint16), _ptr(vp, ctypes.c_uint16), int(kp.shape[0]), int(B), int(Hq), int(Hkv), int(D))
    if rc != ORACLE_OK:
        raise ValueError("oracle_qk_norm_rope_kv_write rejected its inputs (status %d)" % rc)
    return qo, go, kp, vp


def prefill(q, gate_t, k, v, scale: float, causal: bool = True, kv_lens=None, rows=None,
            want=("o_f64", "o_bf16", "out", "lse"), nthreads: int = 0) -> DecodeResult:
    """Gated SDPA for prefill / extend in FP64 (cuDNN FE-OSS "Gated Attention Block
    (SM107)", Overview stages (4)-(5), fuse_gate).

    q, gate_t: [B, Sq, Hq, D] BF16; k, v: [B, Skv, Hkv, D] BF16.  With ``causal`` key j
    is visible to query i when j <= i + (L - Sq), L = kv_lens[b] (Skv when None);
    keys j >= L are never visible.  ``rows``: optional int array [n, 3] of (b, i, h) to
    evaluate; other rows of the outputs are left as zeros (NaN for o_f64 / lse).
    Returns o_f64 / o_bf16 / out [B, Sq, Hq, D] and lse [B, Hq, Sq] (natural log)."""
    lib = _load()
    qa, ka, va = _u16(q), _u16(k), _u16(v)
    ga = None if gate_t is None else _u16(gate_t)
    B, Sq, Hq, D = qa.shape
    Bk, Skv, Hkv, Dk = ka.shape
    assert Bk == B and Dk == D and va.shape == ka.shape
    kl = None if kv_lens is None else _i32(kv_lens)
    rr, n_rows = None, 0
    if rows is not None:
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        n_rows = rr.shape[0]
    o_f64 = np.full((B, Sq, Hq, D), np.nan) if "o_f64" in want else None
    o_bf = np.zeros((B, Sq, Hq, D), np.uint16) if "o_bf16" in want else None
    out = np.zeros((B, Sq, Hq, D), np.uint16) if ("out" in want and ga is not None) else None
    lse = np.full((B, Hq, Sq), np.nan) if "lse" in want else None
    rc = lib.oracle_prefill(
        _ptr(qa, ctypes.c_uint16), _ptr(ga, ctypes.c_uint16), _ptr(ka, ctypes.c_uint16), _ptr(va, ctypes.c_uint16),
        _ptr(kl, ctypes.c_int32), int(B), int(Sq), int(Skv), int(Hq), int(Hkv), int(D), float(scale),
        1 if causal else 0, _ptr(rr, ctypes.c_int32), int(n_rows), _ptr(o_f64, ctypes.c_double),
        _ptr(o_bf, ctypes.c_uint16), _ptr(out, ctypes.c_uint16), _ptr(lse, ctypes.c_double), int(nthreads))
    if rc != ORACLE_OK:
        raise ValueError("oracle_prefill rejected its inputs (status %d)" % rc)
    return DecodeResult(o_f64, o_bf, out, lse)
