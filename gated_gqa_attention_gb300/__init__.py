"""gated_gqa_attention_gb300 -- gated split-KV GQA decode attention for GB300.

A thin ctypes binding over the C ABI in ``include/gda.h`` (``lib/libgda.so``).
Every step of the computation runs in the library's CUDA kernels; this module
only checks tensor metadata, passes device pointers and the current CUDA stream,
and turns status codes into exceptions.  There is no CPU fallback: without the
built library every call raises.

    out = decode(q, gate, k_pool, v_pool, kv_indptr, kv_indices, scale=1/16)

computes, per sequence b and query head h (FreeToken PR #781 "Fuse the BF16
attention output sigmoid gate into the existing Triton decode stage2"):

    O   = softmax(scale * q[b,h] K[rows_b, h // G]^T) V[rows_b, h // G]
    out = bf16( bf16(O) * bf16(sigmoid(gate[b,h])) )     (round-to-nearest-even)

K/V pools of dtype torch.float8_e4m3fn (or uint8 e4m3 codes) select the FP8-cache
kernels; their values are ``k_descale * e4m3(code)`` and ``v_descale * e4m3(code)``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "load", "decode", "decode_ex", "decode_noalloc", "decode_step_host", "StepHost", "step_layout", "small_path_cluster", "auto_splits", "pack_step", "STEP_MAP_IN", "STEP_MAP_OUT", "prefill", "prefill_read_error", "qk_norm_rope_kv_write", "gate", "workspace_bytes", "workspace_init", "reserve",
    "read_error", "debug_wait_limit", "timing_begin", "timing_end", "status_str", "version", "GdaError", "VARIANT_AUTO", "VARIANT_MMA",
    "VARIANT_SIMT", "VARIANT_TMA", "MAX_SPLITS", "LIB_PATH", "KV_BF16", "KV_E4M3",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libgda.so")

VARIANT_AUTO, VARIANT_MMA, VARIANT_SIMT, VARIANT_TMA = 0, 1, 2, 3
KV_BF16, KV_E4M3 = 0, 1
MAX_SPLITS = 256
NOALLOC_SCRATCH_BYTES = 16 << 20
DEVERR_INDEX, DEVERR_TIMEOUT = 0x1, 0x2

_lock = threading.Lock()
_lib = None


class GdaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class _Args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p), ("kv_indptr", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_float), ("num_splits", ctypes.c_int), ("fuse_gate", ctypes.c_int),
        ("check_indices", ctypes.c_int), ("variant", ctypes.c_int), ("min_chunk", ctypes.c_int),
        ("window", ctypes.c_int), ("sinks", ctypes.c_void_p), ("kv_dtype", ctypes.c_int),
        ("k_descale", ctypes.c_float), ("v_descale", ctypes.c_float), ("max_len", ctypes.c_int),
        ("total_len", ctypes.c_int64),
    ]


def load(path: Optional[str] = None):
    """Load the C-ABI library (raises when it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                "libgda.so is not built (%s); run `python -m gated_gqa_attention_gb300.build`" % p)
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.gda_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        lib.gda_workspace_bytes.restype = ctypes.c_size_t
        lib.gda_workspace_init.argtypes = [vp, ctypes.c_size_t, vp]
        lib.gda_workspace_init.restype = i32
        lib.gda_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp]
        lib.gda_decode.restype = i32
        lib.gda_decode_ex.argtypes = [ctypes.POINTER(_Args), vp, ctypes.c_size_t, vp]
        lib.gda_decode_ex.restype = i32
        lib.gda_decode_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, f32, i32, vp]
        lib.gda_decode_e4m3.restype = i32
        lib.gda_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, vp]
        lib.gda_prefill.restype = i32
        lib.gda_prefill_read_error.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_uint32)]
        lib.gda_prefill_read_error.restype = i32
        lib.gda_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp]
        lib.gda_decode_noalloc.restype = i32
        lib.gda_qk_norm_rope_kv_write.argtypes = [vp, i64, vp, vp, f32, vp, vp, i32, vp, i64, vp, vp, vp, vp,
                                                  i32, i32, i32, i32, vp]
        lib.gda_qk_norm_rope_kv_write.restype = i32
        lib.gda_small_path_cluster.argtypes = [i64, i32]
        lib.gda_small_path_cluster.restype = i32
        lib.gda_auto_splits.argtypes = [i32, i32, i32, i32, i32, i64]
        lib.gda_auto_splits.restype = i32
        lib.gda_step_layout.argtypes = [i32, i32, i32, i64, ctypes.POINTER(ctypes.c_size_t)]
        lib.gda_step_layout.restype = ctypes.c_size_t
        lib.gda_decode_step_host.argtypes = [vp, vp, ctypes.c_size_t, vp, vp, i32, f32, f32, vp, vp, i32, i32, i32,
                                             i32, i64, f32, i32, i32, i32, vp]
        lib.gda_decode_step_host.restype = i32
        lib.gda_reserve.argtypes = [i32, i32, i32, i32, i32]
        lib.gda_reserve.restype = i32
        lib.gda_gate.argtypes = [vp, vp, vp, i64, vp]
        lib.gda_gate.restype = i32
        lib.gda_read_error.argtypes = [vp, vp, i32, ctypes.POINTER(ctypes.c_uint32)]
        lib.gda_read_error.restype = i32
        lib.gda_status_str.argtypes = [i32]
        lib.gda_status_str.restype = ctypes.c_char_p
        lib.gda_timing_begin.argtypes = [i32]
        lib.gda_timing_begin.restype = i32
        lib.gda_timing_end.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]
        lib.gda_timing_end.restype = i32
        lib.gda_version.argtypes = []
        lib.gda_version.restype = i32
        lib.gda_debug_wait_limit.argtypes = [i64]
        lib.gda_debug_wait_limit.restype = i32
        _lib = lib
        return lib


def status_str(status: int) -> str:
    return load().gda_status_str(int(status)).decode()


def version() -> int:
    return int(load().gda_version())


def _check(rc: int):
    if rc != 0:
        raise GdaError(rc, status_str(rc))


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_tensor(name, t, dtype, ndim=None, device=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))


def workspace_bytes(B: int, Hq: int, Hkv: int, D: int, num_splits: int = 0) -> int:
    """Bytes of workspace decode_ex needs (0 for invalid sizes)."""
    return int(load().gda_workspace_bytes(int(B), int(Hq), int(Hkv), int(D), int(num_splits)))


def workspace_init(workspace, stream=None):
    """Zero a caller-owned workspace's header (its device error word)."""
    _check(load().gda_workspace_init(ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def reserve(max_B: int, Hq: int = 16, Hkv: int = 2, D: int = 256, max_splits: int = 0):
    """Grow the library's internal workspace on the current device ahead of graph capture."""
    _check(load().gda_reserve(int(max_B), int(Hq), int(Hkv), int(D), int(max_splits)))


def _kv_dtype(k_pool) -> int:
    """KV_E4M3 for float8_e4m3fn / uint8 pools, else KV_BF16."""
    import torch
    return KV_E4M3 if isinstance(k_pool, torch.Tensor) and k_pool.dtype in (torch.float8_e4m3fn, torch.uint8) \
        else KV_BF16


def _decode_checks(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, out):
    """Checks tensor metadata; returns the pools' element type (KV_BF16 or KV_E4M3)."""
    import torch
    _check_tensor("q", q, torch.bfloat16, 3)
    dev = q.device
    if gate_t is not None:
        _check_tensor("gate", gate_t, torch.bfloat16, 3, dev)
        if gate_t.shape != q.shape:
            raise ValueError("gate must have q's shape")
    kv = _kv_dtype(k_pool)
    kdt = k_pool.dtype if kv == KV_E4M3 else torch.bfloat16
    _check_tensor("k_pool", k_pool, kdt, 3, dev)
    _check_tensor("v_pool", v_pool, kdt, 3, dev)
    if v_pool.shape != k_pool.shape:
        raise ValueError("k_pool and v_pool must have the same shape")
    _check_tensor("kv_indptr", kv_indptr, torch.int32, 1, dev)
    _check_tensor("kv_indices", kv_indices, torch.int32, 1, dev)
    if kv_indptr.numel() != q.shape[0] + 1:
        raise ValueError("kv_indptr must have B + 1 entries")
    if k_pool.shape[2] != q.shape[2]:
        raise ValueError("head dims of q and the pools differ")
    if out is not None:
        _check_tensor("out", out, torch.bfloat16, 3, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    return kv


def decode(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, out=None, scale: Optional[float] = None,
           num_splits: int = 0, stream=None, k_descale: float = 1.0, v_descale: float = 1.0):
    """Gated GQA decode attention through ``gda_decode`` (library-owned workspace).

    q, gate_t: [B, Hq, D] bf16; k_pool, v_pool: [num_slots, Hkv, D] bf16, or
    float8_e4m3fn / uint8 e4m3 codes (then ``gda_decode_e4m3`` with the descales);
    kv_indptr: [B+1] int32; kv_indices: [nnz] int32 (all CUDA, contiguous).
    ``num_splits <= 0`` lets the kernel plan the splits on the device."""
    import torch
    kv = _decode_checks(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, out)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    if kv == KV_E4M3:
        _check(load().gda_decode_e4m3(_ptr(q), _ptr(gate_t), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indptr),
                                      _ptr(kv_indices), _ptr(out), B, Hq, Hkv, D, float(scale), float(k_descale),
                                      float(v_descale), int(num_splits), _stream(stream)))
        return out
    _check(load().gda_decode(_ptr(q), _ptr(gate_t), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indptr),
                             _ptr(kv_indices), _ptr(out), B, Hq, Hkv, D, float(scale), int(num_splits),
                             _stream(stream)))
    return out


def decode_noalloc(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, out, scale: Optional[float] = None,
                   num_splits: int = 0, stream=None):
    """``gda_decode_noalloc``: the same result as decode() for callers that must not
    allocate device memory.  ``out`` must be given (this call allocates nothing);
    the library's fixed scratch area (NOALLOC_SCRATCH_BYTES per device) replaces the
    workspace, so calls that may overlap on the GPU must not use it concurrently."""
    if _decode_checks(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, out) != KV_BF16:
        raise TypeError("decode_noalloc serves bf16 pools only")
    if out is None:
        raise ValueError("decode_noalloc needs a preallocated out tensor")
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    _check(load().gda_decode_noalloc(_ptr(q), _ptr(gate_t), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indptr),
                                     _ptr(kv_indices), _ptr(out), B, Hq, Hkv, D, float(scale), int(num_splits),
                                     _stream(stream)))
    return out


def auto_splits(B: int, heads: int, grid: int, lmax: int, total: int, min_chunk: int = 0) -> int:
    """``gda_auto_splits``: the automatic split rule for B sequences (longest lmax,
    total ``total`` positions), ``heads`` segments per sequence, ``grid`` stage-1 CTAs:
    the uniform split count, 0 for the stream schedule, -1 for invalid arguments."""
    return int(load().gda_auto_splits(int(B), int(heads), int(grid), int(min_chunk), int(lmax), int(total)))


def small_path_cluster(pairs: int, max_len: int) -> int:
    """``gda_small_path_cluster``: the cluster size (8, 4 or 2) a bf16 decode of
    ``pairs`` = B * Hkv (sequence, KV head) pairs with the length bound ``max_len``
    takes through the one-kernel path on the current device, or 0 (split path)."""
    return int(load().gda_small_path_cluster(int(pairs), int(max_len)))


def step_layout(B: int, Hq: int, D: int, nnz: int):
    """``gda_step_layout``: (offsets of q, gate, kv_indptr, kv_indices; total bytes) of
    one decode step's inputs packed into a single block."""
    off = (ctypes.c_size_t * 4)()
    total = load().gda_step_layout(int(B), int(Hq), int(D), int(nnz), off)
    if total == 0:
        raise ValueError("gda_step_layout: sizes out of range")
    return tuple(int(x) for x in off), int(total)


def pack_step(host_in, q, gate_t, kv_indptr, kv_indices):
    """Write one step's CPU tensors into the packed host block ``host_in`` (a uint8
    CPU tensor, pinned for asynchronous copies) at the offsets of step_layout."""
    import torch
    B, Hq, D = q.shape
    nnz = kv_indices.numel()
    off, total = step_layout(B, Hq, D, nnz)
    if host_in.dtype != torch.uint8 or host_in.device.type != "cpu" or host_in.numel() < total:
        raise ValueError("host_in must be a CPU uint8 tensor of at least %d bytes" % total)
    parts = ((q, torch.bfloat16), (gate_t, torch.bfloat16), (kv_indptr, torch.int32), (kv_indices, torch.int32))
    for (t, dt), o in zip(parts, off):
        if t.dtype != dt:
            raise TypeError("pack_step: expected %s, got %s" % (dt, t.dtype))
        b = t.detach().cpu().contiguous().view(torch.uint8).reshape(-1)
        host_in[o:o + b.numel()].copy_(b)
    return host_in


STEP_MAP_IN, STEP_MAP_OUT = 0x1, 0x2


class StepHost:
    """A decode step bound to fixed buffers: the packed pinned inputs ``host_in``
    (step_layout), the device staging ``dev_in`` / ``dev_out`` (None when mapped) and
    the pinned result ``host_out`` [B, Hq, D] bf16.  Everything is checked and
    marshalled once here; each call is then one ``gda_decode_step_host`` call (copy
    in, decode, copy out, wait).  ``map_in`` / ``map_out``: the kernels read host_in /
    write host_out in place over the host-device link instead of copies."""

    def __init__(self, host_in, dev_in, k_pool, v_pool, dev_out, host_out, B: int, Hq: int, nnz: int,
                 scale: Optional[float] = None, num_splits: int = 0, map_in: bool = False, map_out: bool = False,
                 synchronize: bool = True, stream=None, k_descale: float = 1.0, v_descale: float = 1.0):
        import torch
        kv = _kv_dtype(k_pool)
        dt = torch.bfloat16 if kv == KV_BF16 else k_pool.dtype
        _check_tensor("k_pool", k_pool, dt, 3)
        _check_tensor("v_pool", v_pool, dt, 3, k_pool.device)
        Hkv, D = k_pool.shape[1], k_pool.shape[2]
        _, total = step_layout(B, Hq, D, nnz)
        if host_in.device.type != "cpu" or host_out.device.type != "cpu":
            raise ValueError("host_in and host_out must be CPU tensors")
        if host_in.numel() * host_in.element_size() < total:
            raise ValueError("host_in holds fewer than %d bytes" % total)
        if not map_in and (dev_in is None or not dev_in.is_cuda or dev_in.numel() * dev_in.element_size() < total):
            raise ValueError("dev_in must be a CUDA tensor of at least %d bytes" % total)
        if tuple(host_out.shape) != (B, Hq, D) or host_out.dtype != torch.bfloat16:
            raise ValueError("host_out must be a [B, Hq, D] bf16 tensor")
        if not map_out and (dev_out is None or tuple(dev_out.shape) != (B, Hq, D)):
            raise ValueError("dev_out must be a [B, Hq, D] CUDA tensor")
        if scale is None:
            scale = 1.0 / (D ** 0.5)
        vp = ctypes.c_void_p
        flags = (STEP_MAP_IN if map_in else 0) | (STEP_MAP_OUT if map_out else 0)
        self.host_in, self.dev_in, self.dev_out, self.host_out = host_in, dev_in, dev_out, host_out
        self.k_pool, self.v_pool = k_pool, v_pool   # kept alive with the call's pointers
        self.in_bytes, self.out_bytes = total, host_out.numel() * 2
        self._f = load().gda_decode_step_host
        self._args = (vp(_ptr(host_in)), vp(_ptr(dev_in)), total, vp(_ptr(k_pool)), vp(_ptr(v_pool)),
                      kv, float(k_descale), float(v_descale), vp(_ptr(dev_out)), vp(_ptr(host_out)), int(B), int(Hq),
                      int(Hkv), int(D), int(nnz), float(scale), int(num_splits), flags, 1 if synchronize else 0,
                      _stream(stream))

    def __call__(self):
        rc = self._f(*self._args)
        if rc != 0:
            _check(rc)
        return self.host_out


def decode_step_host(host_in, dev_in, k_pool, v_pool, dev_out, host_out, B: int, Hq: int, nnz: int,
                     scale: Optional[float] = None, num_splits: int = 0, map_in: bool = False,
                     map_out: bool = False, synchronize: bool = True, stream=None, k_descale: float = 1.0,
                     v_descale: float = 1.0):
    """``gda_decode_step_host`` once (see StepHost, which keeps the marshalled call for
    repeated steps)."""
    return StepHost(host_in, dev_in, k_pool, v_pool, dev_out, host_out, B, Hq, nnz, scale=scale,
                    num_splits=num_splits, map_in=map_in, map_out=map_out, synchronize=synchronize,
                    stream=stream, k_descale=k_descale, v_descale=v_descale)()


def decode_ex(q, gate_t, k_pool, v_pool, kv_indptr, kv_indices, out=None, *, workspace=None,
              scale: Optional[float] = None, num_splits: int = 0, fuse_gate: bool = True, lse=None,
              check_indices: bool = False, variant: int = VARIANT_AUTO, min_chunk: int = 0,
              window: int = 0, sinks=None, stream=None, k_descale: float = 1.0, v_descale: float = 1.0,
              max_len: int = 0, total_len: int = 0):
    """``gda_decode_ex``: caller workspace (allocated here when None), optional LSE
    output, the unfused first half (``fuse_gate=False``), device index checks, the
    stage-1 variant, a sliding window (last ``window`` positions), per-head
    attention sinks (``sinks``: [Hq] float32 CUDA tensor of logits), for e4m3
    pools the per-tensor descales, and ``max_len``: a host-known bound on every
    sequence's length (0: none), which lets small batches run as one cluster kernel,
    and ``total_len``: the batch's exact number of KV positions (kv_indptr[B], 0: not
    given); with both, the split count is chosen on the host (``auto_splits``)."""
    import torch
    kv = _decode_checks(q, gate_t if fuse_gate else None, k_pool, v_pool, kv_indptr, kv_indices, out)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 2, q.device)
    if sinks is not None:
        _check_tensor("sinks", sinks, torch.float32, 1, q.device)
        if sinks.numel() != q.shape[1]:
            raise ValueError("sinks must have Hq entries")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    nbytes = workspace_bytes(B, Hq, Hkv, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
        workspace_init(workspace, stream)
    a = _Args(q=_ptr(q), gate=_ptr(gate_t) if fuse_gate else None, k_pool=_ptr(k_pool),
              v_pool=_ptr(v_pool), kv_indptr=_ptr(kv_indptr), kv_indices=_ptr(kv_indices),
              out=_ptr(out), lse=_ptr(lse), num_slots=int(k_pool.shape[0]), B=B, Hq=Hq, Hkv=Hkv, D=D,
              scale=float(scale), num_splits=int(num_splits), fuse_gate=1 if fuse_gate else 0,
              check_indices=1 if check_indices else 0, variant=int(variant), min_chunk=int(min_chunk),
              window=int(window), sinks=_ptr(sinks), kv_dtype=kv, k_descale=float(k_descale),
              v_descale=float(v_descale), max_len=int(max_len), total_len=int(total_len))
    _check(load().gda_decode_ex(ctypes.byref(a), ctypes.c_void_p(workspace.data_ptr()),
                                workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def prefill(q, gate_t, k, v, *, kv_lens=None, out=None, lse=None, scale: Optional[float] = None,
            causal: bool = True, error_word=None, stream=None):
    """Prefill / extend gated SDPA through ``gda_prefill`` (tcgen05 kernel).

    q, gate_t: [B, Sq, Hq, D] bf16 (gate_t None: out = bf16(O)); k, v: [B, Skv, Hkv, D]
    bf16; kv_lens: [B] int32 or None; lse: [B, Hq, Sq] float32 or None; error_word:
    a 1-element int32/uint32 CUDA tensor or None (the library's word)."""
    import torch
    _check_tensor("q", q, torch.bfloat16, 4)
    dev = q.device
    B, Sq, Hq, D = q.shape
    if gate_t is not None:
        _check_tensor("gate", gate_t, torch.bfloat16, 4, dev)
        if gate_t.shape != q.shape:
            raise ValueError("gate must have q's shape")
    _check_tensor("k", k, torch.bfloat16, 4, dev)
    _check_tensor("v", v, torch.bfloat16, 4, dev)
    if v.shape != k.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Skv, Hkv, D] with q's B and D")
    Skv, Hkv = k.shape[1], k.shape[2]
    if kv_lens is not None:
        _check_tensor("kv_lens", kv_lens, torch.int32, 1, dev)
        if kv_lens.numel() != B:
            raise ValueError("kv_lens must have B entries")
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, 3, dev)
        if tuple(lse.shape) != (B, Hq, Sq):
            raise ValueError("lse must be [B, Hq, Sq]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_tensor("out", out, torch.bfloat16, 4, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    _check(load().gda_prefill(_ptr(q), _ptr(gate_t), _ptr(k), _ptr(v), _ptr(kv_lens), _ptr(out), _ptr(lse),
                              B, Sq, Skv, Hq, Hkv, D, float(scale), 1 if causal else 0, _ptr(error_word),
                              _stream(stream)))
    return out


def prefill_read_error(clear: bool = True, stream=None) -> int:
    """The library's prefill error word on the current device (synchronises)."""
    w = ctypes.c_uint32(0)
    rc = load().gda_prefill_read_error(_stream(stream), 1 if clear else 0, ctypes.byref(w))
    if rc not in (0, -9):
        _check(rc)
    return int(w.value)


def qk_norm_rope_kv_write(qgkv, slots, k_pool, v_pool, Hq: int, w_q_norm=None, w_k_norm=None, eps: float = 1e-6,
                          cos=None, sin=None, rope_dim: int = 0, q_out=None, gate_out=None, stream=None):
    """The step before attention: q_out = rope(rmsnorm(q)), the token's K row
    rope(rmsnorm(k)) and V row written into the pools at ``slots``, and the gate
    copied out.  qgkv: [B, (2 Hq + 2 Hkv) * D] bf16 rows [q | gate | k | v]."""
    import torch
    _check_tensor("qgkv", qgkv, torch.bfloat16, 2)
    dev = qgkv.device
    _check_tensor("slots", slots, torch.int32, 1, dev)
    _check_tensor("k_pool", k_pool, torch.bfloat16, 3, dev)
    _check_tensor("v_pool", v_pool, torch.bfloat16, 3, dev)
    B = qgkv.shape[0]
    num_slots, Hkv, D = k_pool.shape
    for name, t in (("w_q_norm", w_q_norm), ("w_k_norm", w_k_norm), ("cos", cos), ("sin", sin)):
        if t is not None:
            _check_tensor(name, t, torch.bfloat16, device=dev)
    if q_out is None:
        q_out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    if gate_out is None:
        gate_out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    _check(load().gda_qk_norm_rope_kv_write(
        _ptr(qgkv), qgkv.shape[1], _ptr(w_q_norm), _ptr(w_k_norm), float(eps), _ptr(cos), _ptr(sin),
        int(rope_dim), _ptr(slots), num_slots, _ptr(q_out), _ptr(gate_out), _ptr(k_pool), _ptr(v_pool),
        B, int(Hq), Hkv, D, _stream(stream)))
    return q_out, gate_out


def gate(o, gate_t, out=None, stream=None):
    """Standalone gate: out = bf16(o * bf16(sigmoid(gate))) element by element."""
    import torch
    _check_tensor("o", o, torch.bfloat16)
    _check_tensor("gate", gate_t, torch.bfloat16, device=o.device)
    if gate_t.shape != o.shape:
        raise ValueError("gate must have o's shape")
    if out is None:
        out = torch.empty_like(o)
    _check(load().gda_gate(_ptr(o), _ptr(gate_t), _ptr(out), o.numel(), _stream(stream)))
    return out


def timing_begin(max_calls: int):
    """Time the stage-1 kernel of the next ``max_calls`` decode calls with CUDA events."""
    _check(load().gda_timing_begin(int(max_calls)))


def timing_end():
    """(number of timed stage-1 launches, their total milliseconds); synchronises."""
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    _check(load().gda_timing_end(ctypes.byref(n), ctypes.byref(ms)))
    return int(n.value), float(ms.value)


def debug_wait_limit(cycles: int):
    """``gda_debug_wait_limit``: the pipeline wait limit (SM cycles) of later calls;
    a short limit makes the waiting kernels take their timeout path (failure-path
    tests only); ``cycles <= 0`` restores the default."""
    _check(load().gda_debug_wait_limit(int(cycles)))


def read_error(workspace=None, clear: bool = True, stream=None) -> int:
    """The device error word of a workspace (or of the internal one); synchronises."""
    w = ctypes.c_uint32(0)
    ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    rc = load().gda_read_error(ptr, _stream(stream), 1 if clear else 0, ctypes.byref(w))
    if rc not in (0, -9):
        _check(rc)
    return int(w.value)
