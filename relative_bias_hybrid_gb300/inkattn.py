"""Thin ctypes binding of libinkattn.so (declared in include/inkattn.h).

Argument marshalling only: the entry points keep their C names, the params structs
mirror the C structs field by field, and the ``*_params`` helpers fill them from
torch tensors (device pointers, sizes).  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation behind these calls, and
loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libinkattn.so")

INKATTN_OK = 0
INKATTN_ERR_INVALID_ARG = 1
INKATTN_ERR_UNSUPPORTED = 2
INKATTN_ERR_CUDA = 3
INKATTN_ERR_DEVICE_TIMEOUT = 4
INKATTN_ERR_DEVICE_BOUNDS = 5
INKATTN_DTYPE_BF16 = 0
INKATTN_DTYPE_F32 = 1
INKATTN_KV_BF16 = 0
INKATTN_KV_E4M3 = 1

_c_i32 = ctypes.c_int32
_c_ptr = ctypes.c_void_p


class PrologueParams(ctypes.Structure):
    """inkattn_prologue_params."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("B", _c_i32), ("N_tok", _c_i32), ("max_seqlen_q", _c_i32), ("Hq", _c_i32), ("Hkv", _c_i32),
        ("head_dim", _c_i32), ("block_size", _c_i32), ("num_blocks", _c_i32),
        ("num_state_slots", _c_i32), ("eps", ctypes.c_float),
        ("q", _c_ptr), ("k", _c_ptr), ("v", _c_ptr),
        ("conv_w_k", _c_ptr), ("conv_w_v", _c_ptr), ("q_norm_w", _c_ptr), ("k_norm_w", _c_ptr),
        ("cu_seqlens_q", _c_ptr), ("state_slot", _c_ptr), ("slot_mapping", _c_ptr),
        ("conv_state_k", _c_ptr), ("conv_state_v", _c_ptr), ("q_out", _c_ptr),
        ("k_cache", _c_ptr), ("v_cache", _c_ptr), ("kv_dtype", _c_i32), ("k_scale", _c_ptr),
        ("v_scale", _c_ptr), ("dev_status", _c_ptr),
    ]


class AttnParams(ctypes.Structure):
    """inkattn_attn_params."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("B", _c_i32), ("N_tok", _c_i32), ("max_seqlen_q", _c_i32), ("max_seqlen_k", _c_i32),
        ("Hq", _c_i32), ("Hkv", _c_i32), ("head_dim", _c_i32), ("block_size", _c_i32),
        ("num_blocks", _c_i32), ("max_blocks_per_seq", _c_i32), ("d_r", _c_i32),
        ("rel_extent", _c_i32), ("window", _c_i32), ("out_dtype", _c_i32),
        ("softmax_scale", ctypes.c_float), ("log_scale_base", ctypes.c_float),
        ("q", _c_ptr), ("r", _c_ptr), ("P", _c_ptr), ("k_cache", _c_ptr), ("v_cache", _c_ptr),
        ("kv_dtype", _c_i32), ("k_scale", _c_ptr), ("v_scale", _c_ptr), ("cu_seqlens_q", _c_ptr), ("seqlen_k", _c_ptr), ("block_table", _c_ptr),
        ("out", _c_ptr), ("lse", _c_ptr), ("dev_status", _c_ptr),
    ]


class OutputConvParams(ctypes.Structure):
    """inkattn_output_conv_params."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("B", _c_i32), ("N_tok", _c_i32), ("max_seqlen_q", _c_i32), ("D", _c_i32),
        ("num_state_slots", _c_i32), ("eps", ctypes.c_float),
        ("y", _c_ptr), ("conv_w", _c_ptr), ("norm_w", _c_ptr), ("cu_seqlens_q", _c_ptr),
        ("state_slot", _c_ptr), ("conv_state", _c_ptr), ("residual", _c_ptr), ("h_out", _c_ptr),
        ("out", _c_ptr), ("dev_status", _c_ptr),
    ]


class QkvrParams(ctypes.Structure):
    """inkattn_qkvr_params."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("B", _c_i32), ("N_tok", _c_i32), ("max_seqlen_q", _c_i32), ("Hq", _c_i32), ("Hkv", _c_i32),
        ("head_dim", _c_i32), ("d_r", _c_i32), ("d_model", _c_i32), ("block_size", _c_i32),
        ("num_blocks", _c_i32), ("num_state_slots", _c_i32), ("eps", ctypes.c_float),
        ("x", _c_ptr), ("w", _c_ptr),
        ("conv_w_k", _c_ptr), ("conv_w_v", _c_ptr), ("q_norm_w", _c_ptr), ("k_norm_w", _c_ptr),
        ("cu_seqlens_q", _c_ptr), ("state_slot", _c_ptr), ("slot_mapping", _c_ptr),
        ("conv_state_k_in", _c_ptr), ("conv_state_v_in", _c_ptr),
        ("conv_state_k_out", _c_ptr), ("conv_state_v_out", _c_ptr),
        ("q_out", _c_ptr), ("r_out", _c_ptr), ("y_out", _c_ptr),
        ("k_cache", _c_ptr), ("v_cache", _c_ptr), ("kv_dtype", _c_i32), ("k_scale", _c_ptr),
        ("v_scale", _c_ptr), ("dev_status", _c_ptr),
    ]


class InkattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libinkattn.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER
            L.inkattn_status_string.argtypes = [ctypes.c_int]
            L.inkattn_status_string.restype = ctypes.c_char_p
            L.inkattn_abi_version.argtypes = []
            L.inkattn_abi_version.restype = ctypes.c_int
            L.inkattn_prologue.argtypes = [P(PrologueParams), _c_ptr]
            L.inkattn_prologue.restype = ctypes.c_int
            L.inkattn_prefill.argtypes = [P(AttnParams), _c_ptr]
            L.inkattn_prefill.restype = ctypes.c_int
            L.inkattn_decode_num_splits.argtypes = [P(AttnParams), ctypes.c_int]
            L.inkattn_decode_num_splits.restype = ctypes.c_int
            L.inkattn_decode_workspace_bytes.argtypes = [P(AttnParams), ctypes.c_int]
            L.inkattn_decode_workspace_bytes.restype = ctypes.c_size_t
            L.inkattn_decode.argtypes = [P(AttnParams), ctypes.c_int, _c_ptr, ctypes.c_size_t, _c_ptr]
            L.inkattn_decode.restype = ctypes.c_int
            L.inkattn_combine.argtypes = [P(AttnParams), ctypes.c_int, _c_ptr, ctypes.c_size_t, _c_ptr]
            L.inkattn_combine.restype = ctypes.c_int
            L.inkattn_decode_noalloc.argtypes = [P(AttnParams), ctypes.c_int, _c_ptr]
            L.inkattn_decode_noalloc.restype = ctypes.c_int
            L.inkattn_output_conv.argtypes = [P(OutputConvParams), _c_ptr]
            L.inkattn_output_conv.restype = ctypes.c_int
            L.inkattn_qkvr_prologue.argtypes = [P(QkvrParams), _c_ptr]
            L.inkattn_qkvr_prologue.restype = ctypes.c_int
            L.inkattn_prefill_workspace_bytes.argtypes = [P(AttnParams)]
            L.inkattn_prefill_workspace_bytes.restype = ctypes.c_size_t
            L.inkattn_prefill_e4m3.argtypes = [P(AttnParams), _c_ptr, ctypes.c_size_t, _c_ptr]
            L.inkattn_prefill_e4m3.restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().inkattn_status_string(int(status)).decode()


def abi_version() -> int:
    return int(lib().inkattn_abi_version())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str, raise_on_error: bool):
    if raise_on_error and status != INKATTN_OK:
        raise InkattnError(status, where)
    return status


# ------------------------------------------------------------------ entry points

def inkattn_prologue(p: PrologueParams, stream=None, raise_on_error=True) -> int:
    return _check(lib().inkattn_prologue(ctypes.byref(p), _stream(stream)), "inkattn_prologue",
                  raise_on_error)


def inkattn_prefill(p: AttnParams, stream=None, raise_on_error=True) -> int:
    return _check(lib().inkattn_prefill(ctypes.byref(p), _stream(stream)), "inkattn_prefill",
                  raise_on_error)


def inkattn_prefill_workspace_bytes(p: AttnParams) -> int:
    return int(lib().inkattn_prefill_workspace_bytes(ctypes.byref(p)))


def inkattn_prefill_e4m3(p: AttnParams, workspace: Optional[torch.Tensor], stream=None,
                         raise_on_error=True) -> int:
    ptr = workspace.data_ptr() if workspace is not None else None
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return _check(lib().inkattn_prefill_e4m3(ctypes.byref(p), ptr, nbytes, _stream(stream)),
                  "inkattn_prefill_e4m3", raise_on_error)


def inkattn_decode_num_splits(p: AttnParams, num_sms: int) -> int:
    return int(lib().inkattn_decode_num_splits(ctypes.byref(p), int(num_sms)))


def inkattn_decode_workspace_bytes(p: AttnParams, num_splits: int) -> int:
    return int(lib().inkattn_decode_workspace_bytes(ctypes.byref(p), int(num_splits)))


def inkattn_decode(p: AttnParams, num_splits: int, workspace: Optional[torch.Tensor], stream=None,
                   raise_on_error=True) -> int:
    ptr = workspace.data_ptr() if workspace is not None else None
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return _check(lib().inkattn_decode(ctypes.byref(p), int(num_splits), ptr, nbytes, _stream(stream)),
                  "inkattn_decode", raise_on_error)


def inkattn_combine(p: AttnParams, num_splits: int, workspace: Optional[torch.Tensor], stream=None,
                    raise_on_error=True) -> int:
    ptr = workspace.data_ptr() if workspace is not None else None
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return _check(lib().inkattn_combine(ctypes.byref(p), int(num_splits), ptr, nbytes, _stream(stream)),
                  "inkattn_combine", raise_on_error)


DECODE_NOALLOC_MAX_BYTES = 64 << 20


def inkattn_decode_noalloc(p: AttnParams, num_splits: int, stream=None, raise_on_error=True) -> int:
    """Decode + combine with the split partials in the library's static device buffer
    (no workspace argument, no allocation): for callers that cannot allocate device
    memory where they decode."""
    return _check(lib().inkattn_decode_noalloc(ctypes.byref(p), int(num_splits), _stream(stream)),
                  "inkattn_decode_noalloc", raise_on_error)


def inkattn_output_conv(p: OutputConvParams, stream=None, raise_on_error=True) -> int:
    return _check(lib().inkattn_output_conv(ctypes.byref(p), _stream(stream)), "inkattn_output_conv",
                  raise_on_error)


# ------------------------------------------------------------------ marshalling helpers

def inkattn_qkvr_prologue(p: QkvrParams, stream=None, raise_on_error=True) -> int:
    return _check(lib().inkattn_qkvr_prologue(ctypes.byref(p), _stream(stream)), "inkattn_qkvr_prologue",
                  raise_on_error)


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _kv_dtype(cache):
    """kv_dtype of a cache tensor: bf16 values, or E4M3 codes held as uint8."""
    if cache.dtype == torch.bfloat16:
        return INKATTN_KV_BF16, torch.bfloat16
    if cache.dtype == torch.uint8:
        return INKATTN_KV_E4M3, torch.uint8
    raise TypeError(f"KV cache: expected bfloat16 or uint8 (E4M3 codes), got {cache.dtype}")


def prologue_params(*, q, k, v, conv_w_k, conv_w_v, q_norm_w, k_norm_w, cu_seqlens_q, state_slot,
                    slot_mapping, conv_state_k, conv_state_v, q_out, k_cache, v_cache,
                    max_seqlen_q: int, eps: float = 1e-6, dev_status=None, k_scale=None,
                    v_scale=None) -> PrologueParams:
    """Fill an inkattn_prologue_params from torch tensors (see include/inkattn.h)."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    N, Hq, d = q.shape
    Hkv = k.shape[1] // d
    p = PrologueParams()
    p.struct_size = ctypes.sizeof(PrologueParams)
    p.B = cu_seqlens_q.numel() - 1
    p.N_tok = N
    p.max_seqlen_q = int(max_seqlen_q)
    p.Hq, p.Hkv, p.head_dim = Hq, Hkv, d
    p.block_size = k_cache.shape[2]
    p.num_blocks = k_cache.shape[0]
    p.num_state_slots = conv_state_k.shape[0]
    p.eps = float(eps)
    p.q = _ptr(q, bf, "q"); p.k = _ptr(k, bf, "k"); p.v = _ptr(v, bf, "v")
    p.conv_w_k = _ptr(conv_w_k, f32, "conv_w_k"); p.conv_w_v = _ptr(conv_w_v, f32, "conv_w_v")
    p.q_norm_w = _ptr(q_norm_w, f32, "q_norm_w"); p.k_norm_w = _ptr(k_norm_w, f32, "k_norm_w")
    p.cu_seqlens_q = _ptr(cu_seqlens_q, i32, "cu_seqlens_q")
    p.state_slot = _ptr(state_slot, i32, "state_slot")
    p.slot_mapping = _ptr(slot_mapping, i32, "slot_mapping")
    p.conv_state_k = _ptr(conv_state_k, bf, "conv_state_k")
    p.conv_state_v = _ptr(conv_state_v, bf, "conv_state_v")
    p.q_out = _ptr(q_out, bf, "q_out")
    p.kv_dtype, cache_dt = _kv_dtype(k_cache)
    p.k_cache = _ptr(k_cache, cache_dt, "k_cache"); p.v_cache = _ptr(v_cache, cache_dt, "v_cache")
    if p.kv_dtype == INKATTN_KV_E4M3:
        p.k_scale = _ptr(k_scale, f32, "k_scale"); p.v_scale = _ptr(v_scale, f32, "v_scale")
    p.dev_status = _ptr(dev_status, i32, "dev_status")
    return p


def attn_params(*, q, k_cache, v_cache, cu_seqlens_q, seqlen_k, block_table, out, max_seqlen_q: int,
                max_seqlen_k: int, r=None, P=None, rel_extent: int = 0, window: int = 0,
                softmax_scale: float = 0.0, log_scale_base: float = 0.0, lse=None,
                dev_status=None, k_scale=None, v_scale=None) -> AttnParams:
    """Fill an inkattn_attn_params from torch tensors (see include/inkattn.h)."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    N, Hq, d = q.shape
    p = AttnParams()
    p.struct_size = ctypes.sizeof(AttnParams)
    p.B = cu_seqlens_q.numel() - 1
    p.N_tok = N
    p.max_seqlen_q = int(max_seqlen_q)
    p.max_seqlen_k = int(max_seqlen_k)
    p.Hq, p.Hkv, p.head_dim = Hq, k_cache.shape[1], d
    p.block_size = k_cache.shape[2]
    p.num_blocks = k_cache.shape[0]
    p.max_blocks_per_seq = block_table.shape[1]
    p.d_r = r.shape[2] if r is not None else 0
    p.rel_extent = int(rel_extent)
    p.window = int(window)
    p.softmax_scale = float(softmax_scale)
    p.log_scale_base = float(log_scale_base)
    p.q = _ptr(q, bf, "q")
    p.r = _ptr(r, bf, "r") if rel_extent > 0 else None
    p.P = _ptr(P, f32, "P") if rel_extent > 0 else None
    p.kv_dtype, cache_dt = _kv_dtype(k_cache)
    p.k_cache = _ptr(k_cache, cache_dt, "k_cache"); p.v_cache = _ptr(v_cache, cache_dt, "v_cache")
    if p.kv_dtype == INKATTN_KV_E4M3:
        p.k_scale = _ptr(k_scale, f32, "k_scale"); p.v_scale = _ptr(v_scale, f32, "v_scale")
    p.cu_seqlens_q = _ptr(cu_seqlens_q, i32, "cu_seqlens_q")
    p.seqlen_k = _ptr(seqlen_k, i32, "seqlen_k")
    p.block_table = _ptr(block_table, i32, "block_table")
    if out.dtype == torch.float32:
        p.out_dtype = INKATTN_DTYPE_F32
    elif out.dtype == bf:
        p.out_dtype = INKATTN_DTYPE_BF16
    else:
        raise TypeError(f"out: expected bfloat16 or float32, got {out.dtype}")
    p.out = _ptr(out, None, "out")
    p.lse = _ptr(lse, f32, "lse")
    p.dev_status = _ptr(dev_status, i32, "dev_status")
    return p


def output_conv_params(*, y, conv_w, norm_w, cu_seqlens_q, state_slot, conv_state, residual, h_out,
                       out, max_seqlen_q: int, eps: float = 1e-6, dev_status=None) -> OutputConvParams:
    """Fill an inkattn_output_conv_params from torch tensors (see include/inkattn.h)."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    N, D = y.shape
    p = OutputConvParams()
    p.struct_size = ctypes.sizeof(OutputConvParams)
    p.B = cu_seqlens_q.numel() - 1
    p.N_tok = N
    p.max_seqlen_q = int(max_seqlen_q)
    p.D = D
    p.num_state_slots = conv_state.shape[0]
    p.eps = float(eps)
    p.y = _ptr(y, bf, "y")
    p.conv_w = _ptr(conv_w, f32, "conv_w")
    p.norm_w = _ptr(norm_w, f32, "norm_w")
    p.cu_seqlens_q = _ptr(cu_seqlens_q, i32, "cu_seqlens_q")
    p.state_slot = _ptr(state_slot, i32, "state_slot")
    p.conv_state = _ptr(conv_state, bf, "conv_state")
    p.residual = _ptr(residual, bf, "residual")
    p.h_out = _ptr(h_out, bf, "h_out")
    p.out = _ptr(out, bf, "out")
    p.dev_status = _ptr(dev_status, i32, "dev_status")
    return p


def qkvr_params(*, x, w, conv_w_k, conv_w_v, q_norm_w, k_norm_w, cu_seqlens_q, state_slot, slot_mapping,
                conv_state_k_in, conv_state_v_in, conv_state_k_out, conv_state_v_out, q_out, r_out,
                k_cache, v_cache, max_seqlen_q: int, eps: float = 1e-6, dev_status=None, k_scale=None,
                v_scale=None, y_out=None) -> QkvrParams:
    """Fill an inkattn_qkvr_params from torch tensors (see include/inkattn.h): x [N][d_model],
    w [F][d_model], q_out [N][Hq][128], r_out [N][Hq][d_r], y_out None or [N][F]."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    N, Hq, d = q_out.shape
    p = QkvrParams()
    p.struct_size = ctypes.sizeof(QkvrParams)
    p.B = cu_seqlens_q.numel() - 1
    p.N_tok = N
    p.max_seqlen_q = int(max_seqlen_q)
    p.Hq, p.Hkv, p.head_dim = Hq, k_cache.shape[1], d
    p.d_r = r_out.shape[2]
    p.d_model = x.shape[1]
    p.block_size = k_cache.shape[2]
    p.num_blocks = k_cache.shape[0]
    p.num_state_slots = conv_state_k_in.shape[0]
    p.eps = float(eps)
    p.x = _ptr(x, bf, "x"); p.w = _ptr(w, bf, "w")
    p.conv_w_k = _ptr(conv_w_k, f32, "conv_w_k"); p.conv_w_v = _ptr(conv_w_v, f32, "conv_w_v")
    p.q_norm_w = _ptr(q_norm_w, f32, "q_norm_w"); p.k_norm_w = _ptr(k_norm_w, f32, "k_norm_w")
    p.cu_seqlens_q = _ptr(cu_seqlens_q, i32, "cu_seqlens_q")
    p.state_slot = _ptr(state_slot, i32, "state_slot")
    p.slot_mapping = _ptr(slot_mapping, i32, "slot_mapping")
    p.conv_state_k_in = _ptr(conv_state_k_in, bf, "conv_state_k_in")
    p.conv_state_v_in = _ptr(conv_state_v_in, bf, "conv_state_v_in")
    p.conv_state_k_out = _ptr(conv_state_k_out, bf, "conv_state_k_out")
    p.conv_state_v_out = _ptr(conv_state_v_out, bf, "conv_state_v_out")
    p.q_out = _ptr(q_out, bf, "q_out"); p.r_out = _ptr(r_out, bf, "r_out")
    p.y_out = _ptr(y_out, bf, "y_out")
    p.kv_dtype, cache_dt = _kv_dtype(k_cache)
    p.k_cache = _ptr(k_cache, cache_dt, "k_cache"); p.v_cache = _ptr(v_cache, cache_dt, "v_cache")
    if p.kv_dtype == INKATTN_KV_E4M3:
        p.k_scale = _ptr(k_scale, f32, "k_scale"); p.v_scale = _ptr(v_scale, f32, "v_scale")
    p.dev_status = _ptr(dev_status, i32, "dev_status")
    return p
