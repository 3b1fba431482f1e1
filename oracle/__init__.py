"""fp64 CPU oracle for the Inkling attention hot path (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
product path never calls it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent
rows); this module only compiles it with gcc and marshals numpy arrays.
bf16 tensors cross this boundary as their raw uint16 bit patterns.

What each function computes, with the passages it follows, is stated in the
header comment of ``oracle.c``.  Every function here is pinned by tests in
``tests/test_oracle_pins.py`` against library routines (torch SDPA, numpy
correlate, torch rms_norm), closed forms and hand-derived fixtures in
``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_f64_to_bf16.argtypes = [D]
            lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
            lib.oracle_log_scale.argtypes = [D, D]
            lib.oracle_log_scale.restype = D
            lib.oracle_prologue.argtypes = (
                [I, P, I, I, I, P, P, P, P, P, P, P, D, P, I, P, P, P, I, I, P, P, P, P, P, P, P])
            lib.oracle_prologue.restype = I
            lib.oracle_attention.argtypes = (
                [I, P, P, I, I, I, I, I, I, D, D, P, P, P, P, P, P, I, I, I, P, I, P, P, I])
            lib.oracle_attention.restype = I
            lib.oracle_output_conv.argtypes = [I, P, I, P, P, P, I, P, P, P, D, P, P, P]
            lib.oracle_output_conv.restype = I
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f64.restype = D
            lib.oracle_f64_to_e4m3.argtypes = [D]
            lib.oracle_f64_to_e4m3.restype = ctypes.c_uint8
            lib.oracle_quantize_rows_e4m3.argtypes = [P, I, I, P, P]
            lib.oracle_quantize_rows_e4m3.restype = I
            lib.oracle_round_bf16_array.argtypes = [P, ctypes.c_longlong, P]
            lib.oracle_round_bf16_array.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def f64_to_bf16_bits(x: float) -> int:
    """Round one double to bf16 (ties to even) and return its bit pattern."""
    return int(_load().oracle_f64_to_bf16(float(x)))


def log_scale(T: float, base: float) -> float:
    """lambda = max(1, ln T / ln base) (1 when base <= 1)."""
    return float(_load().oracle_log_scale(float(T), float(base)))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def prologue(*, cu_seqlens_q, Hq, Hkv, d, q, k, v, conv_w_k, conv_w_v, q_norm_w, k_norm_w,
             eps, state_slot, conv_state_k, conv_state_v, slot_mapping, block_size,
             k_cache, v_cache, want_f64=False):
    """Run the prologue oracle.

    Inputs are numpy arrays (bf16 as uint16 bits).  conv_state_k/v and
    k_cache/v_cache are copied, updated and returned; the caller's arrays are
    not modified.  Returns a dict with q_out, k_cache, v_cache, conv_state_k,
    conv_state_v, kc (bf16 bits of the conv output), vc and, when want_f64,
    kc_f64 / vc_f64 (the conv sums before rounding).
    """
    lib = _load()
    cu = _c(cu_seqlens_q, np.int32)
    B = cu.shape[0] - 1
    N = int(cu[-1])
    C = Hkv * d
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    wk = _c(conv_w_k, np.float32); wv = _c(conv_w_v, np.float32)
    gq = _c(q_norm_w, np.float32); gk = _c(k_norm_w, np.float32)
    ss = _c(state_slot, np.int32)
    sk = np.array(conv_state_k, dtype=np.uint16, copy=True, order="C")
    sv = np.array(conv_state_v, dtype=np.uint16, copy=True, order="C")
    sm = _c(slot_mapping, np.int32)
    kc_cache = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc_cache = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    q_out = np.zeros((N, Hq, d), dtype=np.uint16)
    kc = np.zeros((N, C), dtype=np.uint16)
    vc = np.zeros((N, C), dtype=np.uint16)
    kc64 = np.zeros((N, C), dtype=np.float64) if want_f64 else None
    vc64 = np.zeros((N, C), dtype=np.float64) if want_f64 else None
    num_state_slots = sk.shape[0]
    num_blocks = kc_cache.shape[0]
    rc = lib.oracle_prologue(B, _ptr(cu), Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v), _ptr(wk), _ptr(wv),
                             _ptr(gq), _ptr(gk), float(eps), _ptr(ss), num_state_slots,
                             _ptr(sk), _ptr(sv), _ptr(sm), block_size, num_blocks,
                             _ptr(q_out), _ptr(kc_cache), _ptr(vc_cache),
                             _ptr(kc64), _ptr(vc64), _ptr(kc), _ptr(vc))
    if rc != 0:
        raise ValueError(f"oracle_prologue failed with code {rc}")
    out = dict(q_out=q_out, k_cache=kc_cache, v_cache=vc_cache, conv_state_k=sk,
               conv_state_v=sv, kc=kc, vc=vc)
    if want_f64:
        out["kc_f64"] = kc64
        out["vc_f64"] = vc64
    return out


def attention(*, cu_seqlens_q, seqlen_k, Hq, Hkv, d, d_r, rel_extent, window,
              softmax_scale, log_scale_base, q, r, P, k_cache, v_cache, block_table,
              block_size, rows=None, n_threads=0):
    """Run the attention oracle; returns (out float64, lse float64).

    P is [Hq][rel_extent][d_r]: P[h][delta] holds the d_r weights that project r onto
    the relative logit of distance delta (the matrix P_h of the method, distance-major).

    With rows=None every token row is computed and out has shape [N][Hq][d];
    otherwise out is [len(rows)][Hq][d] for the listed token indices.
    """
    lib = _load()
    cu = _c(cu_seqlens_q, np.int32)
    sk = _c(seqlen_k, np.int32)
    B = cu.shape[0] - 1
    N = int(cu[-1])
    q = _c(q, np.uint16)
    r = _c(r, np.uint16) if r is not None else None
    P = _c(P, np.float32) if P is not None else None
    kcache = _c(k_cache, np.uint16)
    vcache = _c(v_cache, np.uint16)
    bt = _c(block_table, np.int32)
    max_blocks = bt.shape[1]
    num_blocks = kcache.shape[0]
    rws = None if rows is None else _c(rows, np.int32)
    nr = N if rows is None else int(rws.shape[0])
    out = np.zeros((nr, Hq, d), dtype=np.float64)
    lse = np.zeros((nr, Hq), dtype=np.float64)
    rc = lib.oracle_attention(B, _ptr(cu), _ptr(sk), Hq, Hkv, d, d_r, rel_extent, window,
                              float(softmax_scale), float(log_scale_base), _ptr(q), _ptr(r),
                              _ptr(P), _ptr(kcache), _ptr(vcache), _ptr(bt), max_blocks,
                              block_size, num_blocks, _ptr(rws), nr, _ptr(out), _ptr(lse),
                              int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with code {rc}")
    return out, lse


# ------------------------------------------------------------------ workload adapters

def _bits(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().contiguous().cpu().numpy()


def prologue_for_inputs(x, workload):
    """The prologue oracle on a dict of workload tensors (any device, as produced by
    relative_bias_hybrid_gb300.inputs.make_inputs).  Returns numpy arrays."""
    d = workload.head_dim
    return prologue(cu_seqlens_q=_bits(x["cu_seqlens_q"]), Hq=workload.Hq, Hkv=workload.Hkv, d=d,
                    q=_bits(x["q"]), k=_bits(x["k"]), v=_bits(x["v"]),
                    conv_w_k=_bits(x["conv_w_k"]), conv_w_v=_bits(x["conv_w_v"]),
                    q_norm_w=_bits(x["q_norm_w"]), k_norm_w=_bits(x["k_norm_w"]), eps=workload.eps,
                    state_slot=_bits(x["state_slot"]), conv_state_k=_bits(x["conv_state_k"]),
                    conv_state_v=_bits(x["conv_state_v"]), slot_mapping=_bits(x["slot_mapping"]),
                    block_size=workload.block_size, k_cache=_bits(x["k_cache"]),
                    v_cache=_bits(x["v_cache"]))


def qkvr_prologue_for_inputs(x, workload):
    """qkvr_prologue on a dict of workload tensors (any device, as produced by
    relative_bias_hybrid_gb300.inputs.make_qkvr_inputs).  Returns numpy arrays."""
    return qkvr_prologue(x=_bits(x["x"]), w=_bits(x["w_qkvr"]), d_r=workload.d_r,
                         cu_seqlens_q=_bits(x["cu_seqlens_q"]), Hq=workload.Hq, Hkv=workload.Hkv,
                         d=workload.head_dim, conv_w_k=_bits(x["conv_w_k"]), conv_w_v=_bits(x["conv_w_v"]),
                         q_norm_w=_bits(x["q_norm_w"]), k_norm_w=_bits(x["k_norm_w"]), eps=workload.eps,
                         state_slot=_bits(x["state_slot"]), conv_state_k=_bits(x["conv_state_k"]),
                         conv_state_v=_bits(x["conv_state_v"]), slot_mapping=_bits(x["slot_mapping"]),
                         block_size=workload.block_size, k_cache=_bits(x["k_cache"]),
                         v_cache=_bits(x["v_cache"]))


def attention_for_inputs(x, workload, q_bits, k_cache_bits, v_cache_bits, rows=None, n_threads=0):
    """The attention oracle for a workload, on the given normalised queries and caches
    (bf16 bit arrays) and the workload's r, P, lengths and block table."""
    return attention(cu_seqlens_q=_bits(x["cu_seqlens_q"]), seqlen_k=_bits(x["seqlen_k"]),
                     Hq=workload.Hq, Hkv=workload.Hkv, d=workload.head_dim, d_r=workload.d_r,
                     rel_extent=workload.rel_extent, window=workload.window, softmax_scale=0.0,
                     log_scale_base=workload.log_scale_base, q=q_bits, r=_bits(x["r"]),
                     P=_bits(x["P"]), k_cache=k_cache_bits, v_cache=v_cache_bits,
                     block_table=_bits(x["block_table"]), block_size=workload.block_size,
                     rows=rows, n_threads=n_threads)


def output_conv(*, cu_seqlens_q, D, y, conv_w, state_slot, conv_state, residual, norm_w, eps,
                want_conv=False):
    """Run the attention-output ShortConv + residual add + RMSNorm oracle.

    Inputs are numpy arrays (bf16 as uint16 bits): y, residual [N][D]; conv_w [D][4];
    norm_w [D]; conv_state [slots][3][D] (copied, updated and returned).  Returns a dict
    with h (the new residual stream), out (its RMSNorm), conv_state and, when want_conv,
    conv (the rounded conv outputs).
    """
    lib = _load()
    cu = _c(cu_seqlens_q, np.int32)
    B = cu.shape[0] - 1
    N = int(cu[-1])
    y = _c(y, np.uint16)
    w = _c(conv_w, np.float32)
    ss = _c(state_slot, np.int32)
    st = np.array(conv_state, dtype=np.uint16, copy=True, order="C")
    res = _c(residual, np.uint16)
    g = _c(norm_w, np.float32)
    h = np.zeros((N, D), dtype=np.uint16)
    out = np.zeros((N, D), dtype=np.uint16)
    conv = np.zeros((N, D), dtype=np.uint16) if want_conv else None
    rc = lib.oracle_output_conv(B, _ptr(cu), int(D), _ptr(y), _ptr(w), _ptr(ss), st.shape[0],
                                _ptr(st), _ptr(res), _ptr(g), float(eps), _ptr(h), _ptr(out),
                                _ptr(conv))
    if rc != 0:
        raise ValueError(f"oracle_output_conv failed with code {rc}")
    d = dict(h=h, out=out, conv_state=st)
    if want_conv:
        d["conv"] = conv
    return d


def e4m3_to_f64(code: int) -> float:
    """Value of one E4M3 code (OCP FP8 E4M3FN)."""
    return float(_load().oracle_e4m3_to_f64(int(code) & 0xFF))


def f64_to_e4m3(x: float) -> int:
    """Nearest E4M3 code to x, ties to even, saturating at 448."""
    return int(_load().oracle_f64_to_e4m3(float(x)))


def quantize_rows_e4m3(x_bits):
    """Quantise rows of bf16 values (uint16 bits, shape [..., width]) to E4M3 codes with
    one power-of-two scale per row.  Returns (codes uint8 same shape, scales float32
    shape [...])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    width = x.shape[-1]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(x.shape[:-1], dtype=np.float32)
    rc = _load().oracle_quantize_rows_e4m3(_ptr(x), rows, width, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError(f"oracle_quantize_rows_e4m3 failed with code {rc}")
    return codes, scales


def dequantize_e4m3(codes, scales) -> np.ndarray:
    """code * scale for every element (scales broadcast over the last axis), as float64.
    For the power-of-two scales of quantize_rows_e4m3 the result is exact."""
    lut = np.array([e4m3_to_f64(c) for c in range(256)], dtype=np.float64)
    return lut[np.asarray(codes, dtype=np.uint8)] * np.asarray(scales, dtype=np.float64)[..., None]


def round_bf16(x) -> np.ndarray:
    """float64 array -> bf16 bit patterns, each value rounded once (ties to even)."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(a.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(_ptr(a), a.size, _ptr(out))
    return out


def qkvr_projection(x, w, *, Hq, Hkv, d, d_r):
    """Step 8 of oracle.c: y = x . w^T in float64 (numpy's matrix product), each value
    rounded once to bf16, split into q [N][Hq][d], k [N][Hkv*d], v [N][Hkv*d] and
    r [N][Hq][d_r] (bf16 bit patterns).  x: [N][d_model] bits, w: [Hq*d + 2*Hkv*d + Hq*d_r]
    [d_model] bits."""
    xf = bf16_bits_to_f64(np.asarray(x, dtype=np.uint16))
    wf = bf16_bits_to_f64(np.asarray(w, dtype=np.uint16))
    y = round_bf16(xf @ wf.T)
    N = y.shape[0]
    c = np.cumsum([0, Hq * d, Hkv * d, Hkv * d, Hq * d_r])
    assert y.shape[1] == c[-1]
    return (y[:, c[0]:c[1]].reshape(N, Hq, d), y[:, c[1]:c[2]], y[:, c[2]:c[3]],
            y[:, c[3]:c[4]].reshape(N, Hq, d_r))


def qkvr_prologue(*, x, w, d_r, **prologue_args):
    """Steps 8 then 1-4: the projections of the hidden states x, then the prologue on the
    projected q, k, v.  prologue_args are those of prologue() except q, k and v.  Returns
    prologue()'s dict plus r (bf16 bits) and q_proj, k_proj, v_proj (the projections)."""
    q, k, v, r = qkvr_projection(x, w, Hq=prologue_args["Hq"], Hkv=prologue_args["Hkv"],
                                 d=prologue_args["d"], d_r=d_r)
    out = prologue(q=q, k=k, v=v, **prologue_args)
    out.update(r=r, q_proj=q, k_proj=k, v_proj=v)
    return out
