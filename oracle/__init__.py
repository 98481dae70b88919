"""CPU oracle for the FP8 W8A8 rollout linear path (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code
with them.

The quantisation, GEMM and KV-cache arithmetic lives in ``oracle.c`` (plain
C, fp64 where the pages leave the precision open); this module compiles it
with gcc and marshals numpy arrays.  See the header of ``oracle.c`` for what
each function follows and the readings taken where the FP8-RL pages are
silent.  The SwiGLU helpers below, the MoE dispatch/combine
(``moe_routing.py``) and the TIS weight / mismatch KL (``tis.py``) are plain
fp64 numpy and Python loops, each module with its own header of citations
and readings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SCALE_FP32 = 0
SCALE_UE8M0 = 1


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (portable flags only)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, vp, f32, f64 = (ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_float, ctypes.c_double)
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = f64
        lib.oracle_e4m3_encode.argtypes = [f32]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode_f64.argtypes = [f64]
        lib.oracle_e4m3_encode_f64.restype = ctypes.c_uint8
        lib.oracle_scale_fp32.argtypes = [f32]
        lib.oracle_scale_fp32.restype = f32
        lib.oracle_scale_ue8m0_exponent.argtypes = [f32]
        lib.oracle_scale_ue8m0_exponent.restype = i32
        lib.oracle_e4m3_encode_array.argtypes = [vp, i64, vp, i32]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_quant_weight_blockwise.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i32]
        lib.oracle_quant_weight_blockwise.restype = i32
        lib.oracle_quant_act_group.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i32]
        lib.oracle_kv_calibrate.restype = i32
        lib.oracle_kv_calibrate.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
        lib.oracle_kv_append.restype = i32
        lib.oracle_kv_append.argtypes = [vp, vp, i64, i64, i64, i64, vp, vp, vp, i64, i64, vp]
        lib.oracle_quant_group_f32.restype = i32
        lib.oracle_quant_group_f32.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i32]
        lib.oracle_quant_act_group.restype = i32
        lib.oracle_gemm_blockscaled.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32]
        lib.oracle_gemm_blockscaled.restype = i32
        lib.oracle_gemm_blockscaled_at.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32,
                                                   vp, vp, i64, vp, i32]
        lib.oracle_gemm_blockscaled_at.restype = i32
        lib.oracle_grouped_gemm_blockscaled.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                                        vp, i32, i32]
        lib.oracle_grouped_gemm_blockscaled.restype = i32
        lib.oracle_grouped_gemm_blockscaled_at.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                                           i32, vp, vp, i64, vp, i32]
        lib.oracle_grouped_gemm_blockscaled_at.restype = i32
        _lib = lib
        return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _scale_dtype(fmt: int):
    if fmt == SCALE_FP32:
        return np.float32
    if fmt == SCALE_UE8M0:
        return np.uint8
    raise ValueError(f"unknown scale format {fmt}")


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


# --------------------------------------------------------------------------- format

def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (NaN for 0x7F / 0xFF)."""
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    """fp64 values of all 256 codes, indexed by code."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: float) -> int:
    """Saturating round-to-nearest-even of an fp32 value to an E4M3 code."""
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_encode_f64(v: float) -> int:
    """Saturating round-to-nearest-even of an exact fp64 value to an E4M3 code."""
    return int(_load().oracle_e4m3_encode_f64(float(v)))


def e4m3_encode_array(v: np.ndarray, threads: int | None = None) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out), threads or default_threads())
    return out


def scale_fp32(amax: float) -> float:
    return float(_load().oracle_scale_fp32(float(amax)))


def scale_ue8m0_exponent(amax: float) -> int:
    return int(_load().oracle_scale_ue8m0_exponent(float(amax)))


# --------------------------------------------------------------------------- quantisers

def quant_weight_blockwise(w_bf16_bits: np.ndarray, fmt: int = SCALE_FP32,
                           threads: int | None = None):
    """128x128 blockwise quantisation of a bf16 matrix given as uint16 bit patterns.

    Returns (q uint8 [n,k], scale [ceil(n/128), ceil(k/128)] fp32 or uint8)."""
    w = _c(w_bf16_bits, np.uint16)
    n, k = w.shape
    q = np.empty((n, k), dtype=np.uint8)
    s = np.empty(((n + 127) // 128, (k + 127) // 128), dtype=_scale_dtype(fmt))
    rc = _load().oracle_quant_weight_blockwise(_ptr(w), n, k, k, _ptr(q), k, _ptr(s), fmt,
                                               threads or default_threads())
    _check(rc, "quant_weight_blockwise")
    return q, s


def quant_act_group(x_bf16_bits: np.ndarray, fmt: int = SCALE_FP32, threads: int | None = None):
    """1x128 group quantisation of a bf16 activation matrix [m, k] (uint16 bits).

    Returns (q uint8 [m,k], scale [ceil(k/128), m] fp32 or uint8)."""
    x = _c(x_bf16_bits, np.uint16)
    m, k = x.shape
    q = np.empty((m, k), dtype=np.uint8)
    s = np.empty(((k + 127) // 128, m), dtype=_scale_dtype(fmt))
    rc = _load().oracle_quant_act_group(_ptr(x), m, k, k, _ptr(q), k, _ptr(s), fmt,
                                        threads or default_threads())
    _check(rc, "quant_act_group")
    return q, s


def quant_group_f32(x_f32: np.ndarray, fmt: int = SCALE_FP32, threads: int | None = None):
    """1x128 group quantisation of an fp32 matrix [m, k] (values never rounded
    to bf16).  Returns (q uint8 [m,k], scale [ceil(k/128), m] fp32 or uint8)."""
    x = _c(x_f32, np.float32)
    m, k = x.shape
    q = np.empty((m, k), dtype=np.uint8)
    s = np.empty(((k + 127) // 128, m), dtype=_scale_dtype(fmt))
    rc = _load().oracle_quant_group_f32(_ptr(x), m, k, k, _ptr(q), k, _ptr(s), fmt, threads or default_threads())
    _check(rc, "quant_group_f32")
    return q, s


def kv_calibrate(k_bf16_bits: np.ndarray, v_bf16_bits: np.ndarray, q_bf16_bits: np.ndarray | None = None):
    """Per-tensor fp32 scales (amax / 448) of the calibration pass's K, V
    [tokens, kv_dim] and optionally Q [tokens, q_dim]: float32 [3] (k, v, q;
    q is 0 without a Q tensor)."""
    k = _c(k_bf16_bits, np.uint16)
    v = _c(v_bf16_bits, np.uint16)
    t, d = k.shape
    scales = np.zeros(3, np.float32)
    if q_bf16_bits is None:
        rc = _load().oracle_kv_calibrate(_ptr(k), _ptr(v), None, t, d, d, d, 0, 0, _ptr(scales))
    else:
        q = _c(q_bf16_bits, np.uint16)
        rc = _load().oracle_kv_calibrate(_ptr(k), _ptr(v), _ptr(q), t, d, d, d, q.shape[1], q.shape[1],
                                         _ptr(scales))
    _check(rc, "kv_calibrate")
    return scales


def kv_append(k_bf16_bits, v_bf16_bits, slots, k_cache, v_cache, scales):
    """Quantise rows of K and V into the caches (uint8 [num_slots, kv_dim],
    updated in place) at `slots` (int32 [tokens]; out-of-range: skipped)."""
    k = _c(k_bf16_bits, np.uint16)
    v = _c(v_bf16_bits, np.uint16)
    sl = _c(slots, np.int32)
    sc = _c(scales, np.float32)
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    t, d = k.shape
    rc = _load().oracle_kv_append(_ptr(k), _ptr(v), t, d, d, d, _ptr(sl), _ptr(k_cache), _ptr(v_cache),
                                  k_cache.shape[1], k_cache.shape[0], _ptr(sc))
    _check(rc, "kv_append")


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU (swish) in fp64: x * sigmoid(x) = x / (1 + exp(-x)).  The gated
    MLP of the pages' Qwen3 models applies SiLU to the gate projection and
    multiplies by the up projection (SwiGLU)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SiLU(gate) * up, elementwise, in fp64."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


def interleave_gate_up_rows(rows: int) -> np.ndarray:
    """Row order of the fused gate-up weight that the fused kernel consumes:
    128-row blocks alternate gate, up, gate, up ...; returns, for each row of
    the interleaved matrix, its row in [gate; up] (rows = 2 * inter)."""
    inter = rows // 2
    idx = np.empty(rows, dtype=np.int64)
    for b in range(inter // 128):
        idx[256 * b:256 * b + 128] = np.arange(128 * b, 128 * b + 128)
        idx[256 * b + 128:256 * b + 256] = inter + np.arange(128 * b, 128 * b + 128)
    return idx


def gemm_swiglu_quant(xq, sx, wq_il, sw_il, fmt_w: int = SCALE_FP32, fmt_h: int = SCALE_FP32,
                      offsets=None, threads: int | None = None):
    """Reference of the fused gate-up path: the block-scaled GEMM against the
    interleaved gate-up weight (dense, or grouped by `offsets`), de-interleaved
    into gate and up, h = SiLU(gate) * up in fp64, rounded once to fp32, then
    quantised in 1x128 groups.  Returns (h fp64 [m, inter], hq, h_scale)."""
    if offsets is None:
        y = gemm_blockscaled(xq, sx, wq_il, sw_il, fmt_w, threads)
    else:
        y = grouped_gemm_blockscaled(xq, sx, wq_il, sw_il, offsets, fmt_w, threads)
    rows = y.shape[1]
    inter = rows // 2
    order = interleave_gate_up_rows(rows)
    plain = np.empty_like(y)
    plain[:, order] = y          # column j of y is row order[j] of [gate; up]
    h = swiglu(plain[:, :inter], plain[:, inter:])
    hq, hs = quant_group_f32(h.astype(np.float32), fmt_h, threads)
    return h, hq, hs


# --------------------------------------------------------------------------- GEMMs

def gemm_blockscaled(xq, sx, wq, sw, fmt: int = SCALE_FP32, threads: int | None = None) -> np.ndarray:
    """fp64 Y[m,n] = sum_k dec(xq)*sx * dec(wq)*sw over the full output."""
    xq = _c(xq, np.uint8)
    wq = _c(wq, np.uint8)
    sx = _c(sx, _scale_dtype(fmt))
    sw = _c(sw, _scale_dtype(fmt))
    m, k = xq.shape
    n = wq.shape[0]
    if wq.shape[1] != k or sx.shape != (k // 128, m) or sw.shape != (n // 128, k // 128):
        raise ValueError("shape mismatch")
    y = np.empty((m, n), dtype=np.float64)
    rc = _load().oracle_gemm_blockscaled(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), _ptr(y), m, n, k,
                                         fmt, threads or default_threads())
    _check(rc, "gemm_blockscaled")
    return y


def gemm_blockscaled_at(xq, sx, wq, sw, rows, cols, fmt: int = SCALE_FP32,
                        threads: int | None = None) -> np.ndarray:
    """The same product evaluated at the listed (row, col) positions only."""
    xq = _c(xq, np.uint8)
    wq = _c(wq, np.uint8)
    sx = _c(sx, _scale_dtype(fmt))
    sw = _c(sw, _scale_dtype(fmt))
    rows = _c(np.asarray(rows, dtype=np.int64), np.int64)
    cols = _c(np.asarray(cols, dtype=np.int64), np.int64)
    m, k = xq.shape
    n = wq.shape[0]
    if wq.shape[1] != k or sx.shape != (k // 128, m) or sw.shape != (n // 128, k // 128):
        raise ValueError("shape mismatch")
    out = np.empty(rows.shape, dtype=np.float64)
    rc = _load().oracle_gemm_blockscaled_at(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), m, n, k, fmt,
                                            _ptr(rows), _ptr(cols), rows.size, _ptr(out),
                                            threads or default_threads())
    _check(rc, "gemm_blockscaled_at")
    return out


def grouped_gemm_blockscaled(xq, sx, wq, sw, offsets, fmt: int = SCALE_FP32,
                             threads: int | None = None) -> np.ndarray:
    """Per-expert product over row segments; wq [E,n,k], sw [E,n/128,k/128]."""
    xq = _c(xq, np.uint8)
    wq = _c(wq, np.uint8)
    sx = _c(sx, _scale_dtype(fmt))
    sw = _c(sw, _scale_dtype(fmt))
    offsets = _c(np.asarray(offsets, dtype=np.int32), np.int32)
    rows, k = xq.shape
    e, n, _ = wq.shape
    if offsets.shape != (e + 1,):
        raise ValueError("offsets must have experts+1 entries")
    y = np.empty((rows, n), dtype=np.float64)
    rc = _load().oracle_grouped_gemm_blockscaled(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw),
                                                 _ptr(offsets), e, rows, n, k, _ptr(y), fmt,
                                                 threads or default_threads())
    _check(rc, "grouped_gemm_blockscaled")
    return y


def grouped_gemm_blockscaled_at(xq, sx, wq, sw, offsets, rows_at, cols_at, fmt: int = SCALE_FP32,
                                threads: int | None = None) -> np.ndarray:
    xq = _c(xq, np.uint8)
    wq = _c(wq, np.uint8)
    sx = _c(sx, _scale_dtype(fmt))
    sw = _c(sw, _scale_dtype(fmt))
    offsets = _c(np.asarray(offsets, dtype=np.int32), np.int32)
    rows_at = _c(np.asarray(rows_at, dtype=np.int64), np.int64)
    cols_at = _c(np.asarray(cols_at, dtype=np.int64), np.int64)
    rows, k = xq.shape
    e, n, _ = wq.shape
    out = np.empty(rows_at.shape, dtype=np.float64)
    rc = _load().oracle_grouped_gemm_blockscaled_at(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw),
                                                    _ptr(offsets), e, rows, n, k, fmt,
                                                    _ptr(rows_at), _ptr(cols_at), rows_at.size,
                                                    _ptr(out), threads or default_threads())
    _check(rc, "grouped_gemm_blockscaled_at")
    return out


def dequantize(q: np.ndarray, scale: np.ndarray, block_rows: int, block_cols: int,
               fmt: int = SCALE_FP32) -> np.ndarray:
    """fp64 dequantised values dec(q) * scale of the block each element sits in.

    ``scale`` is indexed [row_block, col_block]; activation scales stored
    [group, m] are passed transposed by the caller."""
    table = e4m3_decode_table()
    vals = table[q]
    if fmt == SCALE_UE8M0:
        s = np.ldexp(1.0, scale.astype(np.int64) - 127)
    else:
        s = scale.astype(np.float64)
    r_idx = np.arange(q.shape[0]) // block_rows
    c_idx = np.arange(q.shape[1]) // block_cols
    return vals * s[r_idx][:, c_idx]


from .moe_routing import combine as moe_combine  # noqa: E402
from .moe_routing import dispatch_plan as moe_dispatch_plan  # noqa: E402
from .moe_routing import gather_rows as moe_gather_rows  # noqa: E402
from .tis import TIS_CLIP, mismatch_kl, tis_weights  # noqa: E402


def moe_dispatch_quant(x_bf16_bits: np.ndarray, token_of_row: np.ndarray, fmt: int = SCALE_FP32):
    """Grouped activation of the dispatch: gathered token rows, quantised in
    1x128 groups.  Returns (codes [R, K], scales [K/128, R], live rows)."""
    from .moe_routing import dispatch_quant
    return dispatch_quant(x_bf16_bits, token_of_row, fmt, quant_act_group)
