"""GB300-native FP8 W8A8 rollout linear path: Python binding of ``libfp8rl.so``.

The functions named ``fp8rl_*`` mirror the C ABI in ``include/fp8rl.h`` one
to one: they only marshal arguments (a torch tensor becomes its device
pointer, ``stream=None`` becomes torch's current stream) and raise
``Fp8rlError`` on a non-OK status.  Every step of the path runs in the CUDA
kernels of the library; there is no CPU or PyTorch fallback, and loading fails
loudly when the library has not been built.

The convenience helpers below them (``quant_weight``, ``quant_act``,
``gemm``, ``grouped_gemm``, ``quant_weights_batched``) allocate the outputs
with torch and call the same entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "Fp8rlError", "SCALE_FP32", "SCALE_UE8M0", "load_library", "library_path",
    "fp8rl_quant_weight_blockwise", "fp8rl_quant_weight_blockwise_batched",
    "fp8rl_host_sync_staging_bytes", "fp8rl_quant_weight_host_batched",
    "fp8rl_quant_act_group", "fp8rl_gemm_blockscaled", "fp8rl_grouped_gemm_blockscaled",
    "fp8rl_gemm_act_quant", "gemm_act_quant",
    "fp8rl_gemm_workspace_size", "fp8rl_gemm_blockscaled_ws", "gemm_workspace",
    "fp8rl_gemm_blockscaled_static", "fp8rl_gemm_swiglu_quant", "fp8rl_grouped_gemm_swiglu_quant",
    "gemm_swiglu_quant", "grouped_gemm_swiglu_quant", "quant_gate_up_interleaved",
    "fp8rl_kv_calibrate", "fp8rl_kv_append", "kv_calibrate", "kv_append",
    "fp8rl_e4m3_encode", "fp8rl_debug_set", "fp8rl_sync_status", "fp8rl_status_string", "fp8rl_version",
    "quant_weight", "quant_weights_batched", "quant_act", "gemm", "grouped_gemm", "HostWeightSync",
    "CanaryError", "canaries_enabled", "check_canaries",
]

SCALE_FP32 = 0
SCALE_UE8M0 = 1

STATUS = {0: "FP8RL_OK", 1: "FP8RL_ERR_INVALID_ARG", 2: "FP8RL_ERR_SHAPE",
          3: "FP8RL_ERR_ALIGNMENT", 4: "FP8RL_ERR_UNSUPPORTED", 5: "FP8RL_ERR_CUDA",
          6: "FP8RL_ERR_TIMEOUT", 7: "FP8RL_ERR_DEVICE_CHECK"}


class Fp8rlError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class WeightDesc(ctypes.Structure):
    """fp8rl_weight_desc"""
    _fields_ = [("w_bf16", ctypes.c_void_p), ("q_e4m3", ctypes.c_void_p),
                ("w_scale", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("ldw", ctypes.c_int64), ("ldq", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """``libfp8rl.so``, or ``libfp8rl_debug.so`` when FP8RL_DEBUG=1."""
    return _build.LIB_DEBUG if _build.debug_requested() else _build.LIB


def load_library(build_if_missing: bool = False):
    """Load the library (raises if it is missing and building is not asked for)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing:
            _build.build()
        if not os.path.exists(path):
            raise FileNotFoundError(
                f"{path} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        st = ctypes.c_int
        sig = {
            "fp8rl_quant_weight_blockwise": [vp, i64, i64, i64, vp, i64, vp, st, vp],
            "fp8rl_quant_weight_blockwise_batched": [ctypes.POINTER(WeightDesc), i32, st, vp],
            "fp8rl_host_sync_staging_bytes": [i64, i64, i32, st],
            "fp8rl_quant_weight_host_batched": [ctypes.POINTER(WeightDesc), i32, st, vp, ctypes.c_size_t, i32, vp],
            "fp8rl_quant_act_group": [vp, i64, i64, i64, vp, i64, vp, st, vp],
            "fp8rl_gemm_blockscaled": [vp, vp, vp, vp, vp, i64, i64, i64, st, vp],
            "fp8rl_gemm_act_quant": [vp, i64, vp, vp, vp, i64, i64, i64, st, vp, vp, vp],
            "fp8rl_gemm_workspace_size": [ctypes.POINTER(ctypes.c_size_t)],
            "fp8rl_gemm_blockscaled_ws": [vp, vp, vp, vp, vp, i64, i64, i64, st, vp, ctypes.c_size_t, vp],
            "fp8rl_gemm_blockscaled_static": [vp, vp, vp, vp, vp, i64, i64, i64, st, vp],
            "fp8rl_gemm_swiglu_quant": [vp, vp, vp, vp, i64, i64, i64, vp, vp, st, vp],
            "fp8rl_kv_calibrate": [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, vp],
            "fp8rl_kv_append": [vp, vp, i64, i64, i64, i64, vp, vp, vp, i64, i64, vp, vp],
            "fp8rl_grouped_gemm_swiglu_quant": [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, vp, st, vp],
            "fp8rl_grouped_gemm_blockscaled": [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, st, vp],
            "fp8rl_e4m3_encode": [vp, i64, vp, vp],
            "fp8rl_moe_plan_workspace_size": [i64, i64, i64],
            "fp8rl_moe_plan": [vp, i64, i64, i64, vp, vp, vp, vp, ctypes.c_size_t, vp],
            "fp8rl_moe_dispatch_quant": [vp, i64, i64, i64, vp, i64, i64, vp, i64, vp, st, vp],
            "fp8rl_moe_combine": [vp, i64, i64, i64, vp, vp, i64, i64, vp, i64, vp],
            "fp8rl_tis_workspace_size": [i64],
            "fp8rl_tis_weights": [vp, vp, vp, i64, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp],
            "fp8rl_debug_set": [i32, i64],
            "fp8rl_sync_status": [vp],
            "fp8rl_status_string": [st],
            "fp8rl_version": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = st
        lib.fp8rl_status_string.restype = ctypes.c_char_p
        lib.fp8rl_moe_plan_workspace_size.restype = ctypes.c_size_t
        lib.fp8rl_host_sync_staging_bytes.restype = ctypes.c_size_t
        lib.fp8rl_tis_workspace_size.restype = ctypes.c_size_t
        lib.fp8rl_version.restype = i32
        _lib = lib
        return lib


# --------------------------------------------------------------------------- marshalling

def _p(x) -> int | None:
    """A device pointer from a tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(stream) -> int | None:
    if stream is None:
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ok(status: int, what: str) -> None:
    if status != 0:
        raise Fp8rlError(status, what)


# --------------------------------------------------------------------------- C ABI, 1:1

def fp8rl_quant_weight_blockwise(w_bf16, n, k, ldw, q_e4m3, ldq, w_scale, fmt=SCALE_FP32,
                                 stream=None) -> None:
    _ok(load_library().fp8rl_quant_weight_blockwise(_p(w_bf16), n, k, ldw, _p(q_e4m3), ldq,
                                                    _p(w_scale), fmt, _stream(stream)),
        "fp8rl_quant_weight_blockwise")


def fp8rl_quant_weight_blockwise_batched(descs, count, fmt=SCALE_FP32, stream=None) -> None:
    _ok(load_library().fp8rl_quant_weight_blockwise_batched(descs, count, fmt, _stream(stream)),
        "fp8rl_quant_weight_blockwise_batched")


def fp8rl_host_sync_staging_bytes(rows, k, slots, fmt=SCALE_FP32) -> int:
    return int(load_library().fp8rl_host_sync_staging_bytes(rows, k, slots, fmt))


def fp8rl_quant_weight_host_batched(descs, count, fmt, d_staging, staging_bytes, slots, stream=None) -> None:
    _ok(load_library().fp8rl_quant_weight_host_batched(descs, count, fmt, _p(d_staging), int(staging_bytes),
                                                       slots, _stream(stream)),
        "fp8rl_quant_weight_host_batched")


def fp8rl_quant_act_group(x_bf16, m, k, ldx, q_e4m3, ldq, x_scale, fmt=SCALE_FP32,
                          stream=None) -> None:
    _ok(load_library().fp8rl_quant_act_group(_p(x_bf16), m, k, ldx, _p(q_e4m3), ldq, _p(x_scale),
                                             fmt, _stream(stream)),
        "fp8rl_quant_act_group")


def fp8rl_gemm_blockscaled(xq, x_scale, wq, w_scale, y_bf16, m, n, k, fmt=SCALE_FP32,
                           stream=None) -> None:
    _ok(load_library().fp8rl_gemm_blockscaled(_p(xq), _p(x_scale), _p(wq), _p(w_scale),
                                              _p(y_bf16), m, n, k, fmt, _stream(stream)),
        "fp8rl_gemm_blockscaled")


def fp8rl_gemm_act_quant(x_bf16, ldx, wq, w_scale, y_bf16, m, n, k, fmt, xq, x_scale,
                         stream=None) -> None:
    _ok(load_library().fp8rl_gemm_act_quant(_p(x_bf16), ldx, _p(wq), _p(w_scale), _p(y_bf16), m, n, k,
                                            fmt, _p(xq), _p(x_scale), _stream(stream)),
        "fp8rl_gemm_act_quant")


def fp8rl_gemm_workspace_size() -> int:
    n = ctypes.c_size_t(0)
    _ok(load_library().fp8rl_gemm_workspace_size(ctypes.byref(n)), "fp8rl_gemm_workspace_size")
    return int(n.value)


def fp8rl_gemm_blockscaled_ws(xq, x_scale, wq, w_scale, y_bf16, m, n, k, fmt, workspace,
                              workspace_bytes, stream=None) -> None:
    _ok(load_library().fp8rl_gemm_blockscaled_ws(_p(xq), _p(x_scale), _p(wq), _p(w_scale),
                                                 _p(y_bf16), m, n, k, fmt, _p(workspace),
                                                 int(workspace_bytes), _stream(stream)),
        "fp8rl_gemm_blockscaled_ws")


def fp8rl_gemm_blockscaled_static(xq, x_scale, wq, w_scale, y_bf16, m, n, k, fmt=SCALE_FP32,
                                  stream=None) -> None:
    _ok(load_library().fp8rl_gemm_blockscaled_static(_p(xq), _p(x_scale), _p(wq), _p(w_scale),
                                                     _p(y_bf16), m, n, k, fmt, _stream(stream)),
        "fp8rl_gemm_blockscaled_static")


def fp8rl_gemm_swiglu_quant(xq, x_scale, wq_gate_up, w_scale_gate_up, m, inter, k, hq, h_scale,
                            fmt=SCALE_FP32, stream=None) -> None:
    _ok(load_library().fp8rl_gemm_swiglu_quant(_p(xq), _p(x_scale), _p(wq_gate_up), _p(w_scale_gate_up), m,
                                               inter, k, _p(hq), _p(h_scale), fmt, _stream(stream)),
        "fp8rl_gemm_swiglu_quant")


def fp8rl_grouped_gemm_swiglu_quant(xq, x_scale, wq_gate_up, w_scale_gate_up, d_offsets, num_experts, rows,
                                    inter, k, hq, h_scale, fmt=SCALE_FP32, stream=None) -> None:
    _ok(load_library().fp8rl_grouped_gemm_swiglu_quant(_p(xq), _p(x_scale), _p(wq_gate_up),
                                                       _p(w_scale_gate_up), _p(d_offsets), num_experts, rows,
                                                       inter, k, _p(hq), _p(h_scale), fmt, _stream(stream)),
        "fp8rl_grouped_gemm_swiglu_quant")


def fp8rl_kv_calibrate(k_bf16, v_bf16, q_bf16, tokens, kv_dim, ldk, ldv, q_dim, ldq, d_scales,
                       stream=None) -> None:
    _ok(load_library().fp8rl_kv_calibrate(_p(k_bf16), _p(v_bf16), _p(q_bf16), tokens, kv_dim, ldk, ldv, q_dim,
                                          ldq, _p(d_scales), _stream(stream)),
        "fp8rl_kv_calibrate")


def fp8rl_kv_append(k_bf16, v_bf16, tokens, kv_dim, ldk, ldv, d_slot_mapping, k_cache, v_cache, ld_cache,
                    num_slots, d_scales, stream=None) -> None:
    _ok(load_library().fp8rl_kv_append(_p(k_bf16), _p(v_bf16), tokens, kv_dim, ldk, ldv, _p(d_slot_mapping),
                                       _p(k_cache), _p(v_cache), ld_cache, num_slots, _p(d_scales),
                                       _stream(stream)),
        "fp8rl_kv_append")


def fp8rl_moe_plan_workspace_size(tokens, topk, experts) -> int:
    return int(load_library().fp8rl_moe_plan_workspace_size(tokens, topk, experts))


def fp8rl_moe_plan(d_topk, tokens, topk, experts, d_offsets, d_row_of_pair, d_token_of_row, d_workspace,
                   workspace_bytes, stream=None) -> None:
    _ok(load_library().fp8rl_moe_plan(_p(d_topk), tokens, topk, experts, _p(d_offsets), _p(d_row_of_pair),
                                      _p(d_token_of_row), _p(d_workspace), workspace_bytes, _stream(stream)),
        "fp8rl_moe_plan")


def fp8rl_moe_dispatch_quant(x_bf16, tokens, k, ldx, d_row_of_pair, topk, rows, q_e4m3, ldq, x_scale,
                             fmt=SCALE_FP32, stream=None) -> None:
    _ok(load_library().fp8rl_moe_dispatch_quant(_p(x_bf16), tokens, k, ldx, _p(d_row_of_pair), topk, rows,
                                                _p(q_e4m3), ldq, _p(x_scale), fmt, _stream(stream)),
        "fp8rl_moe_dispatch_quant")


def fp8rl_moe_combine(y_bf16, rows, n, ldy, d_row_of_pair, d_gate, tokens, topk, out_bf16, ldo,
                      stream=None) -> None:
    _ok(load_library().fp8rl_moe_combine(_p(y_bf16), rows, n, ldy, _p(d_row_of_pair), _p(d_gate), tokens, topk,
                                         _p(out_bf16), ldo, _stream(stream)),
        "fp8rl_moe_combine")


def fp8rl_tis_workspace_size(n) -> int:
    return int(load_library().fp8rl_tis_workspace_size(n))


def fp8rl_tis_weights(d_lp_train, d_lp_rollout, d_mask, n, clip, d_w, d_kl, d_workspace, workspace_bytes,
                      stream=None) -> None:
    _ok(load_library().fp8rl_tis_weights(_p(d_lp_train), _p(d_lp_rollout), _p(d_mask), n, clip, _p(d_w),
                                         _p(d_kl), _p(d_workspace), workspace_bytes, _stream(stream)),
        "fp8rl_tis_weights")


def fp8rl_grouped_gemm_blockscaled(xq, x_scale, wq, w_scale, d_offsets, num_experts, rows, n, k,
                                   y_bf16, fmt=SCALE_FP32, stream=None) -> None:
    _ok(load_library().fp8rl_grouped_gemm_blockscaled(_p(xq), _p(x_scale), _p(wq), _p(w_scale),
                                                      _p(d_offsets), num_experts, rows, n, k,
                                                      _p(y_bf16), fmt, _stream(stream)),
        "fp8rl_grouped_gemm_blockscaled")


def fp8rl_e4m3_encode(d_in, n, d_out, stream=None) -> None:
    _ok(load_library().fp8rl_e4m3_encode(_p(d_in), n, _p(d_out), _stream(stream)), "fp8rl_e4m3_encode")


DEBUG_RESET, DEBUG_GEMM_BN, DEBUG_FAULT_SKIP_KB, DEBUG_TIMEOUT_NS = 0, 1, 2, 3
DEBUG_WAIT_MODE, DEBUG_L2_PREFETCH, DEBUG_SPLITS, DEBUG_STREAMK, DEBUG_STREAMK_GRID = 4, 5, 6, 7, 8
DEBUG_OUT_STAGE, DEBUG_DECODE, DEBUG_MX, DEBUG_PAIR, DEBUG_PDL = 9, 10, 11, 12, 13


def fp8rl_debug_set(key, value) -> None:
    _ok(load_library().fp8rl_debug_set(int(key), int(value)), "fp8rl_debug_set")


def fp8rl_sync_status(stream=None) -> int:
    """Synchronise and return the status code (0 = OK, 6 = a device wait ran
    out).  With FP8RL_CANARY=1, also checks the guard zones of every output
    allocated since the last call (raises CanaryError)."""
    st = int(load_library().fp8rl_sync_status(_stream(stream)))
    if canaries_enabled():
        check_canaries()
    return st


def fp8rl_status_string(status: int) -> str:
    return load_library().fp8rl_status_string(int(status)).decode()


def fp8rl_version() -> int:
    return int(load_library().fp8rl_version())


# --------------------------------------------------------------------------- helpers

def _scale_dtype(fmt):
    return torch.float32 if fmt == SCALE_FP32 else torch.uint8


# ---------------------------------------------------------------- canary guards
# With FP8RL_CANARY=1 in the environment (a debugging aid, off by default),
# every output the helpers below allocate sits between two guard zones filled
# with a fixed byte; fp8rl_sync_status() checks every guard zone allocated
# since its last call and raises CanaryError if a kernel wrote outside its
# output.  The guarded buffers are kept alive until that check.
CANARY_BYTE = 0xA5
_CANARY_PRE = 4096           # bytes before the output (keeps its 256-byte alignment)
_CANARY_POST = 64 * 1024     # bytes after it (a ragged tile overrun lands here)
_guards = []
_guards_lock = threading.Lock()


class CanaryError(RuntimeError):
    pass


def canaries_enabled() -> bool:
    return os.environ.get("FP8RL_CANARY") == "1"


def _out(shape, dtype, device):
    """An output tensor: plain torch.empty, or guarded when FP8RL_CANARY=1."""
    numel = 1
    for d in shape:
        numel *= int(d)
    if not canaries_enabled() or numel == 0:
        return torch.empty(shape, dtype=dtype, device=device)
    nbytes = numel * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((_CANARY_PRE + nbytes + _CANARY_POST,), CANARY_BYTE, dtype=torch.uint8, device=device)
    with _guards_lock:
        _guards.append((buf, nbytes))
    return buf[_CANARY_PRE:_CANARY_PRE + nbytes].view(dtype).view(tuple(shape))


def check_canaries() -> int:
    """Check (and forget) every guarded output allocated so far; returns how
    many were checked, raises CanaryError naming the first damaged one."""
    with _guards_lock:
        guards = list(_guards)
        _guards.clear()
    for buf, nbytes in guards:
        pre = buf[:_CANARY_PRE]
        post = buf[_CANARY_PRE + nbytes:]
        if not bool((pre == CANARY_BYTE).all()) or not bool((post == CANARY_BYTE).all()):
            bad_pre = int((pre != CANARY_BYTE).sum())
            bad_post = int((post != CANARY_BYTE).sum())
            raise CanaryError(f"a kernel wrote outside an output of {nbytes} bytes: "
                              f"{bad_pre} guard bytes before it and {bad_post} after it changed")
    return len(guards)


def _check_cuda(*tensors):
    """The kernels dereference device pointers on the current device: every
    tensor argument of a helper must be a CUDA tensor on it (None and
    non-tensor arguments are skipped)."""
    cur = None
    for t in tensors:
        if not isinstance(t, torch.Tensor):
            continue
        if not t.is_cuda:
            raise ValueError("fp8rl helpers take CUDA tensors; a host tensor's pointer would reach the kernels")
        if cur is None:
            cur = torch.cuda.current_device()
        if t.device.index != cur:
            raise ValueError(f"a tensor on {t.device} while the current device is cuda:{cur}")


def _check_bf16_2d(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D bf16 tensor with unit column stride")


def quant_weight(w: torch.Tensor, fmt=SCALE_FP32, stream=None):
    """E4M3 codes (uint8 [n,k]) and block scales ([ceil(n/128), ceil(k/128)]) of w."""
    _check_cuda(w)
    _check_bf16_2d(w, "w")
    n, k = w.shape
    q = _out((n, k), torch.uint8, w.device)
    s = _out(((n + 127) // 128, (k + 127) // 128), _scale_dtype(fmt), w.device)
    fp8rl_quant_weight_blockwise(w, n, k, w.stride(0), q, k, s, fmt, stream)
    return q, s


def weight_descs(items):
    """fp8rl_weight_desc array from (w, q, scale) tensor triples."""
    arr = (WeightDesc * max(1, len(items)))()
    for i, (w, q, s) in enumerate(items):
        arr[i] = WeightDesc(w.data_ptr(), q.data_ptr(), s.data_ptr(), w.shape[0], w.shape[1],
                            w.stride(0), q.stride(0))
    return arr


def quant_weights_batched(weights, fmt=SCALE_FP32, stream=None, outputs=None):
    """Quantise a list of bf16 matrices in one pass; returns [(q, scale), ...]."""
    weights = list(weights)
    _check_cuda(*weights, *(t for pair in (outputs or ()) for t in pair))
    if outputs is None:
        outputs = []
        for w in weights:
            _check_bf16_2d(w, "w")
            n, k = w.shape
            outputs.append((_out((n, k), torch.uint8, w.device),
                            _out(((n + 127) // 128, (k + 127) // 128),
                                        dtype=_scale_dtype(fmt), device=w.device)))
    descs = weight_descs([(w, q, s) for w, (q, s) in zip(weights, outputs)])
    fp8rl_quant_weight_blockwise_batched(descs, len(weights), fmt, stream)
    return outputs


def quant_act(x: torch.Tensor, fmt=SCALE_FP32, stream=None):
    """E4M3 codes (uint8 [m,k]) and group scales ([ceil(k/128), m]) of x."""
    _check_cuda(x)
    _check_bf16_2d(x, "x")
    m, k = x.shape
    q = _out((m, k), torch.uint8, x.device)
    s = _out(((k + 127) // 128, m), _scale_dtype(fmt), x.device)
    fp8rl_quant_act_group(x, m, k, x.stride(0), q, k, s, fmt, stream)
    return q, s


def gemm_workspace(device=None) -> torch.Tensor:
    """A zero-filled workspace for fp8rl_gemm_blockscaled_ws on `device`."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        nbytes = fp8rl_gemm_workspace_size()
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def gemm(xq, x_scale, wq, w_scale, fmt=SCALE_FP32, out=None, stream=None, workspace=None):
    """bf16 Y [m, n] = block-scaled X W^T.  With a workspace (gemm_workspace),
    shapes that fill the SMs unevenly run the stream-K schedule."""
    _check_cuda(xq, x_scale, wq, w_scale, out, workspace)
    m, k = xq.shape
    n = wq.shape[0]
    if out is None:
        out = _out((m, n), torch.bfloat16, xq.device)
    if workspace is None:
        fp8rl_gemm_blockscaled(xq, x_scale, wq, w_scale, out, m, n, k, fmt, stream)
    else:
        fp8rl_gemm_blockscaled_ws(xq, x_scale, wq, w_scale, out, m, n, k, fmt, workspace,
                                  workspace.numel() * workspace.element_size(), stream)
    return out


def gemm_act_quant(x, wq, w_scale, fmt=SCALE_FP32, out=None, stream=None):
    """bf16 Y [m, n] = X W^T with X (bf16 [m, k]) quantised 1x128 on the way,
    plus the codes and scales (the results of quant_act(x) then gemm)."""
    _check_cuda(x, wq, w_scale, out)
    _check_bf16_2d(x, "x")
    m, k = x.shape
    n = wq.shape[0]
    if out is None:
        out = _out((m, n), torch.bfloat16, x.device)
    xq = _out((m, k), torch.uint8, x.device)
    sx = _out(((k + 127) // 128, m), _scale_dtype(fmt), x.device)
    fp8rl_gemm_act_quant(x, x.stride(0), wq, w_scale, out, m, n, k, fmt, xq, sx, stream)
    return out, xq, sx


def grouped_gemm(xq, x_scale, wq, w_scale, d_offsets, fmt=SCALE_FP32, out=None, stream=None):
    """bf16 Y [rows, n]: expert e's weights applied to its row segment."""
    _check_cuda(xq, x_scale, wq, w_scale, d_offsets, out)
    rows, k = xq.shape
    e, n, _ = wq.shape
    if out is None:
        out = _out((rows, n), torch.bfloat16, xq.device)
    fp8rl_grouped_gemm_blockscaled(xq, x_scale, wq, w_scale, d_offsets, e, rows, n, k, out, fmt,
                                   stream)
    return out


def quant_gate_up_interleaved(gate: torch.Tensor, up: torch.Tensor, fmt=SCALE_FP32, stream=None,
                              out=None):
    """Quantise a gate and an up weight ([..., inter, k] bf16, optionally with
    leading expert dimensions) straight into the interleaved fused layout that
    fp8rl_gemm_swiglu_quant consumes: 128-row blocks alternate gate, up.  One
    batched quantiser pass (one descriptor per 128-row block); returns
    (q [..., 2 * inter, k] uint8, scale [..., 2 * inter / 128, k / 128])."""
    _check_cuda(gate, up, *(out or ()))
    if gate.shape != up.shape or gate.dtype != torch.bfloat16 or up.dtype != torch.bfloat16:
        raise ValueError("gate and up must be bf16 tensors of one shape")
    *lead, inter, k = gate.shape
    if inter % 128 or k % 128:
        raise ValueError("inter and k must be multiples of 128")
    g2 = gate.reshape(-1, inter, k)
    u2 = up.reshape(-1, inter, k)
    if g2.stride(2) != 1 or u2.stride(2) != 1:
        raise ValueError("weights need unit column stride")
    experts = g2.shape[0]
    if out is None:
        q = _out((experts, 2 * inter, k), torch.uint8, gate.device)
        sc = _out((experts, 2 * inter // 128, k // 128), _scale_dtype(fmt), gate.device)
    else:
        q, sc = (t.view(experts, *t.shape[-2:]) for t in out)
    items = []
    for e in range(experts):
        for b in range(inter // 128):
            for half, src in ((0, g2[e]), (1, u2[e])):
                row = 256 * b + 128 * half
                items.append((src[128 * b:128 * b + 128], q[e, row:row + 128], sc[e, row // 128:row // 128 + 1]))
    for i in range(0, len(items), 256):
        chunk = items[i:i + 256]
        fp8rl_quant_weight_blockwise_batched(weight_descs(chunk), len(chunk), fmt, stream)
    return q.view(*lead, 2 * inter, k), sc.view(*lead, 2 * inter // 128, k // 128)


def gemm_swiglu_quant(xq, x_scale, wq_gate_up, w_scale_gate_up, fmt=SCALE_FP32, out=None, stream=None):
    """(hq [m, inter] uint8, h_scale [inter/128, m]) of SiLU(gate) * up."""
    _check_cuda(xq, x_scale, wq_gate_up, w_scale_gate_up, *(out or ()))
    m, k = xq.shape
    inter = wq_gate_up.shape[0] // 2
    if out is None:
        out = (_out((m, inter), torch.uint8, xq.device),
               _out((inter // 128, m), _scale_dtype(fmt), xq.device))
    fp8rl_gemm_swiglu_quant(xq, x_scale, wq_gate_up, w_scale_gate_up, m, inter, k, out[0], out[1], fmt, stream)
    return out


def grouped_gemm_swiglu_quant(xq, x_scale, wq_gate_up, w_scale_gate_up, d_offsets, fmt=SCALE_FP32, out=None,
                              stream=None):
    """Grouped (MoE) form of gemm_swiglu_quant."""
    _check_cuda(xq, x_scale, wq_gate_up, w_scale_gate_up, d_offsets, *(out or ()))
    rows, k = xq.shape
    e, n2, _ = wq_gate_up.shape
    inter = n2 // 2
    if out is None:
        out = (_out((rows, inter), torch.uint8, xq.device),
               _out((inter // 128, rows), _scale_dtype(fmt), xq.device))
    fp8rl_grouped_gemm_swiglu_quant(xq, x_scale, wq_gate_up, w_scale_gate_up, d_offsets, e, rows, inter, k,
                                    out[0], out[1], fmt, stream)
    return out


def kv_calibrate(k: torch.Tensor, v: torch.Tensor, q: torch.Tensor | None = None, out=None, stream=None):
    """Per-tensor fp32 scales (device float [3]: K, V, Q) of a calibration pass."""
    _check_cuda(k, v, q, out)
    for name, t in (("k", k), ("v", v)) + ((("q", q),) if q is not None else ()):
        _check_bf16_2d(t, name)
    scales = out if out is not None else _out((3,), torch.float32, k.device).zero_()
    tokens, dim = k.shape
    fp8rl_kv_calibrate(k, v, q, tokens, dim, k.stride(0), v.stride(0), 0 if q is None else q.shape[1],
                       0 if q is None else q.stride(0), scales, stream)
    return scales


def kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """Quantise rows of K and V into the E4M3 caches ([num_slots, kv_dim] uint8)."""
    _check_cuda(k, v, slot_mapping, k_cache, v_cache, scales)
    _check_bf16_2d(k, "k")
    _check_bf16_2d(v, "v")
    tokens, dim = k.shape
    fp8rl_kv_append(k, v, tokens, dim, k.stride(0), v.stride(0), slot_mapping, k_cache, v_cache,
                    k_cache.stride(0), k_cache.shape[0], scales, stream)


def moe_plan(topk: torch.Tensor, experts: int, workspace: torch.Tensor | None = None, stream=None):
    """Dispatch plan of replayed top-k indices (device int32 [T, k]): returns
    device int32 (offsets [E+1], row_of_pair [T*k], token_of_row [T*k])."""
    _check_cuda(topk, workspace)
    if topk.dtype != torch.int32 or topk.dim() != 2 or not topk.is_contiguous():
        raise ValueError("topk must be a contiguous int32 [tokens, k] tensor")
    tokens, k = topk.shape
    dev = topk.device
    need = fp8rl_moe_plan_workspace_size(tokens, k, experts)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    offsets = _out((experts + 1,), torch.int32, dev)
    row_of_pair = _out((tokens * k,), torch.int32, dev)
    token_of_row = _out((tokens * k,), torch.int32, dev)
    fp8rl_moe_plan(topk, tokens, k, experts, offsets, row_of_pair, token_of_row, workspace, workspace.numel(),
                   stream)
    return offsets, row_of_pair, token_of_row


def moe_dispatch_quant(x: torch.Tensor, row_of_pair: torch.Tensor, topk: int, fmt=SCALE_FP32, out=None,
                       stream=None):
    """The grouped activation of the dispatch: token t's 1x128 quantisation in
    rows row_of_pair[t * topk + j], (codes uint8 [R, K], scales [K/128, R]
    fp32 or uint8) with R = tokens * topk."""
    _check_cuda(x, row_of_pair, *(out or ()))
    _check_bf16_2d(x, "x")
    tokens, k = x.shape
    rows = row_of_pair.numel()
    if rows != tokens * topk:
        raise ValueError("row_of_pair must have tokens * topk entries")
    if out is None:
        q = _out((rows, k), torch.uint8, x.device)
        sdt = torch.float32 if fmt == SCALE_FP32 else torch.uint8
        s = _out(((k + 127) // 128, rows), sdt, x.device)
    else:
        q, s = out
    fp8rl_moe_dispatch_quant(x, tokens, k, x.stride(0), row_of_pair, topk, rows, q, q.stride(0), s, fmt, stream)
    return q, s


def moe_combine(y: torch.Tensor, row_of_pair: torch.Tensor, gate: torch.Tensor, out=None, stream=None):
    """bf16 [T, N]: each token's expert output rows weighted by its gates."""
    _check_cuda(y, row_of_pair, gate, out)
    _check_bf16_2d(y, "y")
    if gate.dtype != torch.float32 or gate.dim() != 2 or not gate.is_contiguous():
        raise ValueError("gate must be a contiguous fp32 [tokens, k] tensor")
    tokens, k = gate.shape
    n = y.shape[1]
    o = out if out is not None else _out((tokens, n), torch.bfloat16, y.device)
    fp8rl_moe_combine(y, y.shape[0], n, y.stride(0), row_of_pair, gate, tokens, k, o, o.stride(0), stream)
    return o


def tis_weights(lp_train: torch.Tensor, lp_rollout: torch.Tensor, mask: torch.Tensor | None = None,
                clip: float = 2.0, workspace: torch.Tensor | None = None, out=None, stream=None):
    """(w fp32 [n], kl fp64 [3] = mean, sum, count) on the device."""
    _check_cuda(lp_train, lp_rollout, mask, workspace, *(out or ()))
    for name, t in (("lp_train", lp_train), ("lp_rollout", lp_rollout)):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 tensor")
    if mask is not None and (mask.dtype != torch.uint8 or not mask.is_contiguous()):
        raise ValueError("mask must be a contiguous uint8 tensor")
    n = lp_train.numel()
    dev = lp_train.device
    need = fp8rl_tis_workspace_size(n)
    if workspace is None:
        workspace = torch.zeros(max(need, 32), dtype=torch.uint8, device=dev)  # header zeroed once
    w, kl = out if out is not None else (_out((n,), torch.float32, dev),
                                         _out((3,), torch.float64, dev))
    fp8rl_tis_weights(lp_train, lp_rollout, mask, n, clip, w, kl, workspace, workspace.numel(), stream)
    return w, kl


class HostWeightSync:
    """Weight sync from host memory: bf16 weights in pinned host buffers are
    quantised (128x128 blocks) into E4M3 codes and scales in pinned host
    buffers.

    Pipelined (default): one call of ``fp8rl_quant_weight_host_batched``, the
    library's copy-in / quantise / copy-out pipeline over chunks of whole
    128-row block rows; the device staging (``slots`` slots of about
    ``chunk_bytes`` of bf16 each) is allocated once, at construction.
    Direct: the quantiser itself reads the pinned bf16 weights and writes the
    codes and scales in host memory over the CPU-GPU link (one batched launch
    of ``fp8rl_quant_weight_blockwise_batched``, no staging).  ``run()`` only
    enqueues work on the current stream; the caller synchronises."""

    def __init__(self, host_weights, host_codes, host_scales, fmt=SCALE_FP32, chunk_bytes=32 << 20,
                 slots=3, device=None, direct=False):
        device = torch.device(device or "cuda")
        self.fmt = fmt
        self.direct = direct
        self.h2d_bytes = sum(w.numel() * 2 for w in host_weights)
        self.d2h_bytes = sum(q.numel() + s.numel() * s.element_size() for q, s in zip(host_codes, host_scales))
        for t in list(host_weights) + list(host_codes) + list(host_scales):
            if t.is_cuda:
                raise ValueError("HostWeightSync takes host tensors")
            if direct and not t.is_pinned():
                raise ValueError("direct mode needs pinned host tensors")
        self._keep = (list(host_weights), list(host_codes), list(host_scales))
        self.descs = weight_descs(list(zip(host_weights, host_codes, host_scales)))
        self.count = len(host_weights)
        if direct:
            return
        self.slots = slots
        need = 0
        for w in host_weights:
            n, k = w.shape
            if n == 0 or k == 0:
                continue
            rows = min(n, max(128, (chunk_bytes // (2 * k)) // 128 * 128))
            need = max(need, fp8rl_host_sync_staging_bytes(rows, k, slots, fmt))
        self.staging = torch.empty(max(need, 256), dtype=torch.uint8, device=device)

    def run(self):
        """Enqueue one full weight sync; returns immediately (the caller syncs)."""
        if self.direct:
            fp8rl_quant_weight_blockwise_batched(self.descs, self.count, self.fmt)
            return
        fp8rl_quant_weight_host_batched(self.descs, self.count, self.fmt, self.staging, self.staging.numel(),
                                        self.slots)
