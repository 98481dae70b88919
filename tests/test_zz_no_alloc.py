"""fp8rl_gemm_blockscaled_static (stream-K scratch in a fixed device array of
the library, nothing allocated per call) against the workspace entry point
fp8rl_gemm_blockscaled_ws: the two run the same kernel with the same grid, so
the outputs must agree bit for bit, on the first call and on the next one
(which finds the scratch as the first left it).  Named to be collected last,
so that it also runs after every other GPU test in one session."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


def operands(m, n, k, fmt, seed):
    x = synth.activation_bf16(m, k, seed, "static-x", m, n, k)
    w = synth.weight_bf16(n, k, seed + 1, "static-w", m, n, k)
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (xq, sx, wq, sw)]


@pytest.mark.parametrize("fmt", [fp8rl.SCALE_FP32, fp8rl.SCALE_UE8M0])
@pytest.mark.parametrize("m,n,k,grid", [
    (1024, 6144, 4096, None),   # stream-K chosen on its own (last wave of whole tiles ~1/4 full)
    (300, 512, 640, 7),         # forced stream-K, 7 CTAs, ragged rows
    (33, 256, 1280, 4),         # one tile split over four CTAs
    (256, 4096, 4096, None),    # split-K clusters chosen: the scratch is not touched
])
def test_static_scratch_matches_workspace_entry_point(m, n, k, grid, fmt):
    if grid is not None:
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_STREAMK, 2)
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_STREAMK_GRID, grid)
    xq, sx, wq, sw = operands(m, n, k, fmt, 41)
    ws = fp8rl.gemm_workspace()
    ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    fp8rl.fp8rl_gemm_blockscaled_ws(xq, sx, wq, sw, ref, m, n, k, fmt, ws, ws.numel())
    assert fp8rl.fp8rl_sync_status() == 0
    for _ in range(2):  # two calls in a row
        y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        fp8rl.fp8rl_gemm_blockscaled_static(xq, sx, wq, sw, y, m, n, k, fmt)
        assert fp8rl.fp8rl_sync_status() == 0
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_static_scratch_rejects_bad_arguments_before_set_up():
    a16 = 1 << 20
    lib = fp8rl.load_library()
    assert lib.fp8rl_gemm_blockscaled_static(None, a16, a16, a16, a16, 16, 256, 256, 0, None) == 1
    assert lib.fp8rl_gemm_blockscaled_static(a16, a16, a16, a16, a16, 16, 200, 256, 0, None) == 2
    assert lib.fp8rl_gemm_blockscaled_static(a16, a16, a16, a16, a16, 0, 256, 256, 0, None) == 0
