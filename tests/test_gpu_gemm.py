"""GPU parity of the block-scaled W8A8 GEMMs (dense and MoE grouped) against
the fp64 CPU oracle, through the C ABI.

The E4M3 operands and their scales are produced by the ORACLE's quantisers on
the host and uploaded, so the GEMM is checked on inputs that never passed
through the CUDA path.  Bar: |gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref), with
rms over the whole reference output (over the sampled values where the oracle
evaluates a sample)."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu

FMTS = [fp8rl.SCALE_FP32, fp8rl.SCALE_UE8M0]
RTOL, ATOL_RMS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


@pytest.fixture(params=[0, 128, 256], ids=["bn-auto", "bn128", "bn256"])
def bn(request):
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_GEMM_BN, request.param)
    yield request.param
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_GEMM_BN, 0)


def within(got, ref, rms=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = RTOL * np.abs(ref) + ATOL_RMS * rms
    bad = int(np.count_nonzero(err > bound))
    assert bad == 0, f"{bad}/{ref.size} outside tolerance; worst excess {float((err - bound).max()):.3e}"


def oracle_operands(x_bf16, w_bf16, fmt):
    """Oracle-quantised operands (host numpy) for X [m,k] and W [n,k]."""
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x_bf16), fmt)
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w_bf16), fmt)
    return xq, sx, wq, sw


def to_dev(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


def run_gemm(xq, sx, wq, sw, fmt):
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    y = fp8rl.gemm(dx, dsx, dw, dsw, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    return y.float().cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_linear(fmt, bn):
    """256x256 weight with one all-zero block, 16 tokens."""
    w, x = synth.tiny_linear(0)
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    y = run_gemm(xq, sx, wq, sw, fmt)
    within(y, oracle.gemm_blockscaled(xq, sx, wq, sw, fmt))


def test_tiny_linear_zero_block_contributes_nothing():
    w, x = synth.tiny_linear(0)
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    y = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    # the product without K-block 1 for rows 0..127 of W equals Y there
    xq0, sx0 = xq.copy(), sx.copy()
    xq0[:, 128:] = 0
    ref = oracle.gemm_blockscaled(xq0, sx0, wq, sw)
    within(y[:, :128], ref[:, :128])


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m,n,k", [(1, 128, 128), (15, 256, 256), (129, 384, 1024), (300, 256, 640),
                                   (128, 512, 128), (257, 128, 384)])
def test_ragged_shapes(m, n, k, fmt, bn):
    if bn == 256 and n % 256:
        pytest.skip("tile width 256 needs n % 256 == 0 (falls back to 128)")
    x = synth.activation_bf16(m, k, 7, "gemm-ragged", m, n, k)
    w = synth.weight_bf16(n, k, 8, "gemm-ragged", m, n, k)
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    within(run_gemm(xq, sx, wq, sw, fmt), oracle.gemm_blockscaled(xq, sx, wq, sw, fmt))


def test_identity_weight_returns_rounded_activations():
    m, k = 64, 256
    x = synth.activation_bf16(m, k, 9, "gemm-id")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    wq = np.zeros((k, k), np.uint8)
    np.fill_diagonal(wq, 0x38)  # 1.0
    sw = np.ones((k // 128, k // 128), np.float32)
    y = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    xd = oracle.dequantize(xq, sx.T, 1, 128)
    # the kernel rounds the exact product once to fp32 (the FMA) and once to bf16
    expect = torch.from_numpy(xd.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("name,n,k", synth.QWEN3_8B_GEMMS)
@pytest.mark.parametrize("m", [16, 128])
def test_qwen3_8b_shapes_small_m_full(name, n, k, m):
    x = synth.activation_bf16(m, k, 10, "gemm-q", name, m)
    w = synth.weight_bf16(n, k, 11, "gemm-q", name)
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    within(run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32), oracle.gemm_blockscaled(xq, sx, wq, sw))


def sample_positions(m, n, rows_full, count, seed):
    rng = np.random.default_rng(seed)
    full_rows = np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, rows_full)]))
    rr = np.repeat(full_rows, n)
    cc = np.tile(np.arange(n), full_rows.size)
    rr = np.concatenate([rr, rng.integers(0, m, count)])
    cc = np.concatenate([cc, rng.integers(0, n, count)])
    return rr, cc


@pytest.mark.parametrize("name,n,k", synth.QWEN3_8B_GEMMS)
@pytest.mark.parametrize("m", [1024, 8192])
def test_qwen3_8b_shapes_large_m_sampled(name, n, k, m):
    """Full-size launch; the oracle evaluates 4 whole rows plus 4096 random outputs."""
    x = synth.activation_bf16(m, k, 12, "gemm-q", name, m)
    w = synth.weight_bf16(n, k, 13, "gemm-q", name)
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    y = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    rr, cc = sample_positions(m, n, 2, 4096, m + n)
    ref = oracle.gemm_blockscaled_at(xq, sx, wq, sw, rr, cc)
    within(y[rr, cc], ref)


def test_ue8m0_large_m_sampled():
    m, n, k = 8192, 24576, 4096
    x = synth.activation_bf16(m, k, 14, "gemm-ue")
    w = synth.weight_bf16(n, k, 15, "gemm-ue")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_UE8M0)
    y = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_UE8M0)
    rr, cc = sample_positions(m, n, 2, 4096, 3)
    within(y[rr, cc], oracle.gemm_blockscaled_at(xq, sx, wq, sw, rr, cc, fp8rl.SCALE_UE8M0))


def test_m_zero_is_a_no_op():
    y = torch.full((1, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    xq = torch.zeros((1, 128), dtype=torch.uint8, device="cuda")
    fp8rl.fp8rl_gemm_blockscaled(xq, xq, xq, xq, y, 0, 128, 128)
    assert fp8rl.fp8rl_sync_status() == 0 and float(y[0, 0]) == 7.0


# --------------------------------------------------------------------------- grouped

def grouped_case(counts, n, k, fmt, seed):
    offsets = synth.routing_with_counts(counts)
    rows = int(offsets[-1])
    e = len(counts)
    x = synth.normal_bf16((max(rows, 1), k), 1.0, seed, "grp-x", n, k)[:rows]
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    ws = synth.moe_expert_weights(n, k, e, seed, 0, f"grp{n}x{k}")
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(ws.reshape(e * n, k)), fmt)
    wq = wq.reshape(e, n, k)
    sw = sw.reshape(e, n // 128, k // 128)
    return offsets, xq, sx, wq, sw


def run_grouped(offsets, xq, sx, wq, sw, fmt, fill=None):
    dx, dsx, dw, dsw, doff = to_dev(xq, sx, wq, sw, offsets)
    rows, n = xq.shape[0], wq.shape[1]
    out = torch.empty((rows, n), dtype=torch.bfloat16, device="cuda")
    if fill is not None:
        out.fill_(fill)
    fp8rl.grouped_gemm(dx, dsx, dw, dsw, doff, fmt, out=out)
    assert fp8rl.fp8rl_sync_status() == 0
    return out.float().cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [[3, 0, 200, 129], [128, 128], [0, 0, 5], [1], [300, 0, 0, 1, 0]])
def test_grouped_small_full(counts, fmt, bn):
    n, k = 256, 384
    offsets, xq, sx, wq, sw = grouped_case(counts, n, k, fmt, sum(counts))
    y = run_grouped(offsets, xq, sx, wq, sw, fmt)
    within(y, oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, offsets, fmt))


@pytest.mark.parametrize("experts", [256, 257, 300])
def test_grouped_many_experts(experts):
    """Expert counts at and past the shared-memory map of segments (256): the
    map's lookup and the scan over the offsets in global memory give the
    oracle's results; many experts are empty, a few hold ragged segments."""
    rng = np.random.default_rng(experts)
    counts = [int(c) if rng.random() < 0.3 else 0 for c in rng.integers(1, 300, experts)]
    counts[-1] = 131  # the last expert holds rows
    n, k = 256, 256
    offsets, xq, sx, wq, sw = grouped_case(counts, n, k, fp8rl.SCALE_FP32, experts)
    y = run_grouped(offsets, xq, sx, wq, sw, fp8rl.SCALE_FP32, fill=7.0)
    within(y, oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, offsets, fp8rl.SCALE_FP32))


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_grouped_qwen3_30b_a3b_sampled(which):
    """128 experts, T = 4096 tokens routed top-8 by replayed indices; the
    oracle evaluates the first and last row of every non-empty segment plus
    4096 random outputs."""
    r = synth.moe_routing(4096, 128, 8, seed=0, layer=0)
    offsets = oracle.moe_dispatch_plan(r.topk, synth.MOE_EXPERTS)[0]
    n, k = (1536, 2048) if which == "gate_up" else (2048, 768)
    rows = int(offsets[-1])
    x = synth.normal_bf16((rows, k), 1.0, 0, "moe-x", which)
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    ws = synth.moe_expert_weights(n, k, 128, 0, 0, which)
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(ws.reshape(-1, k)))
    wq = wq.reshape(128, n, k)
    sw = sw.reshape(128, n // 128, k // 128)
    y = run_grouped(offsets, xq, sx, wq, sw, fp8rl.SCALE_FP32)
    rng = np.random.default_rng(5)
    edge_rows = []
    for e in range(128):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            edge_rows += [a, b - 1]
    er = np.array(edge_rows)
    rr = np.concatenate([er, rng.integers(0, rows, 4096)])
    cc = np.concatenate([rng.integers(0, n, er.size), rng.integers(0, n, 4096)])
    ref = oracle.grouped_gemm_blockscaled_at(xq, sx, wq, sw, offsets, rr, cc)
    within(y[rr, cc], ref)


def test_grouped_rows_outside_offsets_untouched():
    """Offsets that end before `rows`: the trailing rows belong to no expert and
    are left as they were."""
    counts = [5, 7]
    offsets, xq, sx, wq, sw = grouped_case(counts, 128, 128, fp8rl.SCALE_FP32, 1)
    extra = 9
    xq2 = np.concatenate([xq, np.zeros((extra, 128), np.uint8)])
    sx2 = np.concatenate([sx, np.ones((1, extra), np.float32)], axis=1)
    y = run_grouped(offsets, xq2, sx2, wq, sw, fp8rl.SCALE_FP32, fill=3.0)
    assert np.all(y[12:] == 3.0)
    within(y[:12], oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, offsets))


# --------------------------------------------------------------------------- split-K clusters

@pytest.fixture
def force_splits(request):
    yield lambda s: fp8rl.fp8rl_debug_set(6, s)
    fp8rl.fp8rl_debug_set(6, 0)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("splits", [2, 3, 4, 8])
@pytest.mark.parametrize("m,n,k", [(1, 128, 256), (16, 384, 1280), (100, 256, 640), (128, 128, 1024),
                                   (200, 256, 2048)])
def test_split_k_cluster(m, n, k, splits, fmt, force_splits):
    """K split over a cluster, partial tiles summed through distributed shared
    memory; uneven splits (k/128 not a multiple of the split count) included."""
    force_splits(splits)
    x = synth.activation_bf16(m, k, 21, "splitk", m, n, k)
    w = synth.weight_bf16(n, k, 22, "splitk", m, n, k)
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    within(run_gemm(xq, sx, wq, sw, fmt), oracle.gemm_blockscaled(xq, sx, wq, sw, fmt))


def test_split_k_is_deterministic(force_splits):
    force_splits(4)
    x = synth.activation_bf16(16, 4096, 23, "splitk-det")
    w = synth.weight_bf16(512, 4096, 24, "splitk-det")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    y1 = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    y2 = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    assert np.array_equal(y1, y2)


# --------------------------------------------------------------------------- stream-K (workspace)

@pytest.fixture(scope="module")
def workspace():
    return fp8rl.gemm_workspace()


@pytest.fixture
def force_streamk():
    def set_(grid, bn=0):
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_STREAMK, 2)
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_STREAMK_GRID, grid)
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_GEMM_BN, bn)
    yield set_
    for key in (fp8rl.DEBUG_STREAMK, fp8rl.DEBUG_STREAMK_GRID, fp8rl.DEBUG_GEMM_BN):
        fp8rl.fp8rl_debug_set(key, 0)


def run_gemm_ws(xq, sx, wq, sw, fmt, ws):
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    y = fp8rl.gemm(dx, dsx, dw, dsw, fmt, workspace=ws)
    assert fp8rl.fp8rl_sync_status() == 0
    return y.float().cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("m,n,k,grid", [
    (33, 256, 1280, 4),     # one tile of 10 K chunks over 4 CTAs: two CTAs hold only inner chunks
    (129, 256, 1024, 3),    # two m-tiles, ranges crossing tile boundaries
    (300, 512, 640, 7),     # ragged rows, 7 CTAs
    (256, 256, 256, 16),    # fewer K iterations than CTAs asked for: one iteration per CTA
    (1000, 768, 2048, 0),   # one CTA per SM
    (128, 1024, 128, 5),    # a single K chunk per tile: no tile is ever split
])
def test_stream_k_forced(m, n, k, grid, bn, fmt, workspace, force_streamk):
    if bn == 256 and n % 256:
        pytest.skip("tile width 256 needs n % 256 == 0")
    force_streamk(grid, bn)
    x = synth.activation_bf16(m, k, 31, "streamk", m, n, k)
    w = synth.weight_bf16(n, k, 32, "streamk", m, n, k)
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    within(run_gemm_ws(xq, sx, wq, sw, fmt, workspace), oracle.gemm_blockscaled(xq, sx, wq, sw, fmt))


@pytest.mark.parametrize("name,n,k", synth.QWEN3_8B_GEMMS)
def test_stream_k_qwen3_8b_m1024_sampled(name, n, k, workspace):
    """At M = 1024 the workspace entry point chooses stream-K on its own where
    whole tiles would leave the last wave nearly empty (qkv, gate-up) and whole
    tiles elsewhere; 4 whole rows + 4096 random outputs."""
    m = 1024
    x = synth.activation_bf16(m, k, 12, "gemm-q", name, m)
    w = synth.weight_bf16(n, k, 13, "gemm-q", name)
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    y = run_gemm_ws(xq, sx, wq, sw, fp8rl.SCALE_FP32, workspace)
    rr, cc = sample_positions(m, n, 2, 4096, m + n)
    within(y[rr, cc], oracle.gemm_blockscaled_at(xq, sx, wq, sw, rr, cc))


def test_stream_k_repeated_calls_are_identical(workspace, force_streamk):
    """Every call advances the workspace epoch; five calls in a row give the
    same bits, and the same as a fresh workspace."""
    force_streamk(9, 256)
    x = synth.activation_bf16(200, 2048, 33, "streamk-det")
    w = synth.weight_bf16(512, 2048, 34, "streamk-det")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    ys = [run_gemm_ws(xq, sx, wq, sw, fp8rl.SCALE_FP32, workspace) for _ in range(5)]
    ys.append(run_gemm_ws(xq, sx, wq, sw, fp8rl.SCALE_FP32, fp8rl.gemm_workspace()))
    for y in ys[1:]:
        assert np.array_equal(ys[0], y)
    within(ys[0], oracle.gemm_blockscaled(xq, sx, wq, sw))


def test_stream_k_short_workspace_is_rejected(workspace):
    xq = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 64), dtype=torch.float32, device="cuda")
    y = torch.empty((64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8rl.Fp8rlError) as e:
        fp8rl.fp8rl_gemm_blockscaled_ws(xq, s, xq, s, y, 64, 128, 128, fp8rl.SCALE_FP32, workspace,
                                        workspace.numel() - 1)
    assert e.value.status == 1


# --------------------------------------------------------------------------- tile stores

@pytest.fixture
def out_stage():
    # small shapes would take split-K clusters: force the data-parallel kernel
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, 1)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_OUT_STAGE, 0)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, 0)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m,n,k", [(300, 512, 512), (129, 384, 256), (1000, 768, 384), (33, 256, 256)])
def test_tile_stores_through_shared_memory_match_register_stores(m, n, k, fmt, bn, out_stage):
    """The data-parallel kernel stores finished tiles either from registers
    or through shared memory and TMA stores (boxes of 32 rows clipped at the
    last row): the same bits either way, and within tolerance of the oracle.
    Rows past M keep what the output held."""
    x = synth.activation_bf16(m, k, m + n, "stage-x")
    w = synth.weight_bf16(n, k, m + k, "stage-w")
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    outs = []
    for mode in (1, 2):
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_OUT_STAGE, mode)
        full = torch.full((m + 40, n), 7.0, dtype=torch.bfloat16, device="cuda")
        fp8rl.gemm(dx, dsx, dw, dsw, fmt, out=full[:m])
        assert fp8rl.fp8rl_sync_status() == 0
        assert bool((full[m:] == 7.0).all())
        outs.append(full[:m].cpu())
    assert torch.equal(outs[0], outs[1])
    within(outs[0].float().numpy(), oracle.gemm_blockscaled(xq, sx, wq, sw, fmt))


@pytest.mark.parametrize("counts", [[3, 0, 200, 129], [64, 31, 1, 160], [256, 256], [40, 0, 300]])
def test_grouped_tile_stores_respect_segment_ends(counts, bn, out_stage):
    """Grouped: boxes that would cross a segment end are stored row by row;
    both store paths give the same bits and leave rows outside the offsets
    untouched."""
    n, k = 256, 384
    offsets, xq, sx, wq, sw = grouped_case(counts, n, k, fp8rl.SCALE_FP32, 7 + sum(counts))
    outs = []
    for mode in (1, 2):
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_OUT_STAGE, mode)
        outs.append(run_grouped(offsets, xq, sx, wq, sw, fp8rl.SCALE_FP32, fill=3.0))
    assert np.array_equal(outs[0], outs[1])
    within(outs[0], oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, offsets, fp8rl.SCALE_FP32))


# --------------------------------------------------------------------------- decode kernel

@pytest.fixture
def decode_mode():
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, 0)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, 0)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m,n,k,splits", [(16, 6144, 4096, 0), (1, 4096, 4096, 0), (32, 4096, 12288, 0),
                                          (17, 384, 640, 3), (5, 256, 1280, 8), (31, 128, 256, 2),
                                          (16, 24576, 4096, 0),
                                          # 64 and 128 token columns (forced: 33..128 rows)
                                          (33, 384, 640, 3), (64, 4096, 4096, 0), (50, 256, 2048, 8),
                                          (65, 6144, 4096, 0), (128, 4096, 12288, 0), (100, 128, 384, 2),
                                          (128, 24576, 4096, 0)])
def test_decode_kernel_matches_oracle_and_tile_kernel(m, n, k, splits, fmt, decode_mode):
    """At most 64 rows (up to 128 for narrow weights with fp32 scales) the
    dense GEMM runs the swapped-operand decode kernel (weight rows as the
    MMA's M, tokens as its N, split K over a cluster), and up to 128 for any
    shape when the test hook asks for it; within tolerance of the oracle over
    the whole output, and of the 128-row-tile kernel that the hook selects
    instead."""
    x = synth.activation_bf16(m, k, m + 3, "dec-x", n)
    w = synth.weight_bf16(n, k, k + 5, "dec-w")
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    ref = oracle.gemm_blockscaled(xq, sx, wq, sw, fmt)
    if splits:
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, splits)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, 1)
    y_dec = run_gemm(xq, sx, wq, sw, fmt)
    within(y_dec, ref)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, 2)
    y_tile = run_gemm(xq, sx, wq, sw, fmt)
    within(y_tile, ref)
    # both round once from fp32 sums of the same products (orders differ)
    assert np.max(np.abs(y_dec - y_tile)) <= 2.0 ** -7 * np.max(np.abs(ref)) + 1e-6


@pytest.mark.parametrize("m,n,k,kernel", [(128, 4096, 4096, 1), (100, 4096, 12288, 1), (128, 6144, 4096, 2),
                                          (128, 24576, 4096, 2), (128, 4096, 2048, 2)])
def test_default_kernel_between_65_and_128_rows(m, n, k, kernel, decode_mode):
    """The default choice at 65..128 rows (fp32 scales): the decode kernel
    for weights of at most SMs / 4 blocks of 128 rows with K >= 4096, the
    128-row-tile kernel otherwise; the default's output is bit for bit that
    of the kernel the test hook forces, and within tolerance of the oracle."""
    x = synth.activation_bf16(m, k, m + 7, "dec-default-x", n)
    w = synth.weight_bf16(n, k, k + 9, "dec-default-w")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    y = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, kernel)
    y_forced = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    assert np.array_equal(y.view(np.uint32), y_forced.view(np.uint32))
    within(y, oracle.gemm_blockscaled(xq, sx, wq, sw))


def test_decode_kernel_is_deterministic(decode_mode):
    x = synth.activation_bf16(16, 4096, 3, "dec-det")
    w = synth.weight_bf16(6144, 4096, 4, "dec-det-w")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_FP32)
    a = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    b = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_FP32)
    assert np.array_equal(a, b)


# --------------------------------------------------------------------------- UE8M0 on the block-scaled MMA

@pytest.fixture(params=[2, 1], ids=["mx", "promote"])
def mx_mode(request):
    """UE8M0 tiles on the tensor cores' block-scaled MMA (2; the default for
    K >= 2048) or on the per-chunk fp32 promotion (1)."""
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, request.param)
    yield request.param
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 0)


def exact_operands(m, n, k, seed, experts=1):
    """Integer-valued E4M3 codes in [-4, 4] and UE8M0 scale bytes in
    [125, 129] (2^-2 .. 2^2), drawn independently per row, weight block and K
    chunk: every partial sum of the product is a multiple of 2^-4 below 2^17,
    so fp32 accumulation in any order is exact and Y is bf16_rne of the exact
    value."""
    rng = np.random.default_rng(seed)
    xq = oracle.e4m3_encode_array(rng.integers(-4, 5, size=(m, k)).astype(np.float32))
    wq = oracle.e4m3_encode_array(rng.integers(-4, 5, size=(experts * n, k)).astype(np.float32))
    sx = rng.integers(125, 130, size=(k // 128, m)).astype(np.uint8)
    sw = rng.integers(125, 130, size=(experts * n // 128, k // 128)).astype(np.uint8)
    return xq, sx, wq, sw


def bf16_bits_of(y):
    return torch.from_numpy(np.asarray(y, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


@pytest.mark.parametrize("m,n,k", [(300, 512, 512), (128, 256, 256), (1, 128, 384), (257, 384, 512)])
def test_power_of_two_scales_exact(m, n, k, bn, mx_mode):
    """With exact partial sums both UE8M0 paths must give bf16_rne of the
    exact product bit for bit, and so must the fp32-scale path given the same
    powers of two as fp32 scales: a scale applied to the wrong row, column or
    K chunk shows as a wrong bit."""
    xq, sx, wq, sw = exact_operands(m, n, k, m * 7 + n + k)
    ref_bits = bf16_bits_of(oracle.gemm_blockscaled(xq, sx, wq, sw, fp8rl.SCALE_UE8M0))
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    y = fp8rl.gemm(dx, dsx, dw, dsw, fp8rl.SCALE_UE8M0)
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(y.view(torch.int16).cpu().numpy(), ref_bits)
    fx = np.ldexp(1.0, sx.astype(np.int32) - 127).astype(np.float32)
    fw = np.ldexp(1.0, sw.astype(np.int32) - 127).astype(np.float32)
    dfx, dfw = to_dev(fx, fw)
    y32 = fp8rl.gemm(dx, dfx, dw, dfw, fp8rl.SCALE_FP32)
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(y32.view(torch.int16).cpu().numpy(), ref_bits)


@pytest.mark.parametrize("counts", [[3, 0, 200, 129], [128, 128], [0, 0, 5], [300, 0, 0, 1, 0]])
def test_power_of_two_scales_exact_grouped(counts, bn, mx_mode):
    """The same exactness over expert segments (segments ending inside tiles,
    empty experts); rows outside the offsets keep what the output held."""
    n, k = 256, 384
    offsets = synth.routing_with_counts(counts)
    rows, e = int(offsets[-1]), len(counts)
    xq, sx, wq, sw = exact_operands(rows, n, k, 11 + sum(counts), experts=e)
    wq = wq.reshape(e, n, k)
    sw = sw.reshape(e, n // 128, k // 128)
    ref_bits = bf16_bits_of(oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, offsets, fp8rl.SCALE_UE8M0))
    dx, dsx, dw, dsw, doff = to_dev(xq, sx, wq, sw, offsets)
    out = torch.full((rows + 16, n), 5.0, dtype=torch.bfloat16, device="cuda")
    fp8rl.grouped_gemm(dx, dsx, dw, dsw, doff, fp8rl.SCALE_UE8M0, out=out[:rows])
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(out[:rows].view(torch.int16).cpu().numpy(), ref_bits)
    assert bool((out[rows:] == 5.0).all())


@pytest.mark.parametrize("m,n,k", [(300, 512, 512), (129, 384, 1024), (2000, 768, 384)])
def test_ue8m0_paths_match_oracle(m, n, k, bn, mx_mode):
    """Quantised activations with outlier channels and N(0, 0.02) weights:
    both UE8M0 paths within the stated tolerance of the fp64 oracle."""
    x = synth.activation_bf16(m, k, m + 3, "mx-x")
    w = synth.weight_bf16(n, k, n + 5, "mx-w")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_UE8M0)
    within(run_gemm(xq, sx, wq, sw, fp8rl.SCALE_UE8M0), oracle.gemm_blockscaled(xq, sx, wq, sw, fp8rl.SCALE_UE8M0))


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_grouped_ue8m0_qwen3_30b_a3b_sampled(which, mx_mode):
    """The Qwen3-30B-A3B-shaped expert layer (128 experts, 32768 routed rows)
    with UE8M0 scales, on the block-scaled MMA and on the per-chunk promotion:
    first and last row of every non-empty segment plus 4096 random outputs."""
    fmt = fp8rl.SCALE_UE8M0
    n, k = (2 * synth.MOE_INTER, synth.MOE_HIDDEN) if which == "gate_up" else (synth.MOE_HIDDEN, synth.MOE_INTER)
    r = synth.moe_routing(4096, synth.MOE_EXPERTS, synth.MOE_TOPK, 3, 0)
    offsets = oracle.moe_dispatch_plan(r.topk, synth.MOE_EXPERTS)[0]
    rows = int(offsets[-1])
    x = synth.normal_bf16((rows, k), 1.0, 31, "grp-ue-x", which)
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    ws = synth.moe_expert_weights(n, k, synth.MOE_EXPERTS, 32, 0, which)
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(ws.reshape(-1, k)), fmt)
    wq = wq.reshape(synth.MOE_EXPERTS, n, k)
    sw = sw.reshape(synth.MOE_EXPERTS, n // 128, k // 128)
    y = run_grouped(offsets, xq, sx, wq, sw, fmt)
    seg_rows = [int(v) for e in range(synth.MOE_EXPERTS) if offsets[e + 1] > offsets[e]
                for v in (offsets[e], offsets[e + 1] - 1)]
    rng = np.random.default_rng(9)
    rr = np.concatenate([np.repeat(np.array(seg_rows), 4), rng.integers(0, rows, 4096)]).astype(np.int64)
    cc = np.concatenate([rng.integers(0, n, 4 * len(seg_rows)), rng.integers(0, n, 4096)]).astype(np.int64)
    ref = oracle.grouped_gemm_blockscaled_at(xq, sx, wq, sw, offsets, rr, cc, fmt)
    within(y[rr, cc], ref)


# --------------------------------------------------------------------------- tensor-core pairs

@pytest.fixture(params=[1, 2], ids=["pair", "single"])
def pair_mode(request):
    """Dense UE8M0 tiles forced onto tensor-core pairs (1) or kept on single
    CTAs (2), both on the block-scaled MMA (forced: short K chooses the
    per-chunk promotion)."""
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 2)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, request.param)
    yield request.param
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, 0)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 0)


@pytest.mark.parametrize("m,n,k", [(300, 512, 512),     # second pair: rows 256..299 in its even CTA only
                                   (129, 256, 1024),    # one pair, its odd CTA holds a single row
                                   (256, 256, 256), (1000, 768, 384), (513, 1280, 640)])
def test_pair_matches_oracle(m, n, k, pair_mode):
    fmt = fp8rl.SCALE_UE8M0
    x = synth.activation_bf16(m, k, m + 21, "pair-x")
    w = synth.weight_bf16(n, k, n + 23, "pair-w")
    xq, sx, wq, sw = oracle_operands(x, w, fmt)
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    full = torch.full((m + 8, n), 9.0, dtype=torch.bfloat16, device="cuda")
    fp8rl.gemm(dx, dsx, dw, dsw, fmt, out=full[:m])
    assert fp8rl.fp8rl_sync_status() == 0
    assert bool((full[m:] == 9.0).all()), "rows past M were written"
    within(full[:m].float().cpu().numpy(), oracle.gemm_blockscaled(xq, sx, wq, sw, fmt))


@pytest.mark.parametrize("m,n,k", [(300, 512, 512), (257, 256, 768), (640, 768, 256), (2048, 512, 1024)])
def test_pair_power_of_two_scales_exact(m, n, k, pair_mode):
    """Exact partial sums: bf16_rne of the exact product bit for bit, so every
    row's and column's scale factor of every K chunk reached the right place
    in both CTAs of a pair."""
    xq, sx, wq, sw = exact_operands(m, n, k, m + 2 * n + k)
    ref_bits = bf16_bits_of(oracle.gemm_blockscaled(xq, sx, wq, sw, fp8rl.SCALE_UE8M0))
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    y = fp8rl.gemm(dx, dsx, dw, dsw, fp8rl.SCALE_UE8M0)
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(y.view(torch.int16).cpu().numpy(), ref_bits)


@pytest.mark.parametrize("name,n,k", synth.QWEN3_8B_GEMMS)
def test_pair_qwen3_8b_m8192_sampled(name, n, k):
    """The full-size UE8M0 launches on tensor-core pairs (forced): 4 whole
    rows and 4096 random outputs against the oracle."""
    m = 8192
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 2)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, 1)
    try:
        x = synth.activation_bf16(m, k, 16, "pair-big", name)
        w = synth.weight_bf16(n, k, 17, "pair-big", name)
        xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_UE8M0)
        y = run_gemm(xq, sx, wq, sw, fp8rl.SCALE_UE8M0)
    finally:
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, 0)
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 0)
    rr, cc = sample_positions(m, n, 4, 4096, n + k)
    within(y[rr, cc], oracle.gemm_blockscaled_at(xq, sx, wq, sw, rr, cc, fp8rl.SCALE_UE8M0))


def test_pair_is_deterministic():
    m, n, k = 1024, 1024, 1024
    x = synth.activation_bf16(m, k, 18, "pair-det")
    w = synth.weight_bf16(n, k, 19, "pair-det")
    xq, sx, wq, sw = oracle_operands(x, w, fp8rl.SCALE_UE8M0)
    dx, dsx, dw, dsw = to_dev(xq, sx, wq, sw)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 2)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, 1)
    try:
        ys = [fp8rl.gemm(dx, dsx, dw, dsw, fp8rl.SCALE_UE8M0) for _ in range(3)]
        assert fp8rl.fp8rl_sync_status() == 0
    finally:
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, 0)
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 0)
    assert all(torch.equal(ys[0].view(torch.int16), y.view(torch.int16)) for y in ys[1:])
