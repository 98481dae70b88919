"""GPU parity of the quantisers against the CPU oracle (bit-exact codes and
scales), through the C ABI.  Inputs are drawn once on the host and handed to
both sides."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu

FMTS = [fp8rl.SCALE_FP32, fp8rl.SCALE_UE8M0]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)


def _np(t):
    return t.cpu().numpy()


def _assert_weight_parity(w_cpu, fmt, ldw_pad=0):
    n, k = w_cpu.shape
    dev = torch.device("cuda")
    if ldw_pad:
        big = torch.zeros((n, k + ldw_pad), dtype=torch.bfloat16)
        big[:, :k] = w_cpu
        wd = big.to(dev)[:, :k]
    else:
        wd = w_cpu.to(dev)
    q, s = fp8rl.quant_weight(wd, fmt)
    torch.cuda.synchronize()
    qo, so = oracle.quant_weight_blockwise(synth.bf16_bits(w_cpu), fmt)
    assert np.array_equal(_np(q), qo), "E4M3 codes differ"
    assert np.array_equal(_np(s).view(np.uint8), so.view(np.uint8)), "scales differ"


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_linear_weight_bit_exact(fmt):
    w, _ = synth.tiny_linear(0)
    _assert_weight_parity(w, fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(384, 512), (200, 300), (130, 136), (1, 1), (129, 128), (128, 129)])
def test_weight_ragged_and_multi_tile_bit_exact(n, k, fmt):
    w = synth.weight_bf16(n, k, 1, "gpu-w", n, k)
    _assert_weight_parity(w, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_weight_padded_leading_dimension(fmt):
    w = synth.weight_bf16(256, 256, 2, "gpu-ld")
    _assert_weight_parity(w, fmt, ldw_pad=8)   # 16-byte rows: vector path
    _assert_weight_parity(w, fmt, ldw_pad=3)   # odd stride: scalar path


@pytest.mark.parametrize("fmt", FMTS)
def test_weight_extreme_magnitudes(fmt):
    """Blocks at the ends of the bf16 range, subnormal amax, and mixed signs."""
    rng = np.random.default_rng(3)
    w = synth.weight_bf16(512, 256, 3, "gpu-ext").float()
    w[0:128, 0:128] *= 1e36          # near the top of the range
    w[0:128, 128:256] *= 1e-36       # tiny normals
    w[128:256, 0:128] = torch.from_numpy(rng.standard_normal((128, 128)).astype(np.float32)) * 1e-39
    w[128:256, 128:256] = 0.0
    w[128, 130] = -0.0
    w[256:384, :] = 448.0
    w[384:512, :] = torch.from_numpy(rng.choice([-1.0, 1.0], (128, 256)).astype(np.float32))
    _assert_weight_parity(w.to(torch.bfloat16), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_qwen3_8b_layer_weight_sync_bit_exact(fmt):
    """The seven linears of one Qwen3-8B-shaped layer, in one batched call."""
    layer = synth.qwen3_8b_layer(0, 0)
    dev = torch.device("cuda")
    wd = [w.to(dev) for _, w in layer]
    outs = fp8rl.quant_weights_batched(wd, fmt)
    torch.cuda.synchronize()
    for (name, w), (q, s) in zip(layer, outs):
        qo, so = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
        assert np.array_equal(_np(q), qo), name
        assert np.array_equal(_np(s).view(np.uint8), so.view(np.uint8)), name


def test_batched_equals_single_calls_with_many_descriptors():
    """More descriptors than one launch holds, with ragged shapes mixed in."""
    dev = torch.device("cuda")
    shapes = [(128 + (i % 5) * 37, 128 + (i % 3) * 64) for i in range(300)]
    ws = [synth.weight_bf16(n, k, 4, "gpu-many", i, outliers=False, device=dev) for i, (n, k) in enumerate(shapes)]
    outs = fp8rl.quant_weights_batched(ws)
    for w, (q, s) in zip(ws, outs):
        q1, s1 = fp8rl.quant_weight(w)
        assert torch.equal(q, q1) and torch.equal(s, s1)
    # and spot-check a few against the oracle
    for i in (0, 7, 299):
        qo, so = oracle.quant_weight_blockwise(synth.bf16_bits(ws[i]))
        assert np.array_equal(_np(outs[i][0]), qo) and np.array_equal(_np(outs[i][1]), so)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m,k", [(16, 256), (1, 128), (5, 300), (129, 4096), (1024, 12288), (3, 1)])
def test_act_quant_bit_exact(m, k, fmt):
    x = synth.activation_bf16(m, k, 5, "gpu-act", m, k)
    q, s = fp8rl.quant_act(x.cuda(), fmt)
    torch.cuda.synchronize()
    qo, so = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    assert np.array_equal(_np(q), qo)
    assert np.array_equal(_np(s).view(np.uint8), so.view(np.uint8))


@pytest.mark.slow
@pytest.mark.parametrize("fmt", FMTS)
def test_quotient_domain_exhaustive(fmt):
    """Every bf16 x against every amax mantissa (at exponents spread over the
    range, subnormals included): group [amax, x_0 .. x_126] through the GPU
    quantiser equals the oracle.  This is the whole input domain of the
    division-and-round step up to a shared power of two."""
    all_bits = np.arange(0, 0x7F80, dtype=np.uint32)  # non-negative finite bf16
    mags = (all_bits << 16).view(np.float32)
    # exponents across the range, dense near both ends and around amax ~ 2^-71,
    # where the fp32 path switches between IEEE division and the reciprocal form
    exps = [-126, -125, -124, -120, -110, -100, -91, -90, -89, -80, -75, -73, -72, -71, -70,
            -69, -68, -60, -40, -20, -7, -1, 0, 1, 3, 9, 20, 60, 100, 118, 119, 120, 125, 126, 127]
    amaxes = []
    for e in exps:
        for mant in range(128):
            amaxes.append((e + 127) << 7 | mant)
    amaxes += list(range(1, 128))  # subnormal bf16 amax values
    amax_bits = np.array(sorted(set(b for b in amaxes if 0 < b < 0x7F80)), dtype=np.uint16)
    rows = []
    for ab in amax_bits:
        a = np.float32((np.uint32(ab) << 16).view(np.float32))
        xs = all_bits[mags <= a].astype(np.uint16)
        xs = np.concatenate([xs, xs | np.uint16(0x8000)])  # both signs
        pad = (-len(xs)) % 127
        xs = np.concatenate([xs, np.zeros(pad, np.uint16)]).reshape(-1, 127)
        blk = np.empty((xs.shape[0], 128), np.uint16)
        blk[:, 0] = ab
        blk[:, 1:] = xs
        rows.append(blk)
    x = np.concatenate(rows)
    # chunk to bound device memory
    for start in range(0, x.shape[0], 1 << 19):
        xc = x[start:start + (1 << 19)]
        xt = torch.from_numpy(xc.view(np.int16)).view(torch.bfloat16)
        q, s = fp8rl.quant_act(xt.cuda(), fmt)
        torch.cuda.synchronize()
        qo, so = oracle.quant_act_group(xc, fmt)
        bad = np.count_nonzero(_np(q) != qo)
        assert bad == 0, f"{bad} codes differ in chunk at row {start}"
        assert np.array_equal(_np(s).view(np.uint8), so.view(np.uint8))


@pytest.mark.slow
def test_device_codec_all_fp32_patterns():
    """The device fp32 -> E4M3 convert against the oracle on every finite fp32
    bit pattern (2^32 minus NaN/inf), in chunks."""
    chunk = 1 << 28
    dev_in = torch.empty(chunk, dtype=torch.float32, device="cuda")
    dev_out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    mism = 0
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
        wrapped = (bits - (1 << 32) * (bits >= (1 << 31))).to(torch.int32)  # uint32 -> int32 bits
        dev_in.copy_(wrapped.view(torch.float32))
        fp8rl.fp8rl_e4m3_encode(dev_in, chunk, dev_out)
        torch.cuda.synchronize()
        v = dev_in.cpu().numpy()
        got = dev_out.cpu().numpy()
        fin = np.isfinite(v)
        ref = oracle.e4m3_encode_array(np.where(fin, v, np.float32(0)))
        mism += int(np.count_nonzero((got != ref) & fin))
        del bits, wrapped
    assert mism == 0


def test_status_is_ok_after_quantisers():
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    fp8rl.quant_act(x)
    assert fp8rl.fp8rl_sync_status() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_host_weight_sync_pipeline_bit_exact(fmt):
    """Host-to-host weight sync through HostWeightSync (the C entry point
    fp8rl_quant_weight_host_batched) in small chunks: many more chunks than
    staging slots, ragged shapes; equals the oracle on every matrix, twice."""
    shapes = [(384, 256), (200, 300), (1024, 128), (130, 640)]
    ws = [synth.weight_bf16(n, k, 6, "hostsync", n, k) for n, k in shapes]
    host_w = [w.pin_memory() for w in ws]
    sdt = torch.float32 if fmt == fp8rl.SCALE_FP32 else torch.uint8
    host_q = [torch.empty((n, k), dtype=torch.uint8, pin_memory=True) for n, k in shapes]
    host_s = [torch.empty(((n + 127) // 128, (k + 127) // 128), dtype=sdt, pin_memory=True) for n, k in shapes]
    hs = fp8rl.HostWeightSync(host_w, host_q, host_s, fmt=fmt, chunk_bytes=64 * 1024, slots=2)
    for _ in range(2):
        hs.run()
    torch.cuda.synchronize()
    for w, q, s in zip(ws, host_q, host_s):
        qo, so = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
        assert np.array_equal(q.numpy(), qo)
        assert np.array_equal(s.numpy().view(np.uint8), so.view(np.uint8))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("slots", [2, 3, 8])
def test_host_sync_c_abi_strided_rows(fmt, pinned, slots):
    """fp8rl_quant_weight_host_batched on host rows with padded strides (ldw,
    ldq > k), one chunk per 128-row block row (the staging holds exactly one
    block row per slot), pinned and pageable host memory; the bytes outside
    each row's k columns are left as they were."""
    shapes = [(300, 256), (128, 384), (257, 128), (5, 200)]
    sdt = torch.float32 if fmt == fp8rl.SCALE_FP32 else torch.uint8
    ws, host_w, host_q, host_s = [], [], [], []
    for i, (n, k) in enumerate(shapes):
        w = synth.weight_bf16(n, k, 70 + i, "hostabi", n, k)
        big = torch.zeros((n, k + 24), dtype=torch.bfloat16)
        big[:, :k] = w
        q = torch.full((n, k + 40), 0xA5, dtype=torch.uint8)
        s = torch.empty(((n + 127) // 128, (k + 127) // 128), dtype=sdt)
        if pinned:
            big, q, s = big.pin_memory(), q.pin_memory(), s.pin_memory()
        ws.append(w)
        host_w.append(big)
        host_q.append(q)
        host_s.append(s)
    descs = (fp8rl.WeightDesc * len(shapes))()
    for i, (n, k) in enumerate(shapes):
        descs[i] = fp8rl.WeightDesc(host_w[i].data_ptr(), host_q[i].data_ptr(), host_s[i].data_ptr(), n, k,
                                    k + 24, k + 40)
    need = max(fp8rl.fp8rl_host_sync_staging_bytes(min(n, 128), k, slots, fmt) for n, k in shapes)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    fp8rl.fp8rl_quant_weight_host_batched(descs, len(shapes), fmt, staging, need, slots)
    assert fp8rl.fp8rl_sync_status() == 0
    for (n, k), w, q, s in zip(shapes, ws, host_q, host_s):
        qo, so = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
        assert np.array_equal(q[:, :k].numpy(), qo)
        assert np.all(q[:, k:].numpy() == 0xA5)
        assert np.array_equal(s.numpy().view(np.uint8).reshape(-1), so.view(np.uint8).reshape(-1))


def test_host_weight_sync_direct_bit_exact():
    """The quantiser reading pinned host weights and writing pinned host codes."""
    shapes = [(384, 256), (200, 300)]
    ws = [synth.weight_bf16(n, k, 7, "hostdirect", n, k) for n, k in shapes]
    host_w = [w.pin_memory() for w in ws]
    host_q = [torch.empty((n, k), dtype=torch.uint8, pin_memory=True) for n, k in shapes]
    host_s = [torch.empty(((n + 127) // 128, (k + 127) // 128), dtype=torch.float32, pin_memory=True)
              for n, k in shapes]
    hs = fp8rl.HostWeightSync(host_w, host_q, host_s, direct=True)
    hs.run()
    torch.cuda.synchronize()
    for w, q, s in zip(ws, host_q, host_s):
        qo, so = oracle.quant_weight_blockwise(synth.bf16_bits(w))
        assert np.array_equal(q.numpy(), qo) and np.array_equal(s.numpy(), so)


def _full_parity(ws, outs, fmt):
    """Every code and every scale of the device results against the oracle,
    matrix by matrix: each bf16 matrix and its device codes and scales come to
    the host in turn (host memory stays at one matrix), and the oracle's
    quantisation of the next matrix runs while the current one is copied."""
    from concurrent.futures import ThreadPoolExecutor

    def host(i):
        q, s = outs[i]
        return synth.bf16_bits(ws[i].cpu()), q.cpu().numpy(), s.cpu().numpy()

    with ThreadPoolExecutor(max_workers=1) as pool:
        bits, q, s = host(0)
        for i in range(len(ws)):
            fut = pool.submit(oracle.quant_weight_blockwise, bits, fmt)
            nxt = host(i + 1) if i + 1 < len(ws) else None
            qo, so = fut.result()
            assert np.array_equal(q, qo), f"E4M3 codes of matrix {i} differ"
            assert np.array_equal(s.view(np.uint8), so.view(np.uint8)), f"scales of matrix {i} differ"
            if nxt is not None:
                bits, q, s = nxt


@pytest.mark.slow
def test_full_model_weight_sync_bit_exact():
    """36 Qwen3-8B-shaped layers (252 matrices, 6.95e9 parameters) in the
    single batched launch the benchmark times; every code and scale."""
    dev = torch.device("cuda")
    ws = []
    for layer in range(synth.QWEN3_8B_LAYERS):
        ws += [w for _, w in synth.qwen3_8b_layer(layer, 1000, device=dev)]
    outs = fp8rl.quant_weights_batched(ws)
    torch.cuda.synchronize()
    assert fp8rl.fp8rl_sync_status() == 0
    _full_parity(ws, outs, fp8rl.SCALE_FP32)
    del ws, outs
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("fmt", FMTS)
def test_moe_expert_weight_sync_bit_exact(fmt):
    """48 layers x 128 experts x (gate-up, down) of a Qwen3-30B-A3B-shaped model
    (2.9e10 parameters, 58 GB of bf16) in one batched launch; every code and
    scale."""
    dev = torch.device("cuda")
    ws = []
    for layer in range(synth.MOE_LAYERS):
        for which, n, k in (("gate_up", 2 * synth.MOE_INTER, synth.MOE_HIDDEN),
                            ("down", synth.MOE_HIDDEN, synth.MOE_INTER)):
            ws.append(synth.normal_bf16((synth.MOE_EXPERTS * n, k), synth.WEIGHT_STD, 1000, "moe-sync",
                                        layer, which, device=dev))
    outs = fp8rl.quant_weights_batched(ws, fmt)
    torch.cuda.synchronize()
    assert fp8rl.fp8rl_sync_status() == 0
    _full_parity(ws, outs, fmt)
    del ws, outs
    torch.cuda.empty_cache()
