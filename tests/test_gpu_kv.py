"""GPU parity of the FP8 KV cache kernels (per-step per-tensor calibration and
the quantised append) against the oracle, through the C ABI.  Scales and
cache bytes are integer/byte results of the same fp32 arithmetic on both
sides, so the bar is bit-exactness."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)


def kv_inputs(tokens, dim, seed, spread=1.0, ld=None):
    """K and V [tokens, dim] bf16 (optionally inside rows of ld elements)."""
    ld = ld or dim
    k = synth.normal_bf16((tokens, ld), 1.0, seed, "kv-k")[:, :dim]
    v = synth.normal_bf16((tokens, ld), spread, seed, "kv-v")[:, :dim]
    return k, v


@pytest.mark.parametrize("tokens,dim,qdim,ld", [(1, 1024, 4096, None), (300, 1024, 4096, None),
                                                (8192, 1024, 4096, None), (77, 1000, 1000, None), (5, 8, 0, None),
                                                (300, 1024, 4096, 1088), (64, 1000, 1000, 1003)])
def test_calibrate_scales_bit_exact(tokens, dim, qdim, ld):
    """Contiguous and strided rows (ld - dim padding elements after each row,
    holding 1e30, which must not reach the amax: a padding of 64 keeps 16-byte
    aligned rows, one of 3 takes the scalar loads)."""
    k, v = kv_inputs(tokens, dim, 1, 3.0)
    q = synth.normal_bf16((tokens, qdim), 0.5, 2, "kv-q") if qdim else None
    ref = oracle.kv_calibrate(synth.bf16_bits(k), synth.bf16_bits(v), synth.bf16_bits(q) if qdim else None)
    pad = 0 if ld is None else ld - dim

    def dev(t):  # each row followed by `pad` elements of a huge value
        if not pad:
            return t.cuda()
        full = torch.full((t.shape[0], t.shape[1] + pad), 1e30, dtype=torch.bfloat16)
        full[:, :t.shape[1]] = t
        return full.cuda()[:, :t.shape[1]]
    kd, vd = dev(k), dev(v)
    qd = dev(q) if qdim else None
    assert kd.stride(0) == dim + pad and (qd is None or qd.stride(0) == qdim + pad)
    got = fp8rl.kv_calibrate(kd, vd, qd)
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(got.cpu().numpy(), ref)


def test_calibrate_zero_tensor_gets_unit_scale():
    k = torch.zeros((64, 256), dtype=torch.bfloat16)
    v = synth.normal_bf16((64, 256), 1.0, 3, "kv-v0")
    got = fp8rl.kv_calibrate(k.cuda(), v.cuda()).cpu().numpy()
    assert got[0] == 1.0 and got[1] == oracle.kv_calibrate(synth.bf16_bits(k), synth.bf16_bits(v))[1]


@pytest.mark.parametrize("tokens,dim,ld,slots_total", [
    (40, 1024, 1024, 64),      # vector path
    (300, 1004, 1008, 512),    # vector path with a scalar tail (dim % 8 == 4)
    (33, 1004, 1004, 40),      # rows not 16-byte aligned: the scalar path
    (1, 128, 128, 1),
])
def test_append_bit_exact_with_padding_and_saturation(tokens, dim, ld, slots_total):
    k, v = kv_inputs(tokens, dim, 4, 2.0, ld)
    calib = max(1, tokens // 3)  # scales from a prefix: later tokens may saturate
    s_ref = oracle.kv_calibrate(synth.bf16_bits(k[:calib]), synth.bf16_bits(v[:calib]))
    rng = np.random.default_rng(tokens + dim)
    slots = rng.permutation(max(slots_total, tokens))[:tokens].astype(np.int32)
    slots[::7] = -1
    if tokens > 3:
        slots[2] = slots_total + 5  # beyond the cache: skipped
    kc = np.full((slots_total, dim), 0x55, np.uint8)
    vc = np.full((slots_total, dim), 0x55, np.uint8)
    oracle.kv_append(synth.bf16_bits(k), synth.bf16_bits(v), slots, kc, vc, s_ref)
    dk = torch.empty((tokens, ld), dtype=torch.bfloat16, device="cuda")
    dv = torch.empty((tokens, ld), dtype=torch.bfloat16, device="cuda")
    dk[:, :dim] = k.cuda()
    dv[:, :dim] = v.cuda()
    scales = fp8rl.kv_calibrate(dk[:calib, :dim], dv[:calib, :dim])
    assert np.array_equal(scales.cpu().numpy()[:2], s_ref[:2])
    gk = torch.full((slots_total, dim), 0x55, dtype=torch.uint8, device="cuda")
    gv = torch.full((slots_total, dim), 0x55, dtype=torch.uint8, device="cuda")
    fp8rl.kv_append(dk[:, :dim], dv[:, :dim], torch.from_numpy(slots).cuda(), gk, gv, scales)
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)


def test_append_full_size_prefill_bit_exact():
    """32768 tokens x 8 KV heads x 128 (Qwen3-8B), shuffled slots of a
    65536-slot cache, scales calibrated on the first 8192 tokens."""
    tokens, dim, slots_total = 32768, 1024, 65536
    k, v = kv_inputs(tokens, dim, 5, 1.5)
    dk, dv = k.cuda(), v.cuda()
    slots = np.random.default_rng(6).permutation(slots_total)[:tokens].astype(np.int32)
    scales = fp8rl.kv_calibrate(dk[:8192], dv[:8192])
    gk = torch.zeros((slots_total, dim), dtype=torch.uint8, device="cuda")
    gv = torch.zeros((slots_total, dim), dtype=torch.uint8, device="cuda")
    fp8rl.kv_append(dk, dv, torch.from_numpy(slots).cuda(), gk, gv, scales)
    assert fp8rl.fp8rl_sync_status() == 0
    s_ref = oracle.kv_calibrate(synth.bf16_bits(k[:8192]), synth.bf16_bits(v[:8192]))
    assert np.array_equal(scales.cpu().numpy()[:2], s_ref[:2])
    kc = np.zeros((slots_total, dim), np.uint8)
    vc = np.zeros((slots_total, dim), np.uint8)
    oracle.kv_append(synth.bf16_bits(k), synth.bf16_bits(v), slots, kc, vc, s_ref)
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)


def test_append_rejects_bad_arguments():
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones(3, dtype=torch.float32, device="cuda")
    sl = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.fp8rl_kv_append(x, x, 4, 128, 64, 128, sl, c, c, 128, 4, s)  # ldk < dim
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.fp8rl_kv_append(x, x, 4, 128, 128, 128, None, c, c, 128, 4, s)
    fp8rl.fp8rl_kv_append(x, x, 0, 128, 128, 128, None, None, None, 128, 0, None)  # empty: no-op


@pytest.fixture
def overlap():
    yield lambda off: fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PDL, 1 if off else 0)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PDL, 0)


@pytest.mark.parametrize("tokens", [8192, 0, 3])
def test_calibrate_chain_from_poisoned_scales(tokens, overlap):
    """The calibration's three kernels (zero, reduce, convert; each later one
    started while the one before it runs): d_scales starts out holding values
    larger than any amax, K is written by a kernel enqueued right before the
    call, and the result is the oracle's with the overlap on and off and when
    replayed from a CUDA graph.  At 0 tokens (no Q: torch gives an empty
    tensor a null pointer) only the K and V words are written."""
    dim = 1024
    qdim = 4096 if tokens else 0
    k, v = kv_inputs(max(tokens, 1), dim, 5, 2.0)
    q = synth.normal_bf16((max(tokens, 1), 4096), 0.5, 6, "kv-q-chain")
    ref = oracle.kv_calibrate(synth.bf16_bits(k[:tokens]), synth.bf16_bits(v[:tokens]),
                              synth.bf16_bits(q[:tokens]) if qdim else None)
    written = 3 if qdim else 2
    poison = np.float32(3.0e38)
    kd0, vd = k.cuda()[:tokens], v.cuda()[:tokens]
    qd = q.cuda()[:tokens] if qdim else None
    kd = torch.empty((max(tokens, 1), dim), dtype=torch.bfloat16, device="cuda")[:tokens]
    scales = torch.empty(3, dtype=torch.float32, device="cuda")

    def run():
        kd.copy_(kd0)  # the producer of K, right before the call
        fp8rl.fp8rl_kv_calibrate(kd, vd, qd, tokens, dim, dim, dim, qdim, qdim, scales)

    results = []
    for off in (False, True):
        overlap(off)
        kd.fill_(float("inf"))
        scales.fill_(float(poison))
        run()
        assert fp8rl.fp8rl_sync_status() == 0
        results.append(scales.cpu().numpy().copy())
    overlap(False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(2):
        kd.fill_(float("inf"))
        scales.fill_(float(poison))
        g.replay()
        torch.cuda.synchronize()
        results.append(scales.cpu().numpy().copy())
    expect = np.asarray(ref, np.float32).copy()
    expect[written:] = poison
    for got in results:
        assert np.array_equal(got.view(np.uint32), expect.view(np.uint32))
