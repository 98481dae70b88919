"""GPU parity of the token-level TIS weights and the mismatch KL against the
fp64 oracle, through the C ABI.

Bounds, from the arithmetic: the kernel forms d = lp_train - lp_rollout in
fp32 (absolute error <= 2^-24 |d|) and calls expf (within 2 ulp), so
|w_gpu - w_ref| <= (2^-21 + 2^-23 |d|) w_ref with a factor 2 of margin, plus
2^-146 for results in the fp32 subnormal range (a few of its ulps); a
masked-out token's weight is exactly 0.  The KL sum makes each difference
exact in fp32 (TwoSum) and adds the differences, then the threads' and CTAs'
sums, as fp32 (hi, lo) pairs: a pair addition rounds only the lo word, by at
most 2^-48 of the sum it belongs to, so over the 16 tokens of a thread and the
~20 tree levels above them |sum_gpu - sum_ref| stays below 2^-40 sum |d|; the
test allows 2^-36 sum |d|; the count is exact."""
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


def check(lt, lr, mask, clip=2.0, offset=0):
    """lt, lr fp32 and mask uint8 host arrays; offset > 0 places the device
    arrays off 16-byte alignment (the scalar path)."""
    n = lt.size
    def dev(a):
        buf = torch.zeros(n + offset, dtype=torch.from_numpy(a[:0]).dtype, device="cuda")
        buf[offset:] = torch.from_numpy(a).cuda()
        return buf[offset:]
    dlt, dlr = dev(lt), dev(lr)
    dm = dev(mask) if mask is not None else None
    w, kl = fp8rl.tis_weights(dlt, dlr, dm, clip)
    assert fp8rl.fp8rl_sync_status() == 0
    w = w.cpu().numpy()
    kl = kl.cpu().numpy()
    w_ref = oracle.tis_weights(lt, lr, mask, clip)
    d = lt.astype(np.float64) - lr.astype(np.float64)
    on = np.ones(n, bool) if mask is None else mask != 0
    assert np.all(w[~on] == 0.0)
    assert np.all(np.abs(w[on] - w_ref[on]) <= (2.0 ** -21 + 2.0 ** -23 * np.abs(d[on])) * w_ref[on] + 2.0 ** -146)
    assert np.all(w <= np.float32(clip))
    mean, total, count = oracle.mismatch_kl(lt, lr, mask)
    assert kl[2] == count
    assert abs(kl[1] - total) <= 2.0 ** -36 * float(np.abs(d[on]).sum())
    assert (kl[0] == 0.0) if count == 0 else abs(kl[0] - mean) <= 2.0 ** -35 * float(np.abs(d[on]).sum()) / count
    return w, kl


@pytest.mark.parametrize("n", [1, 3, 4, 1000, 4097, 8192 * 5 + 7])
@pytest.mark.parametrize("masked", [False, True])
def test_tis_small_sizes(n, masked):
    lt, lr, m = synth.rollout_logprobs(1, n, seed=n)
    check(lt.numpy(), lr.numpy(), m.numpy() if masked else None)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_tis_unaligned_scalar_path(offset):
    lt, lr, m = synth.rollout_logprobs(3, 3000, seed=offset)
    check(lt.numpy(), lr.numpy(), m.numpy(), offset=offset)


def test_tis_clip_edges_and_empty_mask():
    lr = np.zeros(8, np.float32)
    lt = np.array([0.0, np.log(2.0), np.log(2.0) + 1e-6, 5.0, -5.0, 100.0, -100.0, 0.5], np.float32)
    w, _ = check(lt, lr, None)
    assert w[0] == 1.0 and w[3] == 2.0 and w[5] == 2.0
    check(lt, lr, np.zeros(8, np.uint8))           # no generated token: mean 0, count 0
    check(lt, lr, None, clip=1.0)                  # another truncation level
    n0 = fp8rl.tis_weights(torch.zeros(0, device="cuda"), torch.zeros(0, device="cuda"))
    assert n0[1].cpu().tolist() == [0.0, 0.0, 0.0]


def test_tis_full_rollout_batch_and_determinism():
    """512 responses x 16384 tokens (8.4 M tokens), generated on the device;
    all weights and the KL checked against the oracle, and a second run gives
    the same bits."""
    lt, lr, m = synth.rollout_logprobs(device="cuda")
    w1, kl1 = fp8rl.tis_weights(lt, lr, m)
    w2, kl2 = fp8rl.tis_weights(lt, lr, m)
    assert fp8rl.fp8rl_sync_status() == 0
    assert torch.equal(w1, w2) and torch.equal(kl1, kl2)
    check(lt.cpu().numpy(), lr.cpu().numpy(), m.cpu().numpy())


def test_tis_reuses_one_workspace_across_sizes():
    """The workspace's header (the CTA ticket) is zeroed once and every call
    leaves it zero: calls of different sizes (different grids) on one
    workspace all match the oracle."""
    ws = torch.zeros(fp8rl.fp8rl_tis_workspace_size(1 << 20), dtype=torch.uint8, device="cuda")
    for n in (1 << 20, 5000, 1, 4096 * 3 + 1, 1 << 20):
        lt, lr, m = synth.rollout_logprobs(1, n, seed=n % 97)
        w, kl = fp8rl.tis_weights(lt.cuda(), lr.cuda(), m.cuda(), workspace=ws)
        assert fp8rl.fp8rl_sync_status() == 0
        mean, total, count = oracle.mismatch_kl(lt.numpy(), lr.numpy(), m.numpy())
        d = np.abs(lt.numpy().astype(np.float64) - lr.numpy())
        assert kl.cpu().numpy()[2] == count
        assert abs(kl.cpu().numpy()[1] - total) <= 2.0 ** -36 * float(d[m.numpy() != 0].sum())
    assert int(ws[:16].sum().item()) == 0
