"""The canary guards of the binding (FP8RL_CANARY=1): outputs the helpers
allocate sit between guard zones that fp8rl_sync_status() checks.  CPU only:
the mechanism itself, with host tensors standing in for device outputs."""
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl


@pytest.fixture
def canary(monkeypatch):
    monkeypatch.setenv("FP8RL_CANARY", "1")
    fp8rl.check_canaries()  # start from an empty list
    yield
    fp8rl.check_canaries()


def test_off_by_default(monkeypatch):
    monkeypatch.delenv("FP8RL_CANARY", raising=False)
    t = fp8rl._out((4, 8), torch.float32, "cpu")
    assert t.shape == (4, 8) and fp8rl.check_canaries() == 0


def test_writes_inside_the_output_pass(canary):
    t = fp8rl._out((3, 5), torch.float32, "cpu")
    q = fp8rl._out((7, 128), torch.uint8, "cpu")
    # the output starts a whole number of 256-byte units into its buffer, so
    # it keeps the allocation's alignment
    for x in (t, q):
        assert (x.data_ptr() - x.untyped_storage().data_ptr()) % 256 == 0
    t.fill_(1.0)
    q.fill_(0)
    assert fp8rl.check_canaries() == 2


@pytest.mark.parametrize("where", ["before", "after", "far_after"])
def test_writes_outside_the_output_are_caught(canary, where):
    t = fp8rl._out((3, 5), torch.bfloat16, "cpu")
    raw = torch.empty(0, dtype=torch.uint8).set_(t.untyped_storage())  # the whole guarded buffer
    start = t.storage_offset() * t.element_size()
    end = start + t.numel() * t.element_size()
    raw[{"before": start - 1, "after": end, "far_after": end + 60000}[where]] = 0
    with pytest.raises(fp8rl.CanaryError):
        fp8rl.check_canaries()


def test_empty_outputs_are_not_guarded(canary):
    t = fp8rl._out((0, 128), torch.uint8, "cpu")
    assert t.numel() == 0 and fp8rl.check_canaries() == 0
