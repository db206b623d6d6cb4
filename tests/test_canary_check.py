"""The guard-canary checker of the GPU tests, exercised on the CPU: it
passes when only the output was written and fails when a byte past either
end of the output changed (the mistake is planted here, on the host)."""
import pytest
import torch

from tests import helpers


def test_canary_check_passes_on_in_bounds_writes(monkeypatch):
    monkeypatch.setattr(torch.cuda, "synchronize", lambda: None)
    t = helpers.guarded_empty((3, 5), torch.float32, device="cpu")
    t.fill_(1.0)
    helpers.check_canaries()


@pytest.mark.parametrize("where", ["before", "after"])
def test_canary_check_catches_a_write_past_the_output(monkeypatch, where):
    monkeypatch.setattr(torch.cuda, "synchronize", lambda: None)
    t = helpers.guarded_empty((4, 8), torch.bfloat16, device="cpu")
    t.zero_()
    buf, nbytes = helpers._guarded[-1]
    if where == "before":
        buf[helpers.CANARY_BYTES - 1] = 0
    else:
        buf[helpers.CANARY_BYTES + nbytes] = 0
    with pytest.raises(AssertionError):
        helpers.check_canaries()
    helpers._guarded.clear()
