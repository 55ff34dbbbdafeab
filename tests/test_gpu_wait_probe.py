"""The expiry path of the kernels' bounded waits, on the GPU, with nothing
stalled: rope_probe_wait_expiry waits on a barrier that nothing arrives at,
for about a millisecond, and the expiry must reach rope_check_errors as
ROPE_ERR_KERNEL_TIMEOUT, once (the check clears the flag)."""
import pytest
import torch

from gpu_util import lib, require_gpu

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_once():
    require_gpu()
    R = lib()
    R.rope_check_errors()                                 # clear anything pending
    assert R.rope_probe_wait_expiry(2_000_000) == R.ROPE_OK
    assert R.rope_check_errors() == R.ROPE_ERR_KERNEL_TIMEOUT
    assert R.rope_check_errors() == R.ROPE_OK            # the check cleared the flag


def test_expired_wait_on_a_side_stream_leaves_later_work_correct():
    require_gpu()
    R = lib()
    R.rope_check_errors()
    s = torch.cuda.Stream()
    assert R.rope_probe_wait_expiry(1_000_000, s) == R.ROPE_OK
    assert R.rope_check_errors(s) == R.ROPE_ERR_KERNEL_TIMEOUT
    # the context is still usable: a rotation afterwards is exact at position 0
    cos, sin = R.build_tables(1e4, 64, 8)
    q = torch.randn(1, 2, 1, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(1, 1, 1, 64, device="cuda", dtype=torch.bfloat16)
    q0, k0 = q.clone(), k.clone()
    R.apply_qk(q, k, cos, sin)
    assert R.rope_check_errors() == R.ROPE_OK
    assert torch.equal(q, q0) and torch.equal(k, k0)
