"""The tensor-core kernels' bounded waits give up, report and leave the
context usable (needs a GPU).

Failure detection of a stalled pipeline: every mbarrier wait of the
tensor-core FC kernels is bounded in wall time; on expiry the CTA sets bit 1
of the device error word, lets its copies in flight land, frees its tensor
memory and returns. The test makes one wait run out without any fault: the
MMA issuer waits on a barrier that nothing arrives on (a flag that nothing
sets), with a 1 ms limit. The error word must report it, and the next call
with the stall off must reproduce a reference call bit for bit.
"""
import numpy as np
import pytest

from tests.gpu_util import small_cfg, upload_tokens
from trellis_quantized_moe_route_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_stalled_issuer_times_out_reports_and_recovers():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    from trellis_quantized_moe_route_gb300 import binding, build
    build.build()
    binding.load_library()
    cfg = small_cfg(T=64, E=8, topk=2)          # 128 routes >= 4E: tensor-core kernels
    L = synth.make_layer(cfg)
    moe = binding.TrellisMoE(L, max_tokens=cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    ref = moe.forward_logits(x, lg, mode="w4a16").clone()
    torch.cuda.synchronize()
    assert moe.poll_error() == 0

    moe.set_wait_test(wait_limit_ns=1_000_000, stall_issuer=True)
    moe.forward_logits(x, lg, mode="w4a16")
    torch.cuda.synchronize()                    # the kernels returned: the context is alive
    assert moe.poll_error() & 2

    moe.set_wait_test(0, False)
    out = moe.forward_logits(x, lg, mode="w4a16")
    torch.cuda.synchronize()
    assert moe.poll_error() == 0
    assert torch.equal(out, ref)
    # the short limit alone (no stall) still completes a normal call
    moe.set_wait_test(wait_limit_ns=200_000_000, stall_issuer=False)
    out2 = moe.forward_logits(x, lg, mode="w4a16")
    torch.cuda.synchronize()
    assert moe.poll_error() == 0 and torch.equal(out2, ref)
    moe.close()
