"""Dense trellis linear layer on the GPU (through the C ABI) against the
float64 oracle."""
import numpy as np
import pytest

from oracle import linear as olinear
from trellis_quantized_moe_route_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# fp16 operands, fp32 accumulation against a float64 oracle that rounds x~ to
# fp16 the same way: what is left is the accumulation order (and x~ rounding
# ties), far below this bound; a wrong row, block or sign is O(1)
TOL = 2e-3


def rel_row_err(out, ref):
    rms = np.sqrt(np.mean(ref * ref, axis=1)) + 1e-30
    return float(np.max(np.abs(out - ref).max(axis=1) / rms))


def _run(lin, x, max_tokens=None):
    from trellis_quantized_moe_route_gb300.binding import TrellisLinear
    m = TrellisLinear(lin, max_tokens=max_tokens or x.shape[0])
    out = m.forward(torch.from_numpy(np.ascontiguousarray(x.view(np.int16))).cuda())
    torch.cuda.synchronize()
    return m, out.cpu().numpy()


@pytest.mark.parametrize("N,K,bits,rot_in,rot_out,T", [
    (256, 512, 4, 128, 128, 5),      # one route block, K=4 expansion, 256-column units
    (384, 256, 3, 64, 128, 300),     # 128-column units, two blocks with a ragged tail, generic K
    (512, 384, 2, 1, 64, 257),       # identity input rotation, 64-wide output blocks, 257 = 256 + 1
    (1024, 1024, 6, 128, 1, 1),      # one token, identity output rotation
    (768, 1280, 5, 128, 128, 513),   # three blocks
])
def test_linear_matches_oracle(N, K, bits, rot_in, rot_out, T):
    lin = synth.make_linear(N, K, bits=bits, rot_in=rot_in, rot_out=rot_out, seed=N + K + T)
    x = synth.make_linear_tokens(lin, T, seed=T)
    m, out = _run(lin, x)
    ref = olinear.linear_forward(lin, x)
    assert rel_row_err(out, ref) < TOL
    assert m.poll_error() == 0


def test_linear_deterministic_poisoned_workspace_and_fewer_tokens():
    lin = synth.make_linear(256, 256, bits=4, seed=3)
    x = synth.make_linear_tokens(lin, 200, seed=4)
    m, a = _run(lin, x, max_tokens=600)
    m.workspace.fill_(0xFF)
    b = m.forward(torch.from_numpy(np.ascontiguousarray(x.view(np.int16))).cuda()).cpu().numpy()
    assert np.array_equal(a, b)
    # a call with fewer tokens than max_tokens gives the same rows
    c = m.forward(torch.from_numpy(np.ascontiguousarray(x[:37].view(np.int16))).cuda()).cpu().numpy()
    assert np.array_equal(c, a[:37])


def test_linear_large_sampled_rows():
    """N = K = 4096 at T = 2048 (the bench workload), 16 sampled tokens
    including the first and the last."""
    lin = synth.make_linear(4096, 4096, bits=4, seed=7)
    T = 2048
    x = synth.make_linear_tokens(lin, T, seed=7)
    m, out = _run(lin, x)
    rows = np.unique(np.concatenate([[0, T - 1], synth.Stream(7, 77).below(14, T)]))
    ref = olinear.linear_forward(lin, x[rows])
    assert rel_row_err(out[rows], ref) < TOL
