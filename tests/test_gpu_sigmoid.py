"""GPU pin of the kernels' sigmoid (1 / (1 + e^-z) from the hardware exponential and reciprocal)
through the gated RMSNorm entry point: with o = 1 on every channel and w = 1 the output is
y = sigmoid(z) / sqrt(1 + eps), so y * sqrt(1 + eps) is compared with the f64 sigmoid over
z in [-100, 100].  Bound: the hardware exponential's documented error grows with |z| (2 + 1.2 |z|
ulp); the reciprocal, the rsqrt and two roundings add a few ulp more.  Far in the tail (sigmoid
below 1e-30) the check is absolute."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    from gated_delta_rule_scan_gb300 import kda
    assert kda.kda_device_status() == 0


def test_gate_sigmoid_against_f64():
    from gated_delta_rule_scan_gb300 import kda
    D = kda.HEAD_DIM
    z = np.concatenate([np.linspace(-100.0, 100.0, 64 * D - 8),
                        [0.0, -0.0, 1e-8, -1e-8, 88.0, -88.0, -69.0, -70.0]]).astype(np.float32)
    rows = z.size // D
    eps = 1e-6
    o = torch.ones(rows, D, device="cuda")
    w = torch.ones(D, device="cuda")
    zt = torch.from_numpy(z.reshape(rows, D)).cuda()
    y = torch.empty(rows, D, device="cuda")
    kda.kda_gated_rmsnorm_out(o, w, zt, y, rows=rows, eps=eps)
    torch.cuda.synchronize()
    got = y.cpu().double().numpy().reshape(-1) * np.sqrt(np.float64(np.float32(1.0 + eps)))
    zd = z.astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-zd))
    big = ref > 1e-30
    ulp = 2.0 ** -24
    bound = (2.0 + 1.2 * np.abs(zd) + 8.0) * ulp
    rel = np.abs(got[big] - ref[big]) / ref[big]
    assert np.all(rel <= bound[big]), (zd[big][np.argmax(rel / bound[big])], rel.max())
    assert np.all(np.abs(got[~big] - ref[~big]) <= 1e-30)
    assert big.sum() > 0.6 * z.size and (~big).sum() > 0.1 * z.size
