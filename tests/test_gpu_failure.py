"""Failure detection on the GPU without a fault: a kernel's bounded wait on
an mbarrier that nothing completes gives up after about a second, records
its code in the device error word and returns; the host reads the code, and
the context stays usable (a product afterwards still matches the oracle)."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import ggml_block_quantized_gb300 as qg  # noqa: E402
import oracle  # noqa: E402
from ggml_block_quantized_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_bounded_wait_runs_out_and_reports():
    assert qg.device_error() == 0
    t0 = time.perf_counter()
    qg.selftest_bounded_wait()
    code = qg.device_error()  # synchronizes
    elapsed = time.perf_counter() - t0
    assert code == 2  # the consumer-wait code
    assert 0.5 < elapsed < 30.0
    assert qg.device_error() == 0  # reading clears it
    # the context is still usable
    rng = np.random.default_rng(7700)
    n_out, n_in = 64, 512
    W = synth.k_blocks(qg.Q4_K, n_out * n_in // 256, rng)
    x = synth.f32_normal(rng, n_in)
    y = qg.qgemv(qg.Q4_K, torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda(), n_out, n_in, 1)
    torch.cuda.synchronize()
    ref = oracle.gemv(qg.Q4_K, W, oracle.quantize(oracle.Q8_K, x), n_out, n_in, 1)[0]
    assert np.allclose(y.cpu().numpy()[0], ref, rtol=1e-4, atol=1e-4 * np.abs(ref).max())
