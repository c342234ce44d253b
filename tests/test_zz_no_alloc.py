"""qgemv_noalloc, the product for callers that cannot allocate device memory
where they run it (a plugin whose host framework hands it no buffer, a
decode loop that must not call cudaMalloc/cudaFree because they can
synchronize the device, code under CUDA stream capture). It keeps the
quantized activations in the library's own fixed device array instead of a
caller workspace.

Checked through the C ABI against qgemv, the entry point with a caller
workspace: bit for bit, and within the tolerance the parity tests use
(1e-5 |y| + 1e-6 ||x_v|| ||w_o||), on calls in a row that share the array,
where a call with shorter activations follows one with longer ones (so stale
bytes of the earlier call sit past the later call's end). Sampled rows are
also checked against the oracle with that tolerance.
This file is collected last on purpose; it passes alone or after the rest.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import ggml_block_quantized_gb300 as qg  # noqa: E402
from ggml_block_quantized_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6
SCRATCH_BYTES = 256 * 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def call_noalloc(t, W, x, y, n_out, n_in, n_vec):
    """Direct C-ABI call: device pointers and the current stream."""
    st = qg.lib().qgemv_noalloc(t, ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), n_out, n_in, n_vec,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def close(t, W, x, got, want, n_out, n_in, n_vec):
    wn = torch.linalg.vector_norm(qg.dequantize_rows(t, W, n_out, n_in).double(), dim=1)
    xn = torch.linalg.vector_norm(x.reshape(n_vec, n_in).double(), dim=1)
    tol = REL * want.double().abs() + ABS * xn[:, None] * wn[None, :]
    return bool(((got.double() - want.double()).abs() <= tol).all())


def oracle_close(t, W, x, got, n_out, n_in, n_vec, rng):
    """Sampled rows of got against the oracle's f64 sum of exact block sums."""
    import oracle
    W_host = W.cpu().numpy()
    x_host = x.cpu().numpy()
    xq = oracle.quantize(oracle.act_type(t), x_host)
    rows = sorted(set([0, n_out - 1] + list(rng.choice(n_out, size=min(24, n_out), replace=False))))
    rb = oracle.type_nbytes(t, n_in)
    ref = np.zeros((n_vec, n_out))
    for r in rows:
        oracle.gemv(t, W_host, xq, n_out, n_in, n_vec, rows=(r, r + 1), out=ref)
    wn = np.array([np.linalg.norm(oracle.dequantize(t, W_host[r * rb:(r + 1) * rb], n_in).astype(np.float64))
                   for r in rows])
    xn = np.linalg.norm(x_host.reshape(n_vec, n_in).astype(np.float64), axis=1)
    g = got.cpu().numpy()[:, rows].astype(np.float64)
    tol = REL * np.abs(ref[:, rows]) + ABS * xn[:, None] * wn[None, :]
    return bool((np.abs(g - ref[:, rows]) <= tol).all())


def test_noalloc_matches_qgemv_on_calls_in_a_row():
    rng = np.random.default_rng(77)
    # Q6_K with 8 vectors and Q8_0 with 4 fill the array further than the
    # calls after them (Q8_0 with 3 shorter vectors, Q4_K with 2), which read
    # only what they wrote; Q4_K 4096 with one vector quantizes inside the
    # product and does not touch the array.
    cases = [(qg.Q6_K, 1000, 11008, 8), (qg.Q4_K, 4096, 4096, 1), (qg.Q8_0, 700, 8192, 4),
             (qg.Q8_0, 300, 2048, 3), (qg.Q4_K, 513, 4096, 2)]
    inputs = []
    for t, n_out, n_in, n_vec in cases:
        if t == qg.Q8_0:
            import oracle
            W = torch.from_numpy(oracle.quantize(t, synth.f32_normal(rng, n_out * n_in, 0.02))).cuda()
        else:
            W = torch.from_numpy(synth.k_blocks(t, n_out * n_in // 256, rng)).cuda()
        x = torch.from_numpy(synth.f32_normal(rng, n_vec * n_in)).cuda()
        inputs.append((t, W, x, n_out, n_in, n_vec))
    ys = [torch.full((c[5], c[3]), np.nan, dtype=torch.float32, device="cuda") for c in inputs]
    for _ in range(2):
        # calls back to back on one stream, sharing the library's array
        for (t, W, x, n_out, n_in, n_vec), y in zip(inputs, ys):
            assert call_noalloc(t, W, x, y, n_out, n_in, n_vec) == 0
        torch.cuda.synchronize()
        for (t, W, x, n_out, n_in, n_vec), y in zip(inputs, ys):
            ref = qg.qgemv(t, W, x, n_out, n_in, n_vec)
            torch.cuda.synchronize()
            assert torch.isfinite(y).all()
            assert torch.equal(y, ref), (t, n_out, n_in, n_vec)
            assert close(t, W, x, y, ref, n_out, n_in, n_vec)
            assert oracle_close(t, W, x, y, n_out, n_in, n_vec, rng)
            y.fill_(np.nan)
        torch.cuda.synchronize()
    assert qg.device_error() == 0


def test_noalloc_rejects_more_than_its_array():
    # 8 vectors x 32768 Q8_K values need 8 * 128 * 292 bytes > 256 KiB
    t, n_in, n_vec = qg.Q4_K, 32768, 8
    assert qg.qgemv_workspace_bytes(t, n_in, n_vec) > SCRATCH_BYTES
    W = torch.zeros(16, dtype=torch.uint8, device="cuda")
    x = torch.zeros(n_vec * n_in, dtype=torch.float32, device="cuda")
    y = torch.zeros(n_vec, dtype=torch.float32, device="cuda")
    assert call_noalloc(t, W, x, y, 1, n_in, n_vec) == -7  # QG_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert y.abs().sum().item() == 0
