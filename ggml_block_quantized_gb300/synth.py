"""Seeded synthetic inputs for the block-quantized GEMV workloads.

This module draws random numbers and packs them into arrays; it contains none
of the method's arithmetic (no quantizer, no dequantizer, no dot product).
Both the tests (which feed the oracle) and the benchmark use it, so both
sides see identical bytes. All arrays are numpy, on the host.

Workloads (names used across tests and bench.py):
  q8_0_256x1024   Q8_0 weights from f32 N(0, 0.02), 256 x 1024, x ~ N(0, 1)
  q4_0_4096       Q4_0 weights from f32 N(0, 0.02), 4096 x 4096, x ~ N(0, 1)
  q4_k_4096       Q4_K random super-blocks, 4096 x 4096: d, dmin = f16 of
                  |N(0,1)| * 1e-3, 12 uniform scale bytes, 128 uniform qs bytes
  q6_k_32000      Q6_K random super-blocks, 32000 x 4096: ql and qh uniform
                  bytes, scales int8 uniform in [-32, 31], d = f16 of
                  |N(0,1)| * 1e-3 (stored last, at byte 208)
  layer_stack     32 decoder layers, each Q4_K q/k/v/o 4096 x 4096, Q4_K
                  gate/up 11008 x 4096, Q6_K down 4096 x 11008 (random blocks
                  as above), a fresh x ~ N(0, 1) per matrix and vector
  q4_1_32000      Q4_1 weights from f32 N(0, 0.02) + 0.01, 32000 x 4096, x ~ N(0, 1)
  q5_0_32000      Q5_0 weights from f32 N(0, 0.02), 32000 x 4096, x ~ N(0, 1)
  q2_k_32000, q3_k_32000, q5_k_32000
                  random Q2_K / Q3_K / Q5_K super-blocks (k_blocks), 32000 x 4096
                  (the output-projection shape of the Q6_K workload: large
                  enough that one call streams at the kernel's rate)
Seeds: weights 1000 + workload index, activations 2000 + workload index; the
layer stack derives per-(layer, matrix) streams from those.
"""
import numpy as np

Q4_0, Q4_1, Q5_0, Q8_0 = 2, 3, 6, 8
Q2_K, Q3_K, Q4_K, Q5_K, Q6_K = 10, 11, 12, 13, 14
BLOCK = {Q4_0: (32, 18), Q4_1: (32, 20), Q5_0: (32, 22), Q8_0: (32, 34), Q2_K: (256, 84),
         Q3_K: (256, 110), Q4_K: (256, 144), Q5_K: (256, 176), Q6_K: (256, 210)}
K_TYPES = (Q2_K, Q3_K, Q4_K, Q5_K, Q6_K)
FROM_F32 = (Q8_0, Q4_0, Q4_1, Q5_0)  # workloads that quantize f32 weights

WORKLOADS = ["q8_0_256x1024", "q4_0_4096", "q4_k_4096", "q6_k_32000", "layer_stack",
             "q4_1_32000", "q5_0_32000", "q2_k_32000", "q3_k_32000", "q5_k_32000"]

# (name, type, n_out, n_in) of one decoder layer of the stack
LAYER_MATRICES = [
    ("q", Q4_K, 4096, 4096),
    ("k", Q4_K, 4096, 4096),
    ("v", Q4_K, 4096, 4096),
    ("o", Q4_K, 4096, 4096),
    ("gate", Q4_K, 11008, 4096),
    ("up", Q4_K, 11008, 4096),
    ("down", Q6_K, 4096, 11008),
]
N_LAYERS = 32


def f32_normal(rng, n, std=1.0) -> np.ndarray:
    x = rng.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def random_bytes(rng, n) -> np.ndarray:
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).copy()


def _half_scales(rng, n) -> np.ndarray:
    """n f16 values |N(0,1)| * 1e-3, as little-endian byte pairs [n, 2]."""
    v = (np.abs(rng.standard_normal(n)) * 1e-3).astype(np.float16)
    return v.view(np.uint8).reshape(n, 2)


def k_blocks(wtype: int, n_blocks: int, rng) -> np.ndarray:
    """Random K-quant super-blocks (flat uint8, n_blocks * block bytes):
    uniform bytes, then the f16 d (and dmin) set to |N(0,1)| * 1e-3 and, for
    Q6_K, the int8 scales drawn uniform in [-32, 31]."""
    _, nbytes = BLOCK[wtype]
    raw = random_bytes(rng, n_blocks * nbytes).reshape(n_blocks, nbytes)
    if wtype in (Q4_K, Q5_K):
        raw[:, 0:2] = _half_scales(rng, n_blocks)
        raw[:, 2:4] = _half_scales(rng, n_blocks)
    elif wtype == Q2_K:
        raw[:, 80:82] = _half_scales(rng, n_blocks)
        raw[:, 82:84] = _half_scales(rng, n_blocks)
    elif wtype == Q3_K:
        raw[:, 108:110] = _half_scales(rng, n_blocks)
    elif wtype == Q6_K:
        sc = rng.integers(-32, 32, size=(n_blocks, 16), dtype=np.int8)
        raw[:, 192:208] = sc.view(np.uint8)
        raw[:, 208:210] = _half_scales(rng, n_blocks)
    else:
        raise ValueError("k_blocks takes a K-quant weight type")
    return raw.reshape(-1)


def legacy_blocks(wtype: int, n_blocks: int, rng) -> np.ndarray:
    """Random 32-element blocks with every code and bit pattern: uniform
    bytes, then d (and Q4_1's m) = f16 of N(0,1) * 1e-2 (d of either sign)."""
    _, nbytes = BLOCK[wtype]
    raw = random_bytes(rng, n_blocks * nbytes).reshape(n_blocks, nbytes)
    raw[:, 0:2] = (rng.standard_normal(n_blocks) * 1e-2).astype(np.float16).view(np.uint8).reshape(n_blocks, 2)
    if wtype == Q4_1:
        raw[:, 2:4] = (rng.standard_normal(n_blocks) * 1e-2).astype(np.float16).view(np.uint8).reshape(n_blocks, 2)
    return raw.reshape(-1)


def workload_index(name: str) -> int:
    return WORKLOADS.index(name) + 1


def single_matrix(name: str, n_vec: int = 1, n_out: int = None, n_in: int = None):
    """Inputs of one of the single-matrix workloads, optionally resized.

    Returns dict(type, n_out, n_in, n_vec, x[f32 n_vec*n_in], and either
    w_f32 (f32 weights to quantize, Q8_0/Q4_0/Q4_1/Q5_0) or w_blocks (uint8
    blocks)).
    """
    idx = workload_index(name)
    spec = {
        "q8_0_256x1024": (Q8_0, 256, 1024),
        "q4_0_4096": (Q4_0, 4096, 4096),
        "q4_k_4096": (Q4_K, 4096, 4096),
        "q6_k_32000": (Q6_K, 32000, 4096),
        "q4_1_32000": (Q4_1, 32000, 4096),
        "q5_0_32000": (Q5_0, 32000, 4096),
        "q2_k_32000": (Q2_K, 32000, 4096),
        "q3_k_32000": (Q3_K, 32000, 4096),
        "q5_k_32000": (Q5_K, 32000, 4096),
    }[name]
    t, d_out, d_in = spec
    n_out = d_out if n_out is None else n_out
    n_in = d_in if n_in is None else n_in
    wr = np.random.default_rng(1000 + idx)
    xr = np.random.default_rng(2000 + idx)
    out = dict(type=t, n_out=n_out, n_in=n_in, n_vec=n_vec, x=f32_normal(xr, n_vec * n_in))
    if t in FROM_F32:
        out["w_f32"] = f32_normal(wr, n_out * n_in, std=0.02)
        if t == Q4_1:  # off-centre rows, where the min of Q4_1 matters
            out["w_f32"] += np.float32(0.01)
    else:
        out["w_blocks"] = k_blocks(t, n_out * n_in // 256, wr)
    return out


def layer_x(layer: int, m: int, n_vec: int = 1) -> np.ndarray:
    """The activations of matrix m of decoder layer `layer` alone (the first
    n_in values are the same for every n_vec)."""
    n_in = LAYER_MATRICES[m][3]
    xr = np.random.default_rng([2000 + workload_index("layer_stack"), layer, m])
    return f32_normal(xr, n_vec * n_in)


def layer_matrix(layer: int, m: int, n_vec: int = 1):
    """Matrix m (index into LAYER_MATRICES) of decoder layer `layer`."""
    name, t, n_out, n_in = LAYER_MATRICES[m]
    idx = workload_index("layer_stack")
    wr = np.random.default_rng([1000 + idx, layer, m])
    return dict(name=name, type=t, n_out=n_out, n_in=n_in, n_vec=n_vec,
                w_blocks=k_blocks(t, n_out * n_in // 256, wr), x=layer_x(layer, m, n_vec))


def layer_stack_bytes() -> int:
    per_layer = sum(n_out * n_in // 256 * BLOCK[t][1] for _, t, n_out, n_in in LAYER_MATRICES)
    return per_layer * N_LAYERS
