"""Host packer (product C++ code, called through the C ABI) against the oracle:
canonical bytes identical byte for byte; device layout decodes to the same
weights; sizes agree.  CPU only."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as ORC
import workloads
import block_quantized_token_format_gb300 as qg
from _layout_ref import decode_device

FMTS = ["q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"]


def _special(n_out, n_in, seed):
    """Gaussian rows plus rows that hit the quantizers' edge cases."""
    W = workloads.gaussian(seed, (n_out, n_in), 0.02)
    if n_out >= 6:
        W[0] = 0.0                                   # all-zero row
        W[1, ::2] = -W[1, 1::2]                       # +- pairs: magnitude ties in every block
        W[2] = np.float32(1e-30)                      # tiny: fp16 scales underflow
        W[3] = workloads.gaussian(seed + 1, (n_in,), 1000.0)   # large values
        W[4, :] = np.float32(0.5)                     # constant row (affine s = 0)
        W[5, 7] = np.float32(3.0)                     # one outlier
    return W


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 64), (7, 128), (33, 256), (130, 2560), (6, 6144)])
def test_quantize_matches_oracle_bytes(fmt, shape):
    n_out, n_in = shape
    W = _special(n_out, n_in, 7 + n_in)
    ref = ORC.quantize(fmt, W)
    got = qg.qg_quantize(fmt, W)
    assert got.size == ref.size == ORC.weight_bytes(fmt, n_out, n_in)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(3, 64), (9, 320), (40, 2560)])
def test_device_layout_decodes_to_oracle_weights(fmt, shape):
    n_out, n_in = shape
    W = _special(n_out, n_in, 99 + n_in)
    canon = ORC.quantize(fmt, W)
    packed = qg.qg_to_device_layout(fmt, canon, n_out, n_in)
    assert packed.size == qg.qg_packed_bytes(fmt, n_out, n_in)
    assert np.array_equal(decode_device(fmt, packed, n_out, n_in), ORC.dequantize(fmt, canon, n_out, n_in))
    assert np.array_equal(qg.qg_pack(fmt, W), packed)


@pytest.mark.parametrize("fmt", FMTS)
def test_sizes(fmt):
    for n_out, n_in in [(1, 256), (248320, 2560), (248320, 5120), (12288, 2560), (3, 64)]:
        assert qg.qg_canonical_bytes(fmt, n_out, n_in) == ORC.weight_bytes(fmt, n_out, n_in)
        stride = qg.qg_row_stride(fmt, n_in)
        assert stride % 16 == 0 and stride >= ORC.weight_bytes(fmt, 1, n_in)
        if n_in % 256 == 0:
            assert qg.qg_packed_bytes(fmt, n_out, n_in) == ORC.weight_bytes(fmt, n_out, n_in)
    assert qg.qg_canonical_bytes(fmt, 0, 256) == 0
    assert qg.qg_packed_bytes(fmt, 4, 17) == 0


def test_row_prefix_is_a_packed_matrix():
    """A reduced draft vocabulary that is a row prefix needs no copy."""
    W = workloads.gaussian(3, (50, 2560), 0.02)
    full = qg.qg_pack("q8_0", W)
    part = qg.qg_pack("q8_0", W[:17])
    assert np.array_equal(full[: part.size], part)


def test_packer_threads_deterministic():
    W = workloads.gaussian(4, (4097, 512), 0.02)
    for fmt in FMTS:
        a = qg.qg_pack(fmt, W)
        b = np.concatenate([qg.qg_pack(fmt, W[i:i + 1000]) for i in range(0, 4097, 1000)])
        assert np.array_equal(a, b)


def test_packer_rejects_bad_shapes():
    with pytest.raises(qg.QGError):
        qg.qg_quantize("q8_0", np.zeros((2, 48), np.float32))
    with pytest.raises(qg.QGError):
        qg.qg_pack("affine4_g64", np.zeros((2, 96), np.float32))
