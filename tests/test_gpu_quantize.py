"""mlx4g32 quantiser on the GPU vs the oracle: codes, scales and biases bit-exact."""
import numpy as np
import pytest
import torch

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import dev, host, need_gpu

pytestmark = pytest.mark.gpu


def _gpu_records(x):
    from prefix_cached_kv_gb300 import binding
    return host(binding.quantize_mlx4g32(dev(x)))


@pytest.mark.parametrize("rows,kv_dim", [(1, 32), (7, 64), (333, 512), (129, 1024), (5, 2048)])
def test_quantizer_bit_exact_fp16(rows, kv_dim):
    need_gpu()
    rng = np.random.default_rng(rows * 31 + kv_dim)
    x = (rng.standard_normal((rows, kv_dim)) * np.exp(rng.standard_normal((rows, 1)))).astype(np.float16)
    got = _gpu_records(x)
    want = orc.quantize_records(x)
    assert got.shape == want.shape == (rows, orc.record_bytes(kv_dim))
    assert np.array_equal(got, want)


def test_quantizer_bit_exact_fp32_input():
    need_gpu()
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((257, 256)) * 3).astype(np.float32)
    assert np.array_equal(_gpu_records(x), orc.quantize_records(x))


def test_quantizer_special_groups():
    """Constant groups, exact grids, tiny (subnormal-scale) groups, wide ranges, exact ties."""
    need_gpu()
    rng = np.random.default_rng(6)
    x = rng.standard_normal((16, 128)).astype(np.float16)
    x[0, :32] = np.float16(0.5)                                    # constant -> scale 0
    x[1, :32] = (np.arange(32) % 16 * 0.25).astype(np.float16)     # exact grid
    x[2, :32] = (rng.standard_normal(32) * 1e-5).astype(np.float16)  # subnormal-range values
    x[3, :32] = (rng.standard_normal(32) * 3000).astype(np.float16)  # wide range
    x[4, :32] = np.float16(0.0)
    x[4, 0] = np.float16(15.0)
    x[4, 1:16] = (np.arange(1, 16) - 0.5).astype(np.float16)       # t lands on .5 ties
    x[5, 32:64] = -np.float16(0.0)
    assert np.array_equal(_gpu_records(x), orc.quantize_records(x))


def test_quantizer_cartridge_layer_sampled():
    """A full cartridge layer (86,580 tokens x kv_dim 1024, N(0,1) fp16) quantised on the device;
    a seeded sample of rows checked against the oracle."""
    need_gpu()
    N, kv = 86580, 1024
    x = synth.torch_gen_rows_device(0, N, kv, "cuda", stream=1)
    from prefix_cached_kv_gb300 import binding
    rec = binding.quantize_mlx4g32(x)
    rows = np.sort(np.random.default_rng(7).choice(N, size=1500, replace=False))
    rows = np.concatenate([[0, N - 1], rows])
    xs = host(x[torch.from_numpy(rows).cuda()])
    got = host(rec[torch.from_numpy(rows).cuda()])
    assert np.array_equal(got, orc.quantize_records(xs))
