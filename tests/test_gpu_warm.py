"""The WARM / FETCH RANGE dequantise-and-transpose (mlx4g32 records -> [H_kv, N, D] fp32 or fp16)
on the GPU: bit-exact against the oracle's definition (fp32 rounded once from the exact value;
fp16 rounded from that fp32)."""
import numpy as np
import pytest
import torch

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import dev, host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,H_kv,D", [(1000, 8, 128), (1, 1, 64), (333, 2, 96), (77, 4, 256), (4096, 8, 64)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_dequantize_records_bit_exact(N, H_kv, D, dtype):
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    rng = np.random.default_rng(N + D)
    x = (rng.standard_normal((N, H_kv * D)) * np.exp(rng.standard_normal((N, 1)))).astype(np.float16)
    x[:, :32] = (60 + 0.02 * rng.standard_normal((N, 32))).astype(np.float16)   # large bias, tiny scale
    rec = orc.quantize_records(x)
    got = host(binding.dequantize_mlx4g32(dev(rec), N, H_kv, D, dtype=dtype))
    want = orc.warm_heads(rec, H_kv, D, np.float32 if dtype == torch.float32 else np.float16)
    assert got.shape == (H_kv, N, D) and got.dtype == want.dtype
    assert np.array_equal(got.view(np.uint32 if dtype == torch.float32 else np.uint16),
                          want.view(np.uint32 if dtype == torch.float32 else np.uint16))


def test_dequantize_device_quantised_cartridge_layer_sampled():
    """One cartridge layer (86,580 tokens x kv_dim 1024) quantised by the library and dequantised
    back to [8, N, 128] fp32; a seeded sample of tokens checked against the oracle."""
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    N, H_kv, D = 86580, 8, 128
    x = synth.torch_gen_rows_device(1, N, H_kv * D, "cuda", stream=2)
    rec = binding.quantize_mlx4g32(x)
    out = binding.dequantize_mlx4g32(rec, N, H_kv, D)
    rows = np.sort(np.random.default_rng(9).choice(N, size=500, replace=False))
    sel = torch.from_numpy(rows).cuda()
    want = orc.warm_heads(host(rec[sel]), H_kv, D)
    got = host(out[:, sel])
    assert np.array_equal(got, want)


def test_dequantize_rejects_bad_arguments():
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library()
    import ctypes
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    p4 = ctypes.c_void_p(buf.data_ptr() + 4)
    p2 = ctypes.c_void_p(buf.data_ptr() + 2)
    assert lib.pck_dequantize_mlx4g32(p, 4, 1, 48, binding.DT_F32, p, None) == binding.EINVAL    # kv_dim % 32
    assert lib.pck_dequantize_mlx4g32(p, 4, 1, 64, 9, p, None) == binding.EINVAL                 # dtype
    assert lib.pck_dequantize_mlx4g32(p2, 4, 1, 64, binding.DT_F32, p, None) == binding.EINVAL   # records align
    assert lib.pck_dequantize_mlx4g32(p, 4, 1, 64, binding.DT_F32, p4, None) == binding.EINVAL   # out align
    assert lib.pck_dequantize_mlx4g32(p, 0, 1, 64, binding.DT_F32, p, None) == binding.OK
