"""Host-side behaviour of the C ABI on a GPU: slot states (HIT / MISS / COLDMISS), drop,
replacement, argument checks that fail before any launch, and counters."""
import numpy as np
import pytest
import torch

from prefix_cached_kv_gb300 import binding, synth
from tests.gpu_util import ctx_factory, dev, need_gpu

pytestmark = pytest.mark.gpu


def test_lookup_drop_and_coldmiss():
    need_gpu()
    c = binding.Context(0, max_slots=2)
    K, V = synth.gen_kv(1, 2, 64, 64)
    assert c.lookup("a", 0) == binding.MISS
    c.store("a", 0, dev(K), dev(V))
    c.store("a", 1, dev(K), dev(V))
    assert c.lookup("a", 0) == binding.OK and c.lookup("a", 1) == binding.OK
    Q = dev(synth.gen_q(1, 2, 1, 64))
    c.query("a", 0, Q)                        # a/0 is now the most recent
    c.store("b", 0, dev(K), dev(V))           # evicts a/1 (LRU)
    assert c.lookup("a", 1) == binding.COLDMISS
    with pytest.raises(binding.PckError) as e:
        c.query("a", 1, Q)
    assert e.value.code == binding.COLDMISS
    c.store("a", 1, dev(K), dev(V))           # re-store: warm again
    assert c.lookup("a", 1) == binding.OK
    info = c.info()
    assert info["slots_used"] == 2 and info["evictions"] >= 2
    assert c.drop("a") >= 1
    assert c.lookup("a", 1) == binding.MISS or c.lookup("a", 1) == binding.COLDMISS
    with pytest.raises(binding.PckError) as e:
        c.query("zz", 0, Q)
    assert e.value.code == binding.MISS
    c.close()


def test_argument_errors_before_launch():
    need_gpu()
    c = ctx_factory()
    K, V = synth.gen_kv(2, 2, 64, 64)
    c.store("e", 0, dev(K), dev(V))
    Q = dev(synth.gen_q(2, 4, 1, 64))
    with pytest.raises(binding.PckError) as e:
        c.query("e", 0, Q, top_k=10)
    assert e.value.code == binding.EUNSUPPORTED
    with pytest.raises(binding.PckError) as e:
        c.query("e", 0, Q, fa_window=-3)
    assert e.value.code == binding.EINVAL
    with pytest.raises(binding.PckError) as e:
        c.query("e", 0, Q, head_map=[0, 1, 2, 0])
    assert e.value.code == binding.EINVAL
    K80 = torch.zeros((1, 8, 80), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.PckError) as e:
        c.store("e", 1, K80, K80)
    assert e.value.code == binding.EUNSUPPORTED
    K96 = torch.zeros((1, 8, 96), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.PckError) as e:   # 96 has fp16 kernels only
        c.store("e", 1, K96, K96, fmt=binding.FMT_MLX4G32)
    assert e.value.code == binding.EUNSUPPORTED
    Q128 = dev(synth.gen_q(2, 4, 1, 128))
    with pytest.raises(binding.PckError) as e:
        c.query("e", 0, Q128)
    assert e.value.code == binding.EINVAL
    # top_k >= N is dense and accepted
    O, _ = c.query("e", 0, Q, top_k=64)
    c.sync()
    assert torch.isfinite(O).all()
    c.close()


def test_replace_slot_changes_answer():
    need_gpu()
    c = ctx_factory()
    K, V = synth.gen_kv(3, 1, 32, 64)
    c.store("r", 0, dev(K), dev(V))
    Q = dev(synth.gen_q(3, 1, 1, 64))
    O1, _ = c.query("r", 0, Q)
    c.store("r", 0, dev(K), dev(np.ascontiguousarray(V * np.float16(2))))
    O2, _ = c.query("r", 0, Q)
    c.sync()
    assert torch.allclose(O2, 2 * O1, atol=2e-3)
    c.close()
