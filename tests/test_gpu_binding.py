"""The binding refuses a tensor that is not on the current CUDA device (the
library launches there, so its kernels would dereference another GPU's
memory).  Nothing is launched: the check raises while the arguments are
marshalled."""

import pytest
import torch

pytestmark = pytest.mark.gpu

qasc = pytest.importorskip("query_aware_sparse_compressed_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qasc._lib.load()


def test_tensor_on_another_device_is_rejected(monkeypatch):
    K = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((1, 128, 32), dtype=torch.bfloat16, device="cuda")
    index = torch.zeros((1, 1, 8, 32), dtype=torch.bfloat16, device="cuda")
    other = K.device.index + 1
    monkeypatch.setattr(torch.cuda, "current_device", lambda: other)
    with pytest.raises(ValueError, match="current device is cuda:%d" % other):
        qasc.ts_index_append(K, W, index, 0, 8)


def test_tensors_on_the_current_device_are_accepted():
    K = torch.randn((1, 1, 8, 128), device="cuda").to(torch.bfloat16)
    W = torch.randn((1, 128, 32), device="cuda").to(torch.bfloat16)
    index = torch.zeros((1, 1, 8, 32), dtype=torch.bfloat16, device="cuda")
    qasc.ts_index_append(K, W, index, 0, 8)
    torch.cuda.synchronize()
    assert index.abs().sum().item() > 0
