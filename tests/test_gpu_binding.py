"""The Python binding on a GPU: arguments are checked before the library is called."""
import pytest
import torch

from speculative_decoding_drafter_gb300 import dflash2 as df

pytestmark = pytest.mark.gpu


def test_binding_refuses_a_tensor_off_the_current_device(monkeypatch):
    """The library launches on the current device (and takes that device's scratch); the binding
    refuses a tensor that lives on another one.  With one GPU the 'current device' is moved
    instead of the tensor."""
    logits = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    here = torch.cuda.current_device()
    monkeypatch.setattr(torch.cuda, "current_device", lambda: here + 1)
    with pytest.raises(ValueError, match="not on the current device"):
        df.dflash2_topk_noalloc(logits, 4)
    with pytest.raises(ValueError, match="not on the current device"):
        df.dflash2_topk(logits, 4)
