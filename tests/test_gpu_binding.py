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


def test_calls_on_a_side_stream_allocate_on_it():
    """With stream= and no workspace, a wrapper allocates its outputs and zeroes its workspace on
    that stream (torch stream or raw handle): the results equal those of the same calls on the
    current stream, bit for bit."""
    g = torch.Generator(device="cuda").manual_seed(3)
    B, T, H, V, k, D = 2, 8, 256, 4096, 8, 64
    hidden = torch.randn(B * T, H, device="cuda", generator=g).to(torch.bfloat16)
    W_vocab = (torch.randn(V, H, device="cuda", generator=g) * H ** -0.5).to(torch.bfloat16)
    W_sel = (torch.randn(D, H, device="cuda", generator=g) * H ** -0.5).to(torch.bfloat16)
    pred_cb = (torch.randn(V, D, device="cuda", generator=g) * 0.1).to(torch.bfloat16)
    succ_cb = (torch.randn(V, D, device="cuda", generator=g) * 0.1).to(torch.bfloat16)
    anchor = torch.randint(0, V, (B,), device="cuda", dtype=torch.int32, generator=g)
    logits = torch.randn(B * T, V, device="cuda", generator=g)
    ref_lat, ref_draft = df.dflash2_select(hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, k, T)
    ref_ids, ref_vals = df.dflash2_topk(logits, k)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    got = []
    for stream in (side, side.cuda_stream):
        for _ in range(3):
            lat, draft = df.dflash2_select(hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, k, T, stream=stream)
            ids, vals = df.dflash2_topk(logits, k, stream=stream)
        got.append((lat, draft, ids, vals))
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for lat, draft, ids, vals in got:
        assert torch.equal(lat.view(torch.int32), ref_lat.view(torch.int32))
        assert torch.equal(draft, ref_draft)
        assert torch.equal(ids, ref_ids)
        assert torch.equal(vals.view(torch.int32), ref_vals.view(torch.int32))
