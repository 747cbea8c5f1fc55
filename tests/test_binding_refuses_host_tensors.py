"""The Python binding only marshals arguments: every compute entry point refuses host (CPU)
tensors with a TypeError before it reaches the library, so a caller without a GPU gets an
error, never a silent CPU computation (no GPU needed)."""
import pytest
import torch

from speculative_decoding_drafter_gb300 import build as build_mod

B, T, H, V, K, D = 1, 8, 256, 4096, 4, 64
R = B * T


@pytest.fixture(scope="module")
def df():
    build_mod.build()
    from speculative_decoding_drafter_gb300 import dflash2

    dflash2.library()
    return dflash2


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_select_refuses_host_tensors(df):
    with pytest.raises(TypeError, match="hidden must be a CUDA tensor"):
        df.dflash2_select(bf16(R, H), bf16(V, H), bf16(D, H), bf16(V, D), bf16(V, D),
                          torch.zeros(B, dtype=torch.int32), K, T)


def test_select_from_logits_refuses_host_tensors(df):
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        df.dflash2_select_from_logits(torch.zeros(R, V), bf16(R, H), bf16(D, H), bf16(V, D), bf16(V, D),
                                      torch.zeros(B, dtype=torch.int32), K, T)


@pytest.mark.parametrize("call", ["lm_head", "topk", "topk_noalloc", "gate", "lattice", "walk", "walk_sample",
                                  "conv"])
def test_stage_entry_points_refuse_host_tensors(df, call):
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        if call == "lm_head":
            df.dflash2_lm_head_logits(bf16(R, H), bf16(V, H))
        elif call == "topk":
            df.dflash2_topk(torch.zeros(R, V), K)
        elif call == "topk_noalloc":
            df.dflash2_topk_noalloc(torch.zeros(R, V), K)
        elif call == "gate":
            df.dflash2_gate(bf16(R, H), bf16(D, H))
        elif call == "lattice":
            df.dflash2_lattice(torch.zeros(R, K, dtype=torch.int32), torch.zeros(R, K), torch.zeros(R, D),
                               bf16(V, D), bf16(V, D), torch.zeros(B, dtype=torch.int32), T)
        elif call == "walk":
            df.dflash2_walk(torch.zeros(R, K + K * K), B, T, K)
        elif call == "walk_sample":
            df.dflash2_walk_sample(torch.zeros(R, K + K * K), B, T, K, p_min=0.5)
        else:
            df.dflash2_dynamic_conv(bf16(R, 64), bf16(2, 64), torch.zeros(R, 2, 4), T)
