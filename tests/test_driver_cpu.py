"""Host-side checks of the multi-segment driver (no GPU needed)."""
import pytest
import torch

import transformer_xl_relative_attn_gb300 as txl


def test_driver_needs_one_memory_per_layer():
    with pytest.raises(ValueError):
        txl.SegmentDriver([])


def test_driver_refuses_host_memories():
    with pytest.raises(ValueError):
        txl.SegmentDriver([torch.zeros(2, 8, 16, dtype=torch.bfloat16)])


def _stack_args(n=2, B=2, M=128, H=4, dh=64):
    d = H * dh
    z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    mems = [z(B, M, d)] + [z(B, H, M, dh) for _ in range(n - 1)]
    return [z(3 * d, d)] * n, [z(2 * M, H, dh)] * n, [z(H, dh)] * n, [z(H, dh)] * n, mems


def test_attn_stack_validates_its_arguments():
    w, r, u, v, mems = _stack_args()
    with pytest.raises(ValueError):           # one parameter set per layer
        txl.AttnStack(w[:1], r, u, v, mems, 0.125, 4, 128)
    with pytest.raises(ValueError):           # layer 0's memory must be rows
        txl.AttnStack(w, r, u, v, [mems[1], mems[1]], 0.125, 4, 128)
    bad = [mems[0], torch.zeros(2, 128, 256, dtype=torch.bfloat16)]
    with pytest.raises(ValueError):           # other memories in the heads layout
        txl.AttnStack(w, r, u, v, bad, 0.125, 4, 128)
    with pytest.raises(ValueError):           # host tensors: there is no CPU path
        txl.AttnStack(w, r, u, v, mems, 0.125, 4, 128)


def test_decoder_stack_validates_its_arguments():
    B, M, d = 2, 128, 256
    mems = [torch.zeros(B, M, d, dtype=torch.bfloat16)] * 2
    with pytest.raises(ValueError):           # one parameter set per layer
        txl.DecoderStack([{}], [None] * 2, [None] * 2, [None] * 2, mems, 0.125, 4, 128)
    with pytest.raises(ValueError):           # host memories
        txl.DecoderStack([{}, {}], [None] * 2, [None] * 2, [None] * 2, mems, 0.125, 4, 128)


def test_library_calls_refuse_host_tensors():
    x = torch.zeros(1, 128, 256, dtype=torch.bfloat16)
    with pytest.raises(Exception):
        txl.layer_norm(x, torch.ones(256, dtype=torch.bfloat16), torch.zeros(256, dtype=torch.bfloat16))
    with pytest.raises(Exception):
        txl.linear(x, torch.zeros(256, 256, dtype=torch.bfloat16))
