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
