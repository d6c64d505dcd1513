"""bpa_select_blocks_noalloc: block selection without caller-provided scratch.

Some callers cannot hand the library device memory: a host program without
a device allocator of its own should not call cudaMalloc next to running GPU
work (it may synchronise the device), and some embedders forbid device
allocations after start-up.  This entry point uses a scratch buffer compiled
into the library instead.  The test calls it through the C ABI twice in a
row, on different inputs, and requires the same block indices as the
workspace-taking entry point (selection is bit-exact, so equal means
identical).  It sits in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

from ring_attention_gb300.inputs import draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bpa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_attention_gb300 import build
    build.build()
    from ring_attention_gb300 import bpa as mod
    return mod


def _dev(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def test_noalloc_selection_matches_workspace_entry_point(bpa):
    B, S, H, d, bs, n = 4, 8192, 8, 64, 32, 8   # 10 MiB of block sums: inside the 16 MiB buffer
    first = draw([(B, S, H, d), (B, S, H, d)], 4, "bf16")
    second = draw([(B, S, H, d), (B, S, H, d)], 5, "bf16")
    for q_np, k_np in (first, second):          # two calls in a row share the buffer
        q, k = _dev(q_np), _dev(k_np)
        want = bpa.bpa_select_blocks(q, k, block_size=bs, top_n=n)
        got = bpa.bpa_select_blocks_noalloc(q, k, block_size=bs, top_n=n)
        torch.cuda.synchronize()
        assert torch.equal(got, want)


def test_noalloc_rejects_problems_beyond_the_buffer(bpa):
    limit = bpa.lib().bpa_select_noalloc_max_bytes()
    assert limit == 16 << 20
    q = torch.zeros((1, 65536, 8, 128), dtype=torch.bfloat16, device="cuda")   # 32 MiB of sums
    with pytest.raises(bpa.BpaError) as e:
        bpa.bpa_select_blocks_noalloc(q, q, block_size=32, top_n=8)
    assert e.value.status == bpa.BPA_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
