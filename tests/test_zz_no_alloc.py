"""moe_align_noalloc against moe_align, through the C ABI.

moe_align_noalloc is for callers that cannot allocate device memory when they
call in (runtimes that plan all device memory up front, plugin hooks that may
not allocate): it uses the library's own fixed scratch array instead of a
caller-supplied workspace.  Its results must equal moe_align's exactly (they
are integers).  This file is collected last, so a failure here leaves every
other test already run."""
import ctypes

import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe

pytestmark = pytest.mark.gpu


def _ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.argsort(torch.rand((T, E), generator=g), dim=1)[:, :k].to(torch.int32).contiguous()


def _noalloc_equals_align(ids, E, dev):
    T, k = ids.shape
    ids = ids.to(dev)
    ref = moe.moe_align(ids, E)
    got = moe.Alignment(T, k, E, dev)
    for t in (got.expert_offsets, got.sorted_slot, got.inv_slot, got.tile_map, got.num_tiles):
        t.fill_(-7)  # every output must be written by the call
    moe.moe_align_noalloc(ids, E, out=got)
    torch.cuda.synchronize()
    S = T * k
    n = int(ref.num_tiles.item())
    assert int(got.num_tiles.item()) == n
    assert torch.equal(got.expert_offsets, ref.expert_offsets)
    assert torch.equal(got.sorted_slot[:S], ref.sorted_slot[:S])
    assert torch.equal(got.inv_slot[:S], ref.inv_slot[:S])
    assert torch.equal(got.tile_map[:n], ref.tile_map[:n])


def test_noalloc_matches_align_on_two_calls_in_a_row(cuda_dev):
    # a large problem, then a small one that starts from the first call's
    # leftover scratch contents
    assert moe.align_workspace_size(4096, 8, 256) <= moe.ALIGN_NOALLOC_SCRATCH_BYTES
    _noalloc_equals_align(_ids(4096, 8, 256, 1), 256, cuda_dev)
    _noalloc_equals_align(_ids(300, 2, 8, 2), 8, cuda_dev)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_dev):
    T, k, E = 100000, 8, 1024
    assert moe.align_workspace_size(T, k, E) > moe.ALIGN_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = moe.lib().moe_align_noalloc(fake, T, k, E, 128, fake, fake, fake, fake, fake, None)
    assert st == moe.MOE_ERR_WORKSPACE
