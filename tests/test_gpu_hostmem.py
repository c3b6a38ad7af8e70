"""Page-locked host buffers from kv_cache_eviction_gb300.hostmem.pinned_empty: page-locked,
the requested shape and dtype, and exact round trips through asynchronous copies."""
import gc

import pytest
import torch

from kv_cache_eviction_gb300.hostmem import pinned_empty

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,dtype", [((3, 5, 7), torch.bfloat16), ((1 << 26,), torch.uint8),
                                         ((2, 1024, 129), torch.float32), ((0, 4), torch.int32)])
def test_pinned_empty_round_trip(shape, dtype):
    h = pinned_empty(shape, dtype)
    assert tuple(h.shape) == shape and h.dtype == dtype and h.device.type == "cpu"
    assert h.numel() == 0 or h.is_pinned()
    g = torch.Generator().manual_seed(5)
    src = (torch.randint(0, 120, shape, generator=g) if not dtype.is_floating_point
           else torch.randn(shape, generator=g)).to(dtype)
    h.copy_(src)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        d = torch.empty(shape, dtype=dtype, device="cuda")
        d.copy_(h, non_blocking=True)
        back = pinned_empty(shape, dtype)
        back.copy_(d * 1, non_blocking=True)
    st.synchronize()
    assert torch.equal(back, src)


def test_pinned_empty_views_keep_the_memory():
    """A slice outlives the tensor it was cut from; freeing both releases the registration,
    and the same size can be registered again."""
    h = pinned_empty((8, 1 << 20), torch.uint8)
    h.fill_(3)
    part = h[2:4]
    del h
    gc.collect()
    d = part.to("cuda", non_blocking=True)
    torch.cuda.synchronize()
    assert int(d.sum()) == 3 * 2 * (1 << 20)
    del part, d
    gc.collect()
    again = pinned_empty((8, 1 << 20), torch.uint8)
    assert again.is_pinned()
