"""Page-locked host buffers for staging a step's inputs to the GPU.

The eviction pass reads every K and V row of a prefill, so a caller whose cache lives in host
memory copies gigabytes per step across the host link.  On GB300 hosts whose memory uses
64 KB pages behind an IOMMU (as in the virtual machines this was measured on), copies from
ordinary pinned memory (``torch.empty(..., pin_memory=True)``) ran anywhere between 28 and
211 GB/s from one 8.6 GB copy to the next, while the same copies from memory backed by the
kernel's huge pages ran at 211 GB/s every time.  ``pinned_empty`` therefore maps an anonymous
region, asks the kernel for transparent huge pages on it (``MADV_HUGEPAGE``, which the
``madvise`` THP mode honours), touches it so the pages exist, and registers it with the CUDA
driver as page-locked memory.  Where any of that is refused it falls back to torch's pinned
allocator, so the result is always page-locked host memory.
"""
from __future__ import annotations

import ctypes
import mmap
import weakref

import torch

__all__ = ["pinned_empty"]


def pinned_empty(shape, dtype: torch.dtype) -> torch.Tensor:
    """An uninitialised, page-locked host tensor of `shape` and `dtype`.

    The memory is an anonymous mapping advised for huge pages and registered with
    cudaHostRegister (unregistered once the tensor and every view of it are freed), or, where
    the advice or the registration is not available, torch's own pinned memory.  Needs a CUDA
    device (registration goes through the CUDA runtime).  As with any page-locked buffer
    handed to asynchronous copies, synchronise with the copies that read or write it before
    dropping the last reference."""
    shape = tuple(int(s) for s in shape)
    elsize = torch.empty((), dtype=dtype).element_size()
    numel = 1
    for s in shape:
        numel *= s
    nbytes = numel * elsize
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    try:
        m = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    except (OSError, ValueError, AttributeError):
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    try:
        m.madvise(mmap.MADV_HUGEPAGE)
    except (AttributeError, OSError, ValueError):
        pass   # no THP advice here: the registration below still pins the pages
    buf = (ctypes.c_char * nbytes).from_buffer(m)
    addr = ctypes.addressof(buf)
    ctypes.memset(addr, 0, nbytes)   # fault the (huge) pages in before they are pinned
    rt = torch.cuda.cudart()
    if int(rt.cudaHostRegister(addr, nbytes, 0)) != 0:
        del buf
        m.close()
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    base = torch.frombuffer(buf, dtype=dtype, count=numel)

    def release(rt=rt, addr=addr, m=m):
        rt.cudaHostUnregister(addr)

    # views keep their base alive, so this runs once nothing refers to the memory any more
    # (the base holds the ctypes buffer, which holds the mapping)
    weakref.finalize(base, release)
    return base.view(shape)
