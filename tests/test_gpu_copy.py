"""mla_copy: stream-ordered copies by the SMs between device memory and
pinned host memory, bit-exact for every size and alignment, refused for
memory a kernel cannot reach and for overlapping ranges (no launch)."""
from __future__ import annotations

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from head_latent_attention_gb300 import _build
    _build.build()
    import head_latent_attention_gb300 as m
    return m


def payload(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 4097, (1 << 20) + 3])
@pytest.mark.parametrize("off", [0, 1, 8])
def test_copy_round_trip(mla, n, off):
    src_h = torch.empty(n + 16, dtype=torch.uint8).pin_memory()
    src_h.copy_(payload(n + 16, n + off))
    dev = torch.zeros(n + 32, dtype=torch.uint8, device="cuda")
    back = torch.zeros(n + 16, dtype=torch.uint8).pin_memory()
    assert mla.mla_copy(dev[off + 3:off + 3 + n], src_h[off:off + n]) == mla.MLA_OK  # host -> device
    assert mla.mla_copy(back[off:off + n], dev[off + 3:off + 3 + n]) == mla.MLA_OK  # device -> host
    torch.cuda.synchronize()
    assert torch.equal(back[off:off + n], src_h[off:off + n])
    assert int(dev[:off + 3].sum()) == 0 and int(dev[off + 3 + n:].sum()) == 0  # nothing outside the range
    dev2 = torch.zeros_like(dev)
    assert mla.mla_copy(dev2, dev) == mla.MLA_OK  # device -> device
    torch.cuda.synchronize()
    assert torch.equal(dev2, dev)


def test_copy_in_a_graph(mla):
    n = 655360
    src_h = payload(n, 7).pin_memory()
    dst_h = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert mla.mla_copy(dev, src_h) == mla.MLA_OK
        dev.add_(1)
        assert mla.mla_copy(dst_h, dev) == mla.MLA_OK
    for k in range(3):
        src_h.copy_(payload(n, 20 + k))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dst_h, src_h + 1)


def test_copy_refusals(mla):
    L = mla.load_library()
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(64, dtype=torch.uint8)  # not registered: no kernel may touch it
    n0 = mla.mla_launch_count()
    assert L.mla_copy(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(pageable.data_ptr()), 64,
                      None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_copy(ctypes.c_void_p(pageable.data_ptr()), ctypes.c_void_p(dev.data_ptr()), 64,
                      None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_copy(ctypes.c_void_p(dev.data_ptr() + 8), ctypes.c_void_p(dev.data_ptr()), 16,
                      None) == mla.MLA_ERR_INVALID_ARG  # overlapping
    assert mla.mla_launch_count() == n0
    with pytest.raises(ValueError):
        mla.mla_copy(dev, pageable)
    with pytest.raises(ValueError):
        mla.mla_copy(dev[:32], torch.zeros(64, dtype=torch.uint8, device="cuda"))
