"""Host checks of a paged cache descriptor and the binding's paged views
(no GPU: the descriptor is checked before the plan, and the fake device
addresses below are never dereferenced)."""

import ctypes

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg

BASE = 1 << 20  # a 16-byte aligned fake address


def host_plan():
    return bg.bgtq_plan_create(np.full((1, 64), 3, np.uint8), np.ones((1, 64)), 4, 384, 3, 1, host_only=True)


def append_with(**kw):
    d = dict(k_codes=BASE, k_norm=BASE, v_codes=BASE, v_norm=BASE, capacity=1024, k_recent=None, recent=0,
             page_table=BASE, max_pages=16, page_tokens=64, n_pages=20)
    d.update(kw)
    desc = bg._native.BgtqCache(**d)
    plan = host_plan()
    rc = bg.lib().bgtq_quantize_append(plan.handle, None, BASE, BASE, 1, 1, BASE, ctypes.byref(desc), None)
    return rc, bg.lib().bgtq_last_error().decode()


def test_valid_paged_descriptor_passes_the_cache_checks():
    rc, msg = append_with()
    assert rc == -1
    assert "host-only" in msg  # refused only because the plan has no device tables


@pytest.mark.parametrize("kw,frag", [
    (dict(page_tokens=24, capacity=16 * 24), "power of two"),
    (dict(page_tokens=8, capacity=16 * 8), "power of two"),
    (dict(page_tokens=1 << 21, capacity=16 << 21), "power of two"),
    (dict(capacity=1000), "capacity == max_pages"),
    (dict(n_pages=0), "n_pages"),
    (dict(max_pages=0, capacity=64), "max_pages"),
    (dict(page_table=BASE + 2), "4-byte aligned"),
    (dict(max_pages=(1 << 21) // 64 + 1, capacity=((1 << 21) // 64 + 1) * 64), "at most 2^21"),
])
def test_bad_paged_descriptors_are_rejected(kw, frag):
    rc, msg = append_with(**kw)
    assert rc == -1 and frag in msg, msg


def test_contiguous_descriptor_ignores_the_paging_fields():
    rc, msg = append_with(page_table=None, max_pages=0, page_tokens=3, n_pages=0)
    assert rc == -1 and "host-only" in msg


def test_paged_cache_views_share_the_pools():
    torch = pytest.importorskip("torch")
    plan = host_plan()
    c = bg.Cache(plan, 3, 256, device="cpu", recent=8, page_tokens=64)
    assert c.max_pages == 4 and c.n_pages == 12
    assert torch.equal(c.page_table.view(-1), torch.arange(12, dtype=torch.int32))
    kb, vb, nb = bg.bgtq_cache_bytes(plan, 12, 64)
    assert c.k_codes.numel() == kb and c.v_codes.numel() == vb and c.k_norm.numel() * 4 == nb
    for b in range(3):
        d = c.sequence_view(b).desc
        assert d.k_codes == c.k_codes.data_ptr() and d.v_norm == c.v_norm.data_ptr()
        assert d.page_table == c.page_table.data_ptr() + 4 * b * c.max_pages
        assert d.k_recent == c.k_recent.data_ptr() + b * 1 * 8 * 128 * 2
        assert (d.max_pages, d.page_tokens, d.n_pages, d.capacity) == (4, 64, 12, 256)
    with pytest.raises(ValueError):
        bg.Cache(plan, 1, 100, device="cpu", page_tokens=64)
    small = bg.Cache(plan, 2, 128, device="cpu", page_tokens=64, n_pages=3)
    assert small.page_table.view(-1).tolist() == [0, 1, 2, -1]
