"""Host checks of bgtq_prefill_attn (no GPU: the descriptor and the
arguments are checked before the plan, and the fake device addresses below
are never dereferenced)."""

import ctypes

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg

BASE = 1 << 20  # a 16-byte aligned fake address


def call(t=100, batch=1, q=BASE, out=BASE, out_dtype=0, scale=0.088, capacity=128):
    plan = bg.bgtq_plan_create(np.full((2, 64), 3, np.uint8), np.ones((2, 64)), 4, 384, 3, 1, host_only=True)
    desc = bg._native.BgtqCache(BASE, BASE, BASE, BASE, capacity)
    rc = bg.lib().bgtq_prefill_attn(plan.handle, None, q, BASE, BASE, batch, t, ctypes.byref(desc), out, out_dtype,
                                    scale, None)
    return rc, bg.lib().bgtq_last_error().decode()


def test_valid_arguments_reach_the_plan_check():
    rc, msg = call()
    assert rc == -1 and "host-only" in msg


def test_empty_prompt_is_a_no_op():
    assert call(t=0)[0] == 0 and call(batch=0)[0] == 0


@pytest.mark.parametrize("kw,code,frag", [
    (dict(t=200), -3, "capacity"),
    (dict(t=-1), -1, ">= 0"),
    (dict(q=BASE + 8), -1, "16-byte aligned"),
    (dict(out=BASE + 8), -1, "16-byte aligned"),
    (dict(out_dtype=2), -1, "out_dtype"),
    (dict(scale=0.0), -1, "softmax_scale"),
    (dict(scale=float("inf")), -1, "softmax_scale"),
    (dict(batch=70000), -2, "65535"),
    (dict(batch=65535, t=5000, capacity=1 << 20), -2, "2^31"),
])
def test_bad_arguments_are_rejected(kw, code, frag):
    rc, msg = call(**kw)
    assert rc == code and frag in msg, (rc, msg)


def chunk_call(t=100, batch=1, q=BASE, out=BASE, pos=BASE, recent=0, capacity=128, max_prefix=16, ws=BASE,
               ws_bytes=1 << 30):
    plan = bg.bgtq_plan_create(np.full((2, 64), 3, np.uint8), np.ones((2, 64)), 4, 384, 3, 1, host_only=True)
    desc = bg._native.BgtqCache(BASE, BASE, BASE, BASE, capacity)
    if recent:
        desc.k_recent = BASE
        desc.recent = recent
    rc = bg.lib().bgtq_prefill_chunk_attn(plan.handle, None, q, BASE, BASE, batch, t, pos, max_prefix,
                                          ctypes.byref(desc), out, 0, 0.088, ws, ws_bytes, None)
    return rc, bg.lib().bgtq_last_error().decode()


def test_chunk_workspace_size():
    plan = bg.bgtq_plan_create(np.full((2, 64), 3, np.uint8), np.ones((2, 64)), 4, 384, 3, 1, host_only=True)
    # (512 + 8) bytes per (sequence, KV head, position up to max_prefix rounded up to 128)
    assert bg.bgtq_prefill_chunk_workspace(plan, 3, 300) == 3 * 2 * 384 * 520
    assert bg.bgtq_prefill_chunk_workspace(plan, 1, 0) == 0


def test_chunk_valid_arguments_reach_the_plan_check():
    rc, msg = chunk_call()
    assert rc == -1 and "host-only" in msg


@pytest.mark.parametrize("kw,code,frag", [
    (dict(t=200), -3, "capacity"),
    (dict(pos=None), -1, "NULL"),
    (dict(q=BASE + 8), -1, "16-byte aligned"),
    (dict(out=BASE + 8), -1, "16-byte aligned"),
    (dict(recent=16), -2, "recent-key"),
    (dict(max_prefix=200), -3, "max_prefix"),
    (dict(max_prefix=-1), -1, "max_prefix"),
    (dict(ws_bytes=100), -4, "workspace"),
    (dict(ws=BASE + 64), -1, "256-byte"),
])
def test_chunk_bad_arguments_are_rejected(kw, code, frag):
    rc, msg = chunk_call(**kw)
    assert rc == code and frag in msg, (rc, msg)
