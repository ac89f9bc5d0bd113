"""bgtq_plan_save / bgtq_plan_load: a plan written as bytes and read back
rebuilds every table bit for bit; foreign, truncated, corrupted and
future-version records are refused.  Host-only plans: no GPU needed."""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from rope_aware_quantized_gb300 import synth


def _plan(seed=7, H=3, G=4, bits_per_key=384, v_bits=3, layout=0):
    li = synth.layer_inputs(seed, 0, H, G, 64, 1e6, 1.2, rope_layout=layout)
    bits, en = zip(*[bg.bgtq_alloc_bits(li.calib[h], bits_per_key, 8, layout) for h in range(H)])
    return bg.bgtq_plan_create(np.stack(bits), np.stack(en), G, bits_per_key, v_bits, 0xC0FFEE + seed, layout,
                               host_only=True)


@pytest.mark.parametrize("bits_per_key,v_bits,layout", [(384, 3, 0), (256, 2, 1), (128, 4, 0)])
def test_round_trip_rebuilds_identical_tables(bits_per_key, v_bits, layout):
    p = _plan(bits_per_key=bits_per_key, v_bits=v_bits, layout=layout)
    data = bg.bgtq_plan_save(p)
    q = bg.bgtq_plan_load(data, host_only=True)
    assert (q.n_kv_heads, q.group, q.bits_per_key, q.v_bits) == (p.n_kv_heads, p.group, p.bits_per_key, p.v_bits)
    for h in range(p.n_kv_heads):
        a, b = p.head_tables(h), q.head_tables(h)
        assert a.keys() == b.keys()
        for k in a:
            assert np.array_equal(a[k], b[k]), k
    for w in range(9):
        ca, ta = p.codebook(w)
        cb, tb = q.codebook(w)
        assert np.array_equal(ca, cb) and np.array_equal(ta, tb)
    assert bg.bgtq_plan_save(q) == data  # and the record itself is reproduced


def test_record_layout_and_size():
    p = _plan(H=2)
    data = bg.bgtq_plan_save(p)
    assert data[:8] == b"BGTQPLAN"
    assert int.from_bytes(data[8:12], "little") == 1
    assert len(data) == 8 + 4 + 5 * 4 + 8 + 2 * 64 * 9 + 8


def _code(fn):
    with pytest.raises(bg.BgtqError) as e:
        fn()
    return e.value.code


def test_bad_records_are_refused():
    data = bytearray(bg.bgtq_plan_save(_plan()))
    assert _code(lambda: bg.bgtq_plan_load(b"NOTAPLAN" + bytes(data[8:]), host_only=True)) == -1
    assert _code(lambda: bg.bgtq_plan_load(bytes(data[:-9]), host_only=True)) == -1
    bad = bytearray(data)
    bad[60] ^= 1  # one widths byte
    assert _code(lambda: bg.bgtq_plan_load(bytes(bad), host_only=True)) == -1
    newer = bytearray(data)
    newer[8] = 2
    assert _code(lambda: bg.bgtq_plan_load(bytes(newer), host_only=True)) == -2
