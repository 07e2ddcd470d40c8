"""The timeline tool's analysis (CPU): per-phase statistics of synthetic
%globaltimer stamps, relative to the previous launch's end."""
import numpy as np

from paged_gqa_decode_head_gb300 import timeline


def _stamps(layers=8, ctas=5, slots=12, period=10_000):
    """Layer l's CTA c stamps phase s at l * period + 100 * s + 10 * c (ns);
    the merge (slot 10) only on CTA 0, the last to finish."""
    d = np.zeros((layers, ctas, slots), dtype=np.int64)
    for l in range(layers):
        for c in range(ctas):
            for s in range(10):
                d[l, c, s] = l * period + 100 * s + 10 * c + 1
        d[l, 0, 10] = l * period + 2000
    return d


def test_layer_ends_take_the_merge_else_the_last_state_write():
    d = _stamps()
    assert timeline._layer_ends(d) == [l * 10_000 + 2000 for l in range(8)]
    d[:, :, 10] = 0  # no in-kernel merge: the last partition state written
    assert timeline._layer_ends(d) == [l * 10_000 + 800 + 40 + 1 for l in range(8)]


def test_summarise_measures_phases_from_the_previous_layer_end():
    d = _stamps()
    out, length = timeline.summarise(d, first_layer=4)
    # each layer starts 10 us after the previous one and ends 2 us into it
    assert np.isclose(length, 10.0)
    for s in range(10):
        lo, med, hi = out[s]
        base = (10_000 + 100 * s + 1 - 2000) / 1e3
        assert np.isclose(lo, base) and np.isclose(med, base + 0.02) and np.isclose(hi, base + 0.04)
    assert np.allclose(out[10], (10.0,) * 3)


def test_summarise_skips_phases_no_cta_stamped():
    d = _stamps()
    d[:, :, 4] = 0  # attention alone: no query rotation
    out, _ = timeline.summarise(d)
    assert 4 not in out and 3 in out
