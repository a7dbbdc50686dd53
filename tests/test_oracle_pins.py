"""The oracle against brute force, closed forms and invariants (no GPU)."""
import numpy as np
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


def test_library_cross_check(orc):
    """torch.softmax and scipy.special.softmax in float64 agree with the FP64 values."""
    torch = pytest.importorskip("torch")
    special = pytest.importorskip("scipy.special")
    import synth
    for name, rows in (("f32_4096x4096", 17), ("f16_causal_524288x2048", 9),
                       ("bf16_16384x1000_ld1024", 5)):
        w = synth.WORKLOADS[name].with_rows(rows)
        x = w.generate()
        xv = synth.storage_to_float64(x[:, :w.N], w.dtype)
        got = orc.softmax_rows_f64(x.reshape(-1), w.M, w.N, w.ld_in, w.dtype)
        t = torch.softmax(torch.from_numpy(xv), dim=1).numpy()
        s = special.softmax(xv, axis=1)
        assert np.allclose(got, t, rtol=1e-13, atol=1e-300)
        assert np.allclose(got, s, rtol=1e-13, atol=1e-300)


def test_oracle_rejects_bad_arguments(orc):
    x = np.zeros(16, dtype=np.float32)
    with pytest.raises(ValueError):
        orc.softmax_rows(x, 2, 8, 4, 8, 0)  # ld_in < N
    with pytest.raises(ValueError):
        orc.softmax_rows(x, 2, 0, 8, 8, 0)  # N < 1
    out = orc.softmax_rows(x, 0, 8, 8, 8, 0)  # M == 0 is a no-op
    assert out.shape == (0, 8)
