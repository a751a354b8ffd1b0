"""The float64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins as pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(lib, pin):
    pin(lib)


def test_thread_count_does_not_change_bits(lib):
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((2, 33, 8)) for _ in range(4))
    a = oracle.attn_fwd_bwd(q, k, v, do, 0.3, True, nthreads=1, lib=lib)
    b = oracle.attn_fwd_bwd(q, k, v, do, 0.3, True, nthreads=5, lib=lib)
    for n in a:
        assert np.array_equal(a[n], b[n]), n


def test_given_mode_matches_full_mode(lib):
    rng = np.random.default_rng(4)
    q, k, v, do = (rng.standard_normal((1, 17, 8)) for _ in range(4))
    for causal in (False, True):
        a = oracle.attn_fwd_bwd(q, k, v, do, 0.5, causal, lib=lib)
        b = oracle.attn_bwd_given(q, k, v, a["o"], a["lse"], do, 0.5, causal, lib=lib)
        for n in ("D", "dq", "dk", "dv"):
            assert np.allclose(a[n], b[n], rtol=0, atol=1e-13), n


def test_row_sampled_mode_matches_whole_head(lib):
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((40, 8)) for _ in range(4))
    qrows, krows = [0, 7, 39, 13], [39, 0, 22]
    for causal in (False, True):
        full = oracle.attn_fwd_bwd(q[None], k[None], v[None], do[None], 0.4, causal, lib=lib)
        for given in (False, True):
            kw = dict(lse_all=full["lse"][0], D_all=full["D"][0]) if given else {}
            part = oracle.attn_rows(q, k, v, do, 0.4, causal, qrows, krows, lib=lib, **kw)
            for n in ("o", "lse", "D", "dq"):
                assert np.array_equal(part[n], full[n][0][qrows]), n
            for n in ("dk", "dv"):
                assert np.array_equal(part[n], full[n][0][krows]), n
