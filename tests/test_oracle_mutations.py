"""Plant plausible mistakes in copies of the oracle; each must fail a pin.

The mistakes are planted in a temporary copy of the oracle's C source, on the
CPU; the committed oracle is never modified.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (label, text to replace, replacement, which occurrence (0-based))
MUTATIONS = [
    ("drop scale on dQ", "dq_r[x] *= h->scale;", ";", 0),
    ("drop scale on dK", "dk_c[x] *= h->scale;", ";", 0),
    ("sign of D in dS", "const double ds = p[c] * (dp - D);", "const double ds = p[c] * (dp + D);", 0),
    ("D forgotten in dK pass", "const double ds = p * (dp - h->D[r]);", "const double ds = p * dp;", 0),
    ("causal keeps future key", "if (h->causal && c > r) return 1;", "if (h->causal && c > r + 1) return 1;", 0),
    ("causal drops diagonal", "if (h->causal && c > r) return 1;", "if (h->causal && c >= r && r > 0) return 1;", 0),
    ("log base 2 for LSE", "m + log(sum)", "m + log2(sum)", 0),
    ("dV uses Q", "dv_c[x] += p * do_r[x];", "dv_c[x] += p * q_r[x];", 0),
    ("dK uses K", "dk_c[x] += ds * q_r[x];", "dk_c[x] += ds * k_c[x];", 0),
    ("dQ uses V", "dq_r[x] += ds * k_c[x];", "dq_r[x] += ds * h->v[(size_t)c * d + x];", 0),
    ("dP transposed (dO.k)", "const double dp = dot(do_r, h->v + (size_t)c * d, d); /* 8 */",
     "const double dp = dot(do_r, h->k + (size_t)c * d, d); /* 8 */", 0),
    ("D from dO.dO", "D = dot(do_r, o_r, d);", "D = dot(do_r, do_r, d);", 0),
    ("masked keys in dK/dV pass", "if (is_masked(h, r, c)) continue;", ";", 2),
    ("block table transposed", "h->tiles[(size_t)(r / BLOCK_TILE) * h->ntiles + c / BLOCK_TILE]",
     "h->tiles[(size_t)(c / BLOCK_TILE) * h->ntiles + r / BLOCK_TILE]", 0),
    ("block mask ignored", "return h->tiles != NULL && ", "return 0 && h->tiles != NULL && ", 0),
    ("empty row gets LSE 0", ": -INFINITY; /* no visible key", ": 0.0; /* no visible key", 0),
    ("no scale in scores", "s[c] = h->scale * dot(q_r, h->k + (size_t)c * d, d);",
     "s[c] = dot(q_r, h->k + (size_t)c * d, d);", 0),
]


def _mutate(text, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"mutation target not found: {old!r} (occurrence {occ})"
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("label,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(label, old, new, occ):
    with open(SRC) as f:
        text = f.read()
    mutated = _mutate(text, old, new, occ)
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "mut.c")
        with open(src, "w") as f:
            f.write(mutated)
        lib_path = oracle.build(src=src, out=os.path.join(td, "libmut.so"), force=True)
        lib = oracle.load(lib_path)
        failures = []
        for pin in pins.ALL_PINS:
            try:
                pin(lib)
            except (AssertionError, RuntimeError, FloatingPointError) as e:
                failures.append(pin.__name__)
        assert failures, f"mutation '{label}' passed every pin"
