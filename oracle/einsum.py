"""Dense einsum for the two contraction shapes on the hot path (test infrastructure only).

``"mk,kn->mn"`` (a matrix product) and ``"bmk,bkn->bmn"`` (a batched one), in
float64. The matrix product itself is a library primitive (NumPy matmul);
``einsum_bruteforce`` writes the sum out with Python loops for tiny inputs and
pins it.
"""

import numpy as np

SPECS = {
    "mk,kn->mn": ("mk", "kn", "mn"),
    "bmk,bkn->bmn": ("bmk", "bkn", "bmn"),
}


def parse_spec(spec):
    """Return (lhs_labels, rhs_labels, out_labels) for a supported spec."""
    key = spec.replace(" ", "")
    if key not in SPECS:
        raise ValueError(f"unsupported einsum spec {spec!r}; supported: {sorted(SPECS)}")
    return SPECS[key]


def einsum(spec, lhs, rhs):
    """out[..., m, n] = sum_k lhs[..., m, k] * rhs[..., k, n] in float64."""
    parse_spec(spec)
    return np.matmul(np.asarray(lhs, np.float64), np.asarray(rhs, np.float64))


def einsum_bruteforce(spec, lhs, rhs):
    """The same contraction as four nested Python loops (tiny inputs only)."""
    lab_l, _, _ = parse_spec(spec)
    lhs = np.asarray(lhs, np.float64)
    rhs = np.asarray(rhs, np.float64)
    if len(lab_l) == 2:
        lhs = lhs[None]
        rhs = rhs[None]
    nb, m, k = lhs.shape
    n = rhs.shape[2]
    out = np.zeros((nb, m, n))
    for b in range(nb):
        for i in range(m):
            for j in range(n):
                s = 0.0
                for t in range(k):
                    s += lhs[b, i, t] * rhs[b, t, j]
                out[b, i, j] = s
    return out[0] if len(lab_l) == 2 else out
