"""FusedAllReduce semantics: AllReduce -> +bias -> Dropout -> +residual (test infrastructure only).

[CoCoNet] Fig. 3 (lines 9-13 of its program): ``sum = AllReduce(layer)``,
then the bias is added with PyTorch broadcasting, dropout is applied as an
activation, and the residual is added. FusedAllReduce (§5.2) computes the same
values without storing ``sum``; the oracle computes them unfused, in float64.

Dropout randomness. The pages give no random number generator, so the mask is
a counter-based hash of (seed, element index), the plainest reading that makes
replicated outputs identical on every rank:

* ``e`` is the 0-based row-major index of the element inside one rank's output
  tensor (the same on every rank and in every group);
* ``z`` is the (e+1)-th output of SplitMix64 started from state ``seed``
  (Steele, Lea and Flood, "Fast Splittable Pseudorandom Number Generators",
  OOPSLA 2014): the state advances by the golden-gamma constant and the
  output is the variant-13 64-bit finaliser of the state;
* an element is kept iff ``z >> 40 < T`` with ``T = floor((1 - p) * 2**24)``,
  ``p`` taken as an IEEE single (the C interface passes a float) and the
  product formed in double precision;
* kept values are scaled by ``1 / (1 - p)``; dropped values become 0 before
  the residual is added. ``p = 0`` keeps everything with scale 1.
"""

import numpy as np

_MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB


def splitmix64(seed, count):
    """The first ``count`` outputs of SplitMix64 seeded with ``seed`` (Python ints).

    The published generator: state += gamma; z = state; z = (z ^ z>>30) * M1;
    z = (z ^ z>>27) * M2; return z ^ z>>31 (all modulo 2**64).
    """
    out = []
    state = seed & _MASK64
    for _ in range(count):
        state = (state + GOLDEN_GAMMA) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * _MIX1) & _MASK64
        z = ((z ^ (z >> 27)) * _MIX2) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def counter_hash(seed, index):
    """Vectorised ``splitmix64(seed, e+1)[e]`` for an array of element indices ``e``.

    uint64 NumPy arithmetic wraps modulo 2**64, as the generator requires.
    """
    e = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + (e + np.uint64(1)) * np.uint64(GOLDEN_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
        z = z ^ (z >> np.uint64(31))
    return z


def keep_threshold(p):
    """T = floor((1 - p) * 2**24) with p rounded to an IEEE single first."""
    p32 = float(np.float32(p))
    if not 0.0 <= p32 <= 1.0:
        raise ValueError("dropout probability must lie in [0, 1]")
    return int(np.floor((1.0 - p32) * float(1 << 24)))


def dropout_scale(p):
    """1 / (1 - p) for kept elements (float64; p rounded to an IEEE single)."""
    p32 = float(np.float32(p))
    return 1.0 if p32 == 0.0 else (np.inf if p32 == 1.0 else 1.0 / (1.0 - p32))


def keep_mask(seed, p, index):
    """Boolean keep mask for element indices ``index`` (see module docstring)."""
    t = keep_threshold(p)
    return (counter_hash(seed, index) >> np.uint64(40)) < np.uint64(t)


def fused_allreduce(partials, bias=None, residual=None, p=0.0, seed=0, index=None):
    """The value every rank holds after [CoCoNet] Fig. 3's lines 9-13.

    ``partials[r]`` is rank r's local tensor; ``bias`` is a 1-D tensor over the
    last dimension (PyTorch broadcast, the only broadcast the interface
    accepts) or None; ``residual`` is the replicated residual or None. Returns
    one float64 array (the replicated result).

    ``index`` (optional, same shape as the partials) gives each value's element
    index in the full per-rank tensor, for evaluating a sample of rows; the
    default is the row-major position inside the given arrays.
    """
    total = None
    for x in partials:  # AllReduce, summed in rank order
        total = np.asarray(x, np.float64).copy() if total is None else total + np.asarray(x, np.float64)
    v = total
    if bias is not None:
        b = np.asarray(bias, np.float64)
        if b.ndim != 1 or b.shape[0] != v.shape[-1]:
            raise ValueError("bias must be 1-D over the last dimension")
        v = v + b
    if float(np.float32(p)) != 0.0:
        idx = np.arange(v.size, dtype=np.uint64) if index is None else np.asarray(index, np.uint64).ravel()
        keep = keep_mask(seed, p, idx).reshape(v.shape)
        v = np.where(keep, v * dropout_scale(p), 0.0)
    if residual is not None:
        v = v + np.asarray(residual, np.float64)
    return v
