"""How much rounding the 8-bit decode's code offset adds to the scores.

"kv-cache-by-model", section 1: an 8-bit cache keeps one-byte codes c with
one fp16 scale per 32 values.  The decode kernel turns a stored K byte
(c + 128) into the fp16 value 1152 + c with one byte permutation and does not
subtract the offset: each score product starts its fp32 accumulator from
-1152 x (the query row's sum over the group).  The result is exact up to the
rounding of the fp32 sums, whose terms are now up to 1279 |q| instead of
127 |q| (the V codes still enter without the offset).

This test models every m16n8k16 accumulation pessimistically (products exact,
each addition rounded toward zero to fp32, in sequence, so that the errors
add up instead of cancelling) and checks
  (a) that the modelled error of both forms stays inside the a-priori bound:
      the sum over a chain's additions of u x (its start + the sum of its
      terms' magnitudes), u = 2^-23;
  (b) that on the decode configurations' value distribution (standard normal
      queries and K, quantised as the cache write does, head_dim 128, scale
      1/sqrt(128)) the modelled offset error changes a softmax weight by less
      than a tenth of the fp16 rounding the kernel applies to every weight
      anyway (2^-11), and at its largest by less than a fiftieth of what
      the 8-bit quantisation itself changes in a typical score.
The GPU tests compare the kernel itself with the oracle on the full-size
configurations.
"""
import math

import numpy as np

U = 2.0 ** -23            # unit roundoff of fp32 with truncation
OFFSET = 1152.0
SCALE_LOG2 = math.log2(math.e) / math.sqrt(128)


def _rz32(x):
    """x (float64) rounded toward zero to fp32, as float64."""
    f = x.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    f[over] = np.nextafter(f[over], np.float32(0))
    return f.astype(np.float64)


def _accumulate(c, terms):
    """c + terms[..., 0] + terms[..., 1] + ..., every partial sum truncated."""
    acc = _rz32(np.asarray(c, np.float64))
    for k in range(terms.shape[-1]):
        acc = _rz32(acc + terms[..., k])
    return acc


def _fp16(x):
    return x.astype(np.float16).astype(np.float64)


def _group_scores(q, c):
    """Exact, plain and offset-form scores of 32-dimension groups (last axis):
    two k-16 products each; the offset form starts from the query sum taken by
    the same kind of products with an all -1152 operand."""
    exact = np.sum(q * c, axis=-1)
    plain = _accumulate(_accumulate(0.0, q[..., :16] * c[..., :16]), q[..., 16:] * c[..., 16:])
    cq = _accumulate(_accumulate(0.0, -OFFSET * q[..., :16]), -OFFSET * q[..., 16:])
    b = OFFSET + c
    off = _accumulate(_accumulate(cq, q[..., :16] * b[..., :16]), q[..., 16:] * b[..., 16:])
    return exact, plain, off


def test_modelled_errors_within_a_priori_bounds():
    rng = np.random.default_rng(5)
    q = _fp16(rng.standard_normal((20000, 32)))
    c = rng.integers(-127, 128, size=(20000, 32)).astype(np.float64)
    # adversarial rows: magnitudes near the prescaled limit 2^15, codes +-127,
    # query sums that cancel
    qa = _fp16(rng.uniform(2.0 ** 14, 2.0 ** 15, (2000, 32)) * rng.choice([-1, 1], (2000, 32)))
    qa[:1000, 16:] = -qa[:1000, :16]
    ca = np.where(rng.random((2000, 32)) < 0.5, 127.0, -127.0)
    for qq, cc in ((q, c), (qa, ca)):
        exact, plain, off = _group_scores(qq, cc)
        s1 = np.sum(np.abs(qq), axis=-1)
        # the query-sum chains (32 terms of 1152 |q|), then the score chains
        # starting from their result (32 terms of up to 1279 |q|)
        bound_off = 32 * U * (OFFSET + OFFSET + OFFSET + 127) * s1
        bound_plain = 32 * U * 127 * s1
        assert np.all(np.abs(off - exact) <= bound_off)
        assert np.all(np.abs(plain - exact) <= bound_plain)
        assert np.any(off != exact)            # the model does round


def test_offset_error_small_against_weight_rounding_and_quantisation():
    rng = np.random.default_rng(7)
    n = 20000
    q = _fp16(rng.standard_normal((n, 4, 32)))
    k = rng.standard_normal((n, 4, 32)).astype(np.float32)
    # the cache write's absmax quantiser: scale = fp16(max |x| / 127), code =
    # round-half-even(x / scale)
    ks = _fp16(np.max(np.abs(k), axis=-1) / 127)
    c = np.clip(np.rint(k / ks[..., None].astype(np.float32)), -127, 127).astype(np.float64)
    exact, plain, off = _group_scores(q, c)
    # a score is sum over the 4 groups of ks x the group's product, times
    # scale x log2(e); a weight is 2^score
    d_off = SCALE_LOG2 * np.sum(ks * np.abs(off - exact), axis=-1)
    d_plain = SCALE_LOG2 * np.sum(ks * np.abs(plain - exact), axis=-1)
    rel_off = 2.0 ** d_off.max() - 1
    assert rel_off < 2.0 ** -11 / 10
    assert d_plain.max() <= d_off.max()
    # what the quantisation itself moves: scores over code x scale against the
    # scores over the original K
    d_quant = SCALE_LOG2 * np.abs(np.sum(q * (ks[..., None] * c - k), axis=(-1, -2)))
    assert d_off.max() < np.median(d_quant) / 50
