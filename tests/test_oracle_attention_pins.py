"""Pins for the decode-attention oracle (DCU decode-GEMV article, sections 6.1
and 7: out = softmax(scale * q K^T) V per query head over a paged KV cache,
query head h reading KV head h / (num_q_heads / num_kv_heads)).

Closed forms and invariants that a slip in the oracle would break: one token
(output = that V row), zero scale (output = mean of the V rows, exact
rational), a known two-token weight ratio, a dominant token, huge scores
(no overflow: the maximum is subtracted), block-table permutation, the GQA
head mapping, batching, empty sequences and out-of-range blocks."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf16(vals):
    t = torch.tensor(np.asarray(vals, np.float64).reshape(-1), dtype=torch.float64).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def dec(bits):
    return oracle.bf16_decode(np.asarray(bits, np.uint16))


def make_cache(rng, num_blocks, block_size, nkv, hd, dist=1.0):
    k = bf16(rng.standard_normal((num_blocks, block_size, nkv, hd)) * dist)
    v = bf16(rng.standard_normal((num_blocks, block_size, nkv, hd)))
    return k.reshape(num_blocks, block_size, nkv, hd), v.reshape(num_blocks, block_size, nkv, hd)


def run(q, k, v, bt, sl, nqh, nkv, hd, bs, scale):
    return oracle.decode_attention_bf16(q, k, v, bt, sl, nqh, nkv, hd, bs, scale)


def test_single_token_returns_its_value_row(oracle_mod):
    rng = np.random.default_rng(1)
    nqh, nkv, hd, bs = 4, 2, 16, 3
    k, v = make_cache(rng, 2, bs, nkv, hd)
    q = bf16(rng.standard_normal((1, nqh, hd)))
    bt = np.array([[1, 0]], np.int32)            # logical block 0 is physical block 1
    ref, out = run(q, k, v, bt, [1], nqh, nkv, hd, bs, 0.3)
    for h in range(nqh):
        g = h // (nqh // nkv)
        assert np.array_equal(out[0, h], v[1, 0, g])


def test_zero_scale_gives_the_exact_mean(oracle_mod):
    rng = np.random.default_rng(2)
    nqh, nkv, hd, bs, L = 2, 1, 8, 4, 7
    k, v = make_cache(rng, 2, bs, nkv, hd)
    q = bf16(rng.standard_normal((1, nqh, hd)))
    bt = np.array([[0, 1]], np.int32)
    ref, out = run(q, k, v, bt, [L], nqh, nkv, hd, bs, 0.0)
    vals = dec(v.reshape(-1)).reshape(2 * bs, nkv, hd)
    for e in range(hd):
        mean = sum((Fraction(float(vals[t, 0, e])) for t in range(L)), Fraction(0)) / L
        assert ref[0, 0, e] == pytest.approx(float(mean), rel=1e-15, abs=1e-300)
        assert out[0, 0, e] == bf16([float(mean)])[0]


def test_two_tokens_with_known_weights(oracle_mod):
    """Scores differing by ln 3 weight the two V rows 1/4 and 3/4."""
    nqh, nkv, hd, bs = 1, 1, 4, 2
    q = bf16([[[1.0, 0.0, 0.0, 0.0]]])
    k = bf16([[[[0.0, 5.0, 0.0, 0.0]], [[2.0, -1.0, 0.0, 0.0]]]]).reshape(1, bs, nkv, hd)
    v = bf16([[[[1.0, 2.0, -4.0, 0.5]], [[5.0, -2.0, 8.0, 0.25]]]]).reshape(1, bs, nkv, hd)
    ref, _ = run(q, k, v, np.array([[0]], np.int32), [2], nqh, nkv, hd, bs, math.log(3.0) / 2.0)
    want = (np.array([1.0, 2.0, -4.0, 0.5]) + 3 * np.array([5.0, -2.0, 8.0, 0.25])) / 4
    assert np.allclose(ref[0, 0], want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("big", [60.0, 5000.0])
def test_dominant_token_and_no_overflow(oracle_mod, big):
    """One score far above the rest: the output is that token's V row.  With
    scores in the thousands exp() would overflow without the max subtraction."""
    rng = np.random.default_rng(3)
    nqh, nkv, hd, bs, L = 1, 1, 8, 5, 5
    q = bf16([[[1.0] + [0.0] * (hd - 1)]])
    kk = np.zeros((1, bs, nkv, hd))
    kk[0, 3, 0, 0] = big
    kk[0, :, 0, 1:] = rng.standard_normal((bs, hd - 1))
    k = bf16(kk).reshape(1, bs, nkv, hd)
    v = bf16(rng.standard_normal((1, bs, nkv, hd))).reshape(1, bs, nkv, hd)
    ref, out = run(q, k, v, np.array([[0]], np.int32), [L], nqh, nkv, hd, bs, 1.0)
    assert np.all(np.isfinite(ref))
    assert np.array_equal(out[0, 0], v[0, 3, 0])


def test_block_table_permutation_invariance(oracle_mod):
    rng = np.random.default_rng(4)
    nqh, nkv, hd, bs, nb = 4, 2, 16, 3, 6
    k, v = make_cache(rng, nb, bs, nkv, hd)
    q = bf16(rng.standard_normal((1, nqh, hd)))
    L = 16
    bt = np.arange(nb, dtype=np.int32)[None, :]
    _, out = run(q, k, v, bt, [L], nqh, nkv, hd, bs, 0.25)
    perm = rng.permutation(nb)                     # physical block p holds old block perm[p]
    k2, v2 = k[perm], v[perm]
    inv = np.argsort(perm).astype(np.int32)
    _, out2 = run(q, k2, v2, inv[None, :], [L], nqh, nkv, hd, bs, 0.25)
    assert np.array_equal(out, out2)


def test_gqa_mapping_matches_replicated_kv_heads(oracle_mod):
    """4 query heads over 2 KV heads == 4 query heads over 4 KV heads where KV head j
    holds a copy of the original KV head j // 2."""
    rng = np.random.default_rng(5)
    nqh, nkv, hd, bs, nb, L = 4, 2, 8, 4, 3, 10
    k, v = make_cache(rng, nb, bs, nkv, hd)
    q = bf16(rng.standard_normal((1, nqh, hd)))
    bt = np.arange(nb, dtype=np.int32)[None, :]
    _, out = run(q, k, v, bt, [L], nqh, nkv, hd, bs, 0.5)
    k4 = np.repeat(k, 2, axis=2)
    v4 = np.repeat(v, 2, axis=2)
    _, out4 = run(q, k4, v4, bt, [L], nqh, 4, hd, bs, 0.5)
    assert np.array_equal(out, out4)


def test_batch_equals_separate_sequences(oracle_mod):
    rng = np.random.default_rng(6)
    nqh, nkv, hd, bs, nb = 2, 1, 8, 4, 8
    k, v = make_cache(rng, nb, bs, nkv, hd)
    q = bf16(rng.standard_normal((2, nqh, hd))).reshape(2, nqh, hd)
    bt = np.array([[5, 2, 7, 0], [1, 3, 0, 0]], np.int32)
    sl = [13, 6]
    _, out = run(q, k, v, bt, sl, nqh, nkv, hd, bs, 0.7)
    for s in range(2):
        _, one = run(q[s:s + 1], k, v, bt[s:s + 1], [sl[s]], nqh, nkv, hd, bs, 0.7)
        assert np.array_equal(out[s], one[0])


def test_empty_sequence_gives_zeros_and_bad_block_raises(oracle_mod):
    rng = np.random.default_rng(7)
    k, v = make_cache(rng, 2, 4, 1, 8)
    q = bf16(rng.standard_normal((1, 1, 8)))
    ref, out = run(q, k, v, np.array([[0, 1]], np.int32), [0], 1, 1, 8, 4, 1.0)
    assert np.all(ref == 0) and np.all(out == 0)
    with pytest.raises(RuntimeError):
        run(q, k, v, np.array([[0, 9]], np.int32), [6], 1, 1, 8, 4, 1.0)
