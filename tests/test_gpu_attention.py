"""GPU parity of decode_attention_bf16 (split-KV decode attention over a paged
BF16 cache) against the oracle, through the C ABI.

Tolerance, derived from FP32 arithmetic on BF16 inputs: a score is a sum of
head_dim exact products formed by the tensor cores, whose FP32 additions need
not round to nearest, so it carries at most head_dim * 2^-23 * scale *
sum|q_e k_e| of accumulation error (one ulp per addition), plus 2^-21 for the
hardware exp2; that perturbs each softmax weight by that much relatively; the
output, a weighted mean of V rows, then moves by at most twice that times
max|v|, plus the FP32 accumulation over the tokens and one BF16 rounding:
    |out - exact| <= (2 * eps_w + n_tok * 2^-24) * max|v| + ulp_bf16 / 2,
with eps_w the worst weight error over the tokens of the call.
"""
import math

import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import BF16_NAN, CANARY, from_dev, poisoned, to_dev, ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()


def make_problem(seed, num_seqs, seq_lens, nqh, nkv, hd, bs, extra_blocks=3):
    """Random paged cache with shuffled physical blocks (draws via inputs.draw)."""
    rng = np.random.default_rng(seed)
    blocks_per_seq = [max(1, -(-L // bs)) for L in seq_lens]
    max_blocks = max(blocks_per_seq)
    num_blocks = sum(blocks_per_seq) + extra_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.zeros((num_seqs, max_blocks), np.int32)
    pos = 0
    for s, nb in enumerate(blocks_per_seq):
        bt[s, :nb] = perm[pos:pos + nb]
        pos += nb
    n_cache = num_blocks * bs * nkv * hd
    k = inputs.to_bf16_bits(inputs.draw("normal1", n_cache, seed + 100))
    v = inputs.to_bf16_bits(inputs.draw("normal1", n_cache, seed + 200))
    q = inputs.to_bf16_bits(inputs.draw("normal1", num_seqs * nqh * hd, seed + 300))
    return q, k, v, bt, np.asarray(seq_lens, np.int32), num_blocks, max_blocks


def run(q, k, v, bt, sl, nqh, nkv, hd, bs, num_blocks, max_blocks, scale, segments=0, max_seq_len=None):
    import torch

    num_seqs = sl.size
    max_seq_len = int(sl.max()) if max_seq_len is None else max_seq_len
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    btd = torch.from_numpy(bt.reshape(-1).copy()).cuda()
    sld = torch.from_numpy(sl.copy()).cuda()
    buf, out = poisoned(num_seqs * nqh * hd, BF16_NAN)
    bsk.decode_attention_bf16(qd, kd, vd, btd, sld, out, num_seqs, nqh, nkv, hd, bs, max_blocks, num_blocks,
                              max_seq_len, scale, segments)
    torch.cuda.synchronize()
    assert np.all(from_dev(buf[num_seqs * nqh * hd:]) == CANARY)
    assert np.array_equal(from_dev(kd), k) and np.array_equal(from_dev(vd), v)
    return from_dev(out).reshape(num_seqs, nqh, hd)


def check(got, ref, q, k, v, hd, scale, n_tok, label):
    gv = oracle.bf16_decode(got.reshape(-1))
    rv = ref.reshape(-1)
    assert np.all(np.isfinite(gv)), label
    qv = np.abs(oracle.bf16_decode(q))
    kv = np.abs(oracle.bf16_decode(k))
    vmax = float(np.max(np.abs(oracle.bf16_decode(v))))
    # worst |scale * sum q_e k_e| bound: head_dim * max|q| * max|k| * scale
    sum_abs = hd * float(qv.max()) * float(kv.max()) * abs(scale)
    eps_w = hd * 2.0 ** -23 * sum_abs + 2.0 ** -21          # tensor-core sums; + the hardware exp2
    bound = (2 * eps_w + n_tok * 2.0 ** -24) * vmax + 0.5 * ulp(np.maximum(np.abs(gv), np.abs(rv)), "bf16")
    err = np.abs(gv - rv)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), f"{label}: err {err[worst]:.3g} > bound {bound[worst]:.3g}"
    rn = oracle.bf16_decode(oracle.bf16_encode(rv))
    flips = float(np.mean(gv != rn))
    assert flips < 0.05, f"{label}: {flips:.1%} of outputs differ from the correctly rounded result"
    return float(err.max()), float(err.mean())


PAGE = dict(nqh=16, nkv=4, hd=256, bs=784)


@pytest.mark.parametrize("L", [1, 5, 783, 784, 785, 3000, 8192, 12288, 16384, 32768])
def test_page_configuration(L):
    """16 query heads over 4 KV heads, head_dim 256, 784-token pages, one sequence."""
    nqh, nkv, hd, bs = PAGE["nqh"], PAGE["nkv"], PAGE["hd"], PAGE["bs"]
    q, k, v, bt, sl, nb, mb = make_problem(L, 1, [L], nqh, nkv, hd, bs)
    scale = 1.0 / math.sqrt(hd)
    got = run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale)
    ref, _ = oracle.decode_attention_bf16(q, k.reshape(nb, bs, nkv, hd), v.reshape(nb, bs, nkv, hd), bt, sl,
                                          nqh, nkv, hd, bs, scale)
    check(got, ref, q, k, v, hd, scale, L, f"L={L}")


@pytest.mark.parametrize("hd,nqh,nkv", [(64, 8, 8), (128, 8, 4), (128, 16, 2), (256, 8, 1), (64, 32, 4)])
@pytest.mark.parametrize("segments", [0, 1, 7, 64])
def test_head_shapes_and_segment_counts(hd, nqh, nkv, segments):
    bs = 32
    seq_lens = [1000, 1, 333]
    q, k, v, bt, sl, nb, mb = make_problem(hd + nqh + segments, 3, seq_lens, nqh, nkv, hd, bs)
    scale = 0.5 / math.sqrt(hd)
    got = run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale, segments)
    ref, _ = oracle.decode_attention_bf16(q, k.reshape(nb, bs, nkv, hd), v.reshape(nb, bs, nkv, hd), bt, sl,
                                          nqh, nkv, hd, bs, scale)
    check(got, ref, q, k, v, hd, scale, max(seq_lens), f"hd={hd} {nqh}/{nkv} segs={segments}")


def test_sixteen_and_thirty_two_segments_agree():
    """The page's cross-check of the two segmentations (section 7): outputs finite,
    max |difference| <= 2.44e-4 and mean |difference| <= 1.58e-5 (here on N(0,1) data)."""
    nqh, nkv, hd, bs, L = PAGE["nqh"], PAGE["nkv"], PAGE["hd"], PAGE["bs"], 16384
    q, k, v, bt, sl, nb, mb = make_problem(77, 1, [L], nqh, nkv, hd, bs)
    scale = 1.0 / math.sqrt(hd)
    a = oracle.bf16_decode(run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale, 16).reshape(-1))
    b = oracle.bf16_decode(run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale, 32).reshape(-1))
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b))
    d = np.abs(a - b)
    assert d.max() <= 2.44e-4 and d.mean() <= 1.58e-5, (d.max(), d.mean())


def test_batch_with_empty_sequence_and_determinism():
    nqh, nkv, hd, bs = 8, 2, 128, 16
    seq_lens = [0, 50, 1, 700]
    q, k, v, bt, sl, nb, mb = make_problem(9, 4, seq_lens, nqh, nkv, hd, bs)
    scale = 1.0 / math.sqrt(hd)
    got = run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale)
    assert np.all(got[0] == 0)
    ref, _ = oracle.decode_attention_bf16(q, k.reshape(nb, bs, nkv, hd), v.reshape(nb, bs, nkv, hd), bt, sl,
                                          nqh, nkv, hd, bs, scale)
    check(got, ref, q, k, v, hd, scale, 700, "batch")
    assert np.array_equal(run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale), got)


def test_out_of_range_block_is_reported_not_read():
    nqh, nkv, hd, bs = 4, 1, 64, 8
    q, k, v, bt, sl, nb, mb = make_problem(11, 1, [20], nqh, nkv, hd, bs)
    bt = bt.copy()
    bt[0, 1] = nb + 1000
    with pytest.raises(bsk.BskError) as exc:
        run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, 0.125)
    assert exc.value.status == 1
    # the library keeps working
    test_batch_with_empty_sequence_and_determinism()


def _random_configs(count, seed):
    """Seeded attention problems: head_dim, query heads per KV head, page size,
    batch, per-sequence lengths (some empty) and segment counts at random."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        hd = int(rng.choice([64, 128, 256]))
        group = int(rng.choice([1, 2, 4, 8]))
        nkv = int(rng.choice([1, 2, 4]))
        bs = int(rng.choice([8, 16, 31, 64, 784]))
        num_seqs = int(rng.integers(1, 4))
        lens = [int(v) for v in np.exp(rng.uniform(0, np.log(6000), num_seqs)).astype(int)]
        if rng.random() < 0.2:
            lens[0] = 0
        segs = int(rng.choice([0, 0, 1, 5, 16, 32, 100]))
        out.append((hd, group * nkv, nkv, bs, lens, segs, int(rng.integers(0, 1 << 20))))
    return out


@pytest.mark.parametrize("hd,nqh,nkv,bs,lens,segs,seed", _random_configs(24, 1234))
def test_random_configurations(hd, nqh, nkv, bs, lens, segs, seed):
    """Random head shapes, page sizes, batches with uneven (and empty) sequences
    and segment counts: within the derived tolerance of the oracle, empty
    sequences give zeros."""
    q, k, v, bt, sl, nb, mb = make_problem(seed, len(lens), lens, nqh, nkv, hd, bs)
    scale = 1.0 / math.sqrt(hd)
    got = run(q, k, v, bt, sl, nqh, nkv, hd, bs, nb, mb, scale, segs)
    ref, _ = oracle.decode_attention_bf16(q, k.reshape(nb, bs, nkv, hd), v.reshape(nb, bs, nkv, hd), bt, sl,
                                          nqh, nkv, hd, bs, scale)
    for s, L in enumerate(lens):
        if L == 0:
            assert np.all(got[s] == 0)
    check(got, ref, q, k, v, hd, scale, max(max(lens), 1), f"hd={hd} {nqh}/{nkv} bs={bs} lens={lens} segs={segs}")
