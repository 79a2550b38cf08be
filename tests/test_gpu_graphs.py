"""The enqueue entry points inside a CUDA graph.

One graph captures every kind of launch the library makes: the CTA-pair GEMM
(with programmatic dependent launch), the GEMM on unaligned operands (pack
kernels into a stream-ordered workspace), stream-K (flag reset + cooperative
launch), split-K over a thread-block cluster (clusters of 2 to 16, the largest
with the non-portable size attribute), the dynamic tile order (cluster launch
control), the CUDA-core GEMV,
the tensor-core skinny GEMM, the FP8 GEMM and split-KV decode attention
(workspace + the merge kernel as a programmatic dependent).  The graph is
replayed on new input contents, written in place between replays: every
output must equal the eager calls' bit for bit, and the integer-valued GEMM /
GEMV outputs must equal the oracle's.
"""
import math

import numpy as np
import pytest

import oracle
from bf16_gemm_skinny_gb300 import _native as bsk
from bf16_gemm_skinny_gb300 import build as bsk_build
from bf16_gemm_skinny_gb300 import inputs
from helpers import from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    bsk_build.build()
    oracle.build()
    torch.cuda.init()
    yield bsk.load()
    for k in bsk.OPTIONS:
        bsk.set_option(k, 0)


class Problem:
    """Device buffers of every call; refill(seed) rewrites the inputs in place."""

    GEMM = (512, 384, 1024)        # CTA pairs, aligned
    RAGGED = (300, 517, 200)       # unaligned leading dimensions: pack path
    SK = (1000, 777, 1030)         # stream-K forced
    DYN = (1000, 777, 1030)        # dynamic tile order forced
    SPLITK = (128, 128, 4096)      # one tile, 64 k-blocks: split-K over a cluster (automatic, and 16 forced)
    GEMV = (1000, 1024)            # M, K; n = 1 (CUDA cores) and n = 8 (tensor cores)
    FP8 = (256, 160, 384)
    ATTN = dict(nqh=16, nkv=4, hd=256, bs=784, L=1500)

    def __init__(self):
        import torch

        M, N, K = self.GEMM
        self.gA, self.gB = self._pair(M * K, N * K)
        self.gC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
        M, N, K = self.RAGGED
        self.rA, self.rB = self._pair(M * K, N * K)
        self.rC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
        M, N, K = self.SK
        self.sA, self.sB = self._pair(M * K, N * K)
        self.sC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
        self.dC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
        M, N, K = self.SPLITK
        self.kA, self.kB = self._pair(M * K, N * K)
        self.kC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
        self.k16C = torch.zeros(M * N, dtype=torch.int16, device="cuda")
        M, K = self.GEMV
        self.W = torch.zeros(M * K, dtype=torch.int16, device="cuda")
        self.x1 = torch.zeros(K, dtype=torch.int16, device="cuda")
        self.x8 = torch.zeros(8 * K, dtype=torch.int16, device="cuda")
        self.y1 = torch.zeros(M, dtype=torch.int16, device="cuda")
        self.y8 = torch.zeros(8 * M, dtype=torch.int16, device="cuda")
        M, N, K = self.FP8
        self.f8A = torch.zeros(M * K, dtype=torch.uint8, device="cuda")
        self.f8B = torch.zeros(N * K, dtype=torch.uint8, device="cuda")
        self.f8C = torch.zeros(M * N, dtype=torch.int32, device="cuda")
        a = self.ATTN
        nb = -(-a["L"] // a["bs"])
        self.nb = nb
        n_cache = nb * a["bs"] * a["nkv"] * a["hd"]
        self.k = torch.zeros(n_cache, dtype=torch.int16, device="cuda")
        self.v = torch.zeros(n_cache, dtype=torch.int16, device="cuda")
        self.q = torch.zeros(a["nqh"] * a["hd"], dtype=torch.int16, device="cuda")
        self.bt = torch.from_numpy(np.arange(nb, dtype=np.int32)[::-1].copy()).cuda()
        self.sl = torch.tensor([a["L"]], dtype=torch.int32, device="cuda")
        self.o = torch.zeros(a["nqh"] * a["hd"], dtype=torch.int16, device="cuda")

    @staticmethod
    def _pair(na, nb):
        import torch

        return (torch.zeros(na, dtype=torch.int16, device="cuda"), torch.zeros(nb, dtype=torch.int16, device="cuda"))

    def refill(self, seed):
        """Integer-valued GEMM / GEMV / FP8 inputs, normal BF16 attention inputs."""
        import torch

        def put(t, bits):
            t.copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16 if t.dtype == torch.int16
                                                                     else np.uint8)))

        for (M, N, K), A, B, s in ((self.GEMM, self.gA, self.gB, 0), (self.RAGGED, self.rA, self.rB, 2),
                                   (self.SK, self.sA, self.sB, 4), (self.SPLITK, self.kA, self.kB, 13)):
            a, b = inputs.gemm_operands(M, N, K, "int2", seed + s, seed + s + 1)
            put(A, a)
            put(B, b)
        M, K = self.GEMV
        W, x8 = inputs.linear_operands(M, K, 8, "int2", "int2", seed_x=seed + 6, seed_w=seed + 7)
        put(self.W, W)
        put(self.x8, x8)
        put(self.x1, x8[:K])
        M, N, K = self.FP8
        a8, b8 = inputs.fp8_operands(M, N, K, "int2", "e4m3", seed + 8, seed + 9)
        put(self.f8A, a8)
        put(self.f8B, b8)
        n = self.k.numel()
        put(self.k, inputs.to_bf16_bits(inputs.draw("normal1", n, seed + 10)))
        put(self.v, inputs.to_bf16_bits(inputs.draw("normal1", n, seed + 11)))
        put(self.q, inputs.to_bf16_bits(inputs.draw("normal1", self.q.numel(), seed + 12)))
        torch.cuda.synchronize()

    def enqueue_all(self):
        """Every call, asynchronously, on torch's current stream."""
        M, N, K = self.GEMM
        bsk.gemm_f16_colmajor_enqueue(self.gA, self.gB, self.gC, M, N, K)
        M, N, K = self.RAGGED
        bsk.gemm_f16_enqueue(bsk.COL_MAJOR, 0, 0, self.rA, M, self.rB, K, self.rC, M, M, N, K)
        M, N, K = self.SK
        bsk.set_option("stream_k", 2)
        try:
            bsk.gemm_f16_colmajor_enqueue(self.sA, self.sB, self.sC, M, N, K)
        finally:
            bsk.set_option("stream_k", 0)
        bsk.set_option("tile_sched", 2)
        try:
            bsk.gemm_f16_colmajor_enqueue(self.sA, self.sB, self.dC, M, N, K)
        finally:
            bsk.set_option("tile_sched", 0)
        M, N, K = self.SPLITK
        bsk.gemm_f16_colmajor_enqueue(self.kA, self.kB, self.kC, M, N, K)
        bsk.set_option("split_k", 16)
        try:
            bsk.gemm_f16_colmajor_enqueue(self.kA, self.kB, self.k16C, M, N, K)
        finally:
            bsk.set_option("split_k", 0)
        M, K = self.GEMV
        bsk.gemv_bf16_enqueue(self.W, self.x1, self.y1, M, K, 1)
        bsk.gemv_bf16_enqueue(self.W, self.x8, self.y8, M, K, 8)
        M, N, K = self.FP8
        bsk.gemm_fp8_enqueue(bsk.FP8_E4M3, self.f8A, K, self.f8B, K, self.f8C, M, bsk.OUT_F32, M, N, K, 0.5)
        a = self.ATTN
        bsk.decode_attention_bf16_enqueue(self.q, self.k, self.v, self.bt, self.sl, self.o, 1, a["nqh"], a["nkv"],
                                          a["hd"], a["bs"], self.nb, self.nb, a["L"], 1.0 / math.sqrt(a["hd"]), 0)

    def outputs(self):
        return [from_dev(t) for t in (self.gC, self.rC, self.sC, self.dC, self.y1, self.y8, self.o)] + \
            [self.f8C.cpu().numpy().view(np.uint32)] + [from_dev(t) for t in (self.kC, self.k16C)]


def check_integer_outputs(prob, outs):
    """The integer-valued calls against the oracle (host copies of the inputs)."""
    M, N, K = prob.GEMM
    _, want = oracle.gemm_f16_colmajor(from_dev(prob.gA), from_dev(prob.gB), M, N, K)
    assert np.array_equal(outs[0], want), "GEMM"
    M, N, K = prob.RAGGED
    _, want = oracle.gemm_f16_colmajor(from_dev(prob.rA), from_dev(prob.rB), M, N, K)
    assert np.array_equal(outs[1], want), "ragged GEMM"
    M, N, K = prob.SK
    _, want = oracle.gemm_f16_colmajor(from_dev(prob.sA), from_dev(prob.sB), M, N, K)
    assert np.array_equal(outs[2], want), "stream-K GEMM"
    assert np.array_equal(outs[3], want), "dynamic-order GEMM"
    M, K = prob.GEMV
    W = from_dev(prob.W)
    _, want1 = oracle.linear_bf16(W, from_dev(prob.x1), M, K, 1)
    _, want8 = oracle.linear_bf16(W, from_dev(prob.x8), M, K, 8)
    assert np.array_equal(outs[4], want1.reshape(-1)), "GEMV n = 1"
    assert np.array_equal(outs[5], want8.reshape(-1)), "GEMV n = 8"
    M, N, K = prob.FP8
    _, want = oracle.gemm_fp8(prob.f8A.cpu().numpy(), prob.f8B.cpu().numpy(), M, N, K, K, K, "e4m3", 0.5, "f32")
    assert np.array_equal(outs[7], want), "FP8 GEMM"
    M, N, K = prob.SPLITK
    _, want = oracle.gemm_f16_colmajor(from_dev(prob.kA), from_dev(prob.kB), M, N, K)
    assert np.array_equal(outs[8], want), "split-K GEMM (automatic plan)"
    assert np.array_equal(outs[9], want), "split-K GEMM (cluster of 16)"


def test_graph_replay_matches_eager_calls():
    import torch

    prob = Problem()
    prob.refill(100)
    # eager run first: also makes every one-time set-up (shared-memory opt-in,
    # occupancy queries, the status word) happen outside the capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        prob.enqueue_all()
        bsk.stream_check(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager_first = prob.outputs()
    check_integer_outputs(prob, eager_first)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        prob.enqueue_all()

    for seed in (200, 300):
        prob.refill(seed)
        for t in (prob.gC, prob.rC, prob.sC, prob.dC, prob.y1, prob.y8, prob.o, prob.f8C, prob.kC, prob.k16C):
            t.fill_(0x5A5A)
        graph.replay()
        torch.cuda.synchronize()
        bsk.stream_check()
        replayed = prob.outputs()
        check_integer_outputs(prob, replayed)
        # the same inputs through eager calls: identical bits
        prob.enqueue_all()
        bsk.stream_check()
        eager = prob.outputs()
        for i, (r, e) in enumerate(zip(replayed, eager)):
            assert np.array_equal(r, e), f"output {i} differs between graph replay and eager call"
        assert not any(np.array_equal(r, f) for r, f in zip(replayed[6:7], eager_first[6:7])), \
            "attention output did not change with its inputs"
