"""mp_gemm inside a captured CUDA graph: replays equal the direct calls bit for
bit and match the fp64 oracle, across the plan kinds (one-CTA and swapped
tiles, CTA pairs, split-K on chip and through L2, unaligned operands that are
repacked), and a replay after new inputs are copied in computes on them."""
import pytest
import torch

import micro_polymerization_gb300 as mp
from micro_polymerization_gb300 import workloads as wl

from gpu_util import assert_parity

pytestmark = pytest.mark.gpu

SHAPES = [
    (2048, 2304, 768, 0.0),    # one-CTA tiles, one wave
    (4096, 4096, 1024, 0.0),   # several waves (CTA pairs where the model picks them)
    (105, 1024, 12544, 1.0),   # skinny: split-K
    (824, 768, 3072, 0.5),     # split-K on chip
    (9, 1000, 700, 0.5),       # swapped tiles
    (333, 101, 77, 0.5),       # rows not 16-byte aligned: repacked
]


def test_graph_replay_equals_direct_calls_and_oracle():
    dev = torch.device("cuda", 0)
    h = mp.mp_init(0)
    s = torch.cuda.Stream(device=dev)
    try:
        probs = []
        for i, (M, N, K, beta) in enumerate(SHAPES):
            g = wl.Gemm(M, N, K, alpha=1.5, beta=beta, seed=900 + i)
            A, B, C = wl.make_operands(g)
            probs.append((g, A, B, C, A.to(dev), B.to(dev), C.to(dev) if C is not None else None,
                          torch.empty(M, N, device=dev)))

        def calls():
            for g, _, _, _, Ad, Bd, Cd, Dd in probs:
                mp.mp_gemm(h, Ad, Bd, Cd, Dd, g.alpha, g.beta, stream=s)

        with torch.cuda.stream(s):
            calls()
        torch.cuda.synchronize()
        direct = [p[7].clone() for p in probs]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            calls()
        for p in probs:
            p[7].fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert mp.mp_check(h) == mp.MP_OK
        for (g, A, B, C, _, _, _, Dd), ref in zip(probs, direct):
            assert torch.equal(Dd, ref), f"replay differs from the direct call {(g.M, g.N, g.K)}"
            assert_parity(Dd.cpu(), A, B, C, g.alpha, g.beta, what=f"graph replay {(g.M, g.N, g.K)}")
        # New inputs in the same buffers: the replay computes on them.
        for i, (g, A, B, C, Ad, Bd, Cd, Dd) in enumerate(probs):
            g2 = wl.Gemm(g.M, g.N, g.K, alpha=g.alpha, beta=g.beta, seed=950 + i)
            A2, B2, C2 = wl.make_operands(g2)
            Ad.copy_(A2)
            Bd.copy_(B2)
            if Cd is not None:
                Cd.copy_(C2)
            probs[i] = (g, A2, B2, C2, Ad, Bd, Cd, Dd)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert mp.mp_check(h) == mp.MP_OK
        for g, A, B, C, _, _, _, Dd in probs:
            assert_parity(Dd.cpu(), A, B, C, g.alpha, g.beta, what=f"second replay {(g.M, g.N, g.K)}")
    finally:
        h.close()
