"""Chains of calls in which each call's output is the next call's activations,
issued back to back on one stream and as one captured CUDA graph.

Every kernel is launched with programmatic dependent launch and reads its
packed weights before the kernel ahead of it has completed; activations, outputs
and split-K workspaces wait for it. So a chained call must see the output its
predecessor wrote, and a workspace shared by consecutive split-K calls must not
be overwritten while the previous reduce still reads it. Each chained run is
compared bit for bit with the same calls separated by device synchronisations
(outputs are filled with NaN before every run, so a read that came too early
shows), and the last layer meets the oracle bound on its GPU-produced input.
"""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu


def _affine_layer(N, K, seed):
    packed, s, b = oracle.quantize(synth.affine_weights(N, K, seed), 4, 64, "bf16")
    return (packed, s, b), (to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"))


def _bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _same(a, c):
    return torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                       c.view(torch.int32) if c.dtype == torch.float32 else c.view(torch.int16))


def _check_chain(run, outs, reps=3):
    """run(sync) issues the chain (with a device synchronisation after every
    call when sync is true). The chained results, eager and replayed from a
    graph, equal the synchronised ones bit for bit."""
    for o in outs:
        o.fill_(float("nan"))
    run(True)
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    for _ in range(reps):
        for o in outs:
            o.fill_(float("nan"))
        run(False)
        torch.cuda.synchronize()
        for i, (a, c) in enumerate(zip(ref, outs)):
            assert _same(a, c), f"eager chain: layer {i} differs from the synchronised run"
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(False)
    for _ in range(reps):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i, (a, c) in enumerate(zip(ref, outs)):
            assert _same(a, c), f"graph chain: layer {i} differs from the synchronised run"
    return ref


def test_qmv_chain():
    dims = [4096, 5120, 2048, 4096, 1024]   # x of 4096 -> 5120 -> 2048 -> 4096 -> 1024
    layers = [_affine_layer(dims[i + 1], dims[i], 100 + i) for i in range(len(dims) - 1)]
    x0 = to_dev(synth.activations(1, dims[0], "bf16", 7).reshape(-1), "bf16")
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in dims[1:]]

    def run(sync):
        x = x0
        for (_, (p, s, b)), o in zip(layers, outs):
            g4.gai4_qmv(p, s, b, x, out=o)
            if sync:
                torch.cuda.synchronize()
            x = o

    ref = _check_chain(run, outs)
    (packed, s, b), _ = layers[-1]
    want, absdot = oracle.qmm(packed, s, b, _bits16(ref[-2]), 4, 64, "bf16")
    assert_within(to_host_f64(ref[-1], "bf16"), want, absdot, "bf16", "qmv chain, last layer")


@pytest.mark.parametrize("split", [0, 2])
def test_qmm_t_chain_shared_workspace(split):
    """Tensor-core qmm_t layers (M = 24) with split-K partials in one
    workspace that every layer reuses."""
    M = 24
    dims = [2048, 4096, 1024, 2048]
    layers = [_affine_layer(dims[i + 1], dims[i], 200 + i) for i in range(len(dims) - 1)]
    assert all(g4.gai4_qmm_t_plan(M, dims[i + 1], dims[i], 4, 64, torch.bfloat16, split)[0] == 1
               for i in range(len(dims) - 1))
    nbytes = max(g4.gai4_qmm_t_workspace_bytes(M, dims[i + 1], dims[i], 4, 64, torch.bfloat16, split)
                 for i in range(len(dims) - 1))
    ws = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    x0 = to_dev(synth.activations(M, dims[0], "bf16", 9), "bf16")
    outs = [torch.empty((M, n), dtype=torch.bfloat16, device="cuda") for n in dims[1:]]

    def run(sync):
        x = x0
        for (_, (p, s, b)), o in zip(layers, outs):
            g4.gai4_qmm_t(p, s, b, x, out=o, split_k=split, workspace=ws)
            if sync:
                torch.cuda.synchronize()
            x = o

    ref = _check_chain(run, outs)
    (packed, s, b), _ = layers[-1]
    want, absdot = oracle.qmm(packed, s, b, _bits16(ref[-2]), 4, 64, "bf16")
    assert_within(to_host_f64(ref[-1], "bf16"), want, absdot, "bf16", f"qmm_t chain split={split}, last layer")


def test_block_gemv_chain():
    """binary32 chain through the Q4_K and Q8_0 GEMVs (TMA-staged kernels)."""
    layers = [("q4_k", 5120, 4096, synth.q4_k_blocks(5120, 4096, 31)),
              ("q8_0", 2048, 5120, synth.q8_0_blocks(2048, 5120, 32)),
              ("q4_k", 4096, 2048, synth.q4_k_blocks(4096, 2048, 33))]
    dev_blocks = [to_dev(blk) for _, _, _, blk in layers]
    x0 = to_dev(synth.f32_vector(4096, 34))
    outs = [torch.empty(n, dtype=torch.float32, device="cuda") for _, n, _, _ in layers]

    def run(sync):
        x = x0
        for (kind, _, _, _), blk, o in zip(layers, dev_blocks, outs):
            (g4.gai4_q4_k_gemv if kind == "q4_k" else g4.gai4_q8_0_gemv)(blk, x, out=o)
            if sync:
                torch.cuda.synchronize()
            x = o

    ref = _check_chain(run, outs)
    want, absdot = oracle.q4_k_gemv(layers[-1][3], ref[-2].cpu().numpy())
    assert_within(ref[-1].cpu().numpy().astype(np.float64), want, absdot, "f32", "block GEMV chain, last layer")
