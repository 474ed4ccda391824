"""The configuration the bench times, checked against the oracle.

bench.py runs each layer of the 7B-like sweep as:
  * decode: the seven N = 1 MUL_MATs (q, k, v, o 4096 x 4096; gate, up
    11008 x 4096; down 4096 x 11008) captured in one CUDA graph, with
    GQ_OPT_WEIGHTS_STATIC and GQ_OPT_X_STATIC set and programmatic dependent
    launch, so consecutive launches overlap;
  * prefill: eagerly, the layer's four activations (one buffer) converted
    to bf16 by one gq_f32_to_bf16 call, then the seven tensor-core MUL_MATs on them
    (gq_mul_mat_q4_0_bf16x) at N = 512, the first without the x-static
    promise and the other six with it.
These tests build one layer from the bench's own input recipe, run it the same
way, and compare with the oracle: every decode output over two graph replays,
and sampled rows (all 512 tokens) of every prefill output.
"""
import numpy as np
import pytest

import bench
import oracle
from gpu_util import assert_mul_mat_close, cores, oracle_mul_mat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None


def _with_options(opts, fn):
    old = {k: gq.gq_get_option(k) for k in opts}
    try:
        for k, v in opts.items():
            gq.gq_set_option(k, v)
        return fn()
    finally:
        for k, v in old.items():
            gq.gq_set_option(k, v)


def _layer(N, tag):
    order, _ = bench.layer_inputs()
    host_w = bench.make_weights(1, 0)
    acts = bench.make_acts(1, N, 0, tag)[0]
    return order, host_w, acts


def test_decode_layer_graph_with_static_promises():
    order, host_w, acts = _layer(bench.DECODE_N, 0)
    W = [torch.from_numpy(w).cuda() for _, _, w in host_w]
    X = [torch.from_numpy(a).cuda() for a in acts]
    Y = [torch.full((1, M), float("nan"), device="cuda") for M, _, _ in host_w]
    s = torch.cuda.Stream()

    def run():
        def layer():
            for j, (M, K, _) in enumerate(host_w):
                gq.gq_mul_mat_q4_0(W[j], M, K, X[order[j]], 1, Y[j], stream=s)
        with torch.cuda.stream(s):
            layer()  # eager once (first calls set kernel attributes outside the capture)
        torch.cuda.synchronize()
        for y in Y:
            y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                layer()
        outs = []
        for _ in range(2):
            for y in Y:
                y.fill_(float("nan"))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            gq.gq_sync_status(s)
            outs.append([y.cpu().numpy() for y in Y])
        return outs
    outs = _with_options({gq.GQ_OPT_WEIGHTS_STATIC: 1, gq.GQ_OPT_X_STATIC: 1}, run)
    for j, (M, K, w) in enumerate(host_w):
        y_ref, s_ref = oracle_mul_mat(w, M, K, acts[order[j]])
        for rep, ys in enumerate(outs):
            assert_mul_mat_close(ys[j], y_ref, s_ref, f"decode graph replay {rep} matrix {j} ({M}x{K})")
        assert np.array_equal(outs[0][j], outs[1][j]), f"matrix {j}: replays differ"


def test_prefill_layer_eager_bf16_chain():
    N = bench.PREFILL_N
    order, host_w, acts = _layer(N, 1)
    W = [torch.from_numpy(w).cuda() for _, _, w in host_w]
    # the layer's activations in one buffer, converted by one call, as the bench does
    Xflat = torch.from_numpy(np.concatenate([a.ravel() for a in acts])).cuda()
    Xbflat = torch.empty(Xflat.numel(), dtype=torch.int16, device="cuda")
    Xb, off = [], 0
    for a in acts:
        Xb.append(Xbflat[off:off + a.size].view(a.shape))
        off += a.size
    Y = [torch.full((N, M), float("nan"), device="cuda") for M, _, _ in host_w]
    s = torch.cuda.Stream()

    def run():
        with torch.cuda.stream(s):
            for _ in range(2):  # twice: the second layer's conversion overwrites X while the first's calls may run
                gq.gq_f32_to_bf16(Xflat, Xbflat, Xflat.numel(), stream=s)
                for j, (M, K, _) in enumerate(host_w):
                    # as the bench: the first call without the x-static promise, the others with it
                    gq.gq_set_option(gq.GQ_OPT_X_STATIC, 1 if j > 0 else 0)
                    gq.gq_mul_mat_q4_0_bf16x(W[j], M, K, Xb[order[j]], N, Y[j], stream=s)
        torch.cuda.synchronize()
        gq.gq_sync_status(s)
        return [y.cpu().numpy() for y in Y]
    ys = _with_options({gq.GQ_OPT_WEIGHTS_STATIC: 1, gq.GQ_OPT_X_STATIC: 1}, run)
    rng = np.random.default_rng(0x51A5)
    orc = oracle.get()
    for j, (M, K, w) in enumerate(host_w):
        rows = np.sort(rng.choice(M, size=48, replace=False))
        # the sampled rows against the oracle on those rows' blocks (all 512 tokens)
        y_ref, s_ref = orc.mul_mat(np.ascontiguousarray(w[rows]), len(rows), K, acts[order[j]], nthreads=cores())
        assert_mul_mat_close(ys[j][:, rows], y_ref, s_ref, f"prefill matrix {j} ({M}x{K}) sampled rows")
