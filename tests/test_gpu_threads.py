"""Two host threads calling the library at the same time.

The library sets each kernel's launch attributes once per (kernel, device)
under a lock, so first calls may race between threads.  The check runs in a
fresh process (so that the first calls of every kernel happen inside the
threads): two threads start together behind a barrier, each runs the same
sequence of calls on its own stream -- the decode kernel at N = 1 and N = 4,
the tensor-core kernel at N = 64, Q8_0 MUL_MAT, dequant and MUL_MAT_ID -- and
every result is compared with the oracle.
"""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
import numpy as np
import torch
sys.path[:0] = [ROOT, ROOT + "/tests"]
import quantized_block_q4_gb300 as gq
import oracle, synth
from gpu_util import assert_mul_mat_close, oracle_mul_mat

torch.cuda.set_device(0)
torch.zeros(1, device="cuda")  # create the context before the threads start
cases = []
for i, (M, K, N) in enumerate([(700, 4096, 1), (500, 2048, 4), (640, 2048, 64)]):
    W = synth.q4_0_weights(M, K, seed=17000 + i)
    X = synth.activations(N, K, seed=17010 + i)
    cases.append(("q4_0", M, K, N, W, X, oracle_mul_mat(W, M, K, X)))
W8 = synth.typed_weights(2, 300, 2048, seed=17020)
X8 = synth.activations(1, 2048, seed=17021)
cases.append(("q8_0", 300, 2048, 1, W8, X8, oracle.get().mul_mat_typed(2, W8, 300, 2048, X8)))
E, Me, Ke, T, S = 4, 256, 1024, 1, 2
We = synth.moe_weights(E, Me, Ke, 17030)
Xe = synth.activations(T * S, Ke, 17031).reshape(T, S, Ke)
ids = synth.expert_ids(T, S, E, 17032)
ref_id = oracle.get().mul_mat_id(We, E, Me, Ke, Xe, ids)
Wdq = synth.q4_0_weights(200, 1024, seed=17040)
ref_dq = oracle.get().dequant(Wdq, 200, 1024)

barrier = threading.Barrier(2)
errors = []

def work(tid):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            dev = {}
            for c in cases:
                dev[id(c)] = (torch.from_numpy(c[4]).cuda(), torch.from_numpy(c[5]).cuda())
            wed, xed, idd = torch.from_numpy(We).cuda(), torch.from_numpy(Xe).cuda(), torch.from_numpy(ids).cuda()
            wdq = torch.from_numpy(Wdq).cuda()
            s.synchronize()
            barrier.wait()
            outs = []
            for c in cases:
                kind, M, K, N = c[:4]
                Wd, Xd = dev[id(c)]
                Y = torch.empty(N, M, device="cuda")
                if kind == "q4_0":
                    gq.gq_mul_mat_q4_0(Wd, M, K, Xd, N, Y, stream=s)
                else:
                    gq.gq_mul_mat(gq.GQ_TYPE_Q8_0, Wd, M, K, Xd, N, Y, stream=s)
                outs.append(Y)
            Yid = torch.empty(T, S, Me, device="cuda")
            gq.gq_mul_mat_id_q4_0(wed, E, Me, Ke, xed, S, idd, T, Yid, stream=s)
            Ydq = torch.empty(200, 1024, device="cuda")
            gq.gq_dequant_q4_0(wdq, 200, 1024, Ydq, stream=s)
            gq.gq_sync_status(s)
        for c, Y in zip(cases, outs):
            kind, M, K, N = c[:4]
            y_ref, s_ref = c[6]
            assert_mul_mat_close(Y.cpu().numpy(), y_ref, s_ref, f"thread {tid} {kind} M={M} K={K} N={N}")
        assert_mul_mat_close(Yid.cpu().numpy(), ref_id[0], ref_id[1], f"thread {tid} MUL_MAT_ID")
        if not np.array_equal(Ydq.cpu().numpy().view(np.uint32), ref_dq.view(np.uint32)):
            raise AssertionError(f"thread {tid}: dequant is not bit-exact")
    except Exception as e:  # reported by the parent
        errors.append(f"{type(e).__name__}: {e}")

ths = [threading.Thread(target=work, args=(i,)) for i in range(2)]
for t in ths: t.start()
for t in ths: t.join()
print("ERRORS" if errors else "OK")
for e in errors: print(e)
'''


def test_two_threads_first_calls_at_once():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    code = f"ROOT = {ROOT!r}\n" + SCRIPT
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[0] == "OK", r.stdout[-3000:]
