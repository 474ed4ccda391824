"""Row-data validation (gq_validate) on the GPU against the oracle.

Integer results, so the bar is equality: the number of blocks with a NaN or
infinite scale field and the first one's flat index.  Inputs: synth weights
with non-finite scale bit patterns planted at seeded positions.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import quantized_block_q4_gb300 as gq
else:  # collected on CPU machines, never run there (marked gpu)
    gq = None

TYPES = [0, 1, 2]
NAMES = {0: "q4_0", 1: "q4_1", 2: "q8_0"}
BAD_BITS = [0x7C00, 0xFC00, 0x7E00, 0x7C01, 0xFFFF]  # +inf, -inf, NaNs


def planted(qtype, M, K, seed, nbad, field=0):
    """Weights with nbad blocks whose scale field (0 = d, 2 = Q4_1's m) is
    set to a non-finite bit pattern; returns the raw bytes."""
    W = synth.typed_weights(qtype, M, K, seed)
    bb = gq.TYPE_BLOCK_BYTES[qtype]
    flat = W.reshape(-1, bb)
    rng = np.random.Generator(np.random.SFC64(seed + 7))
    picks = rng.choice(flat.shape[0], size=nbad, replace=False) if nbad else []
    for i, b in enumerate(picks):
        bits = BAD_BITS[i % len(BAD_BITS)]
        flat[b, field] = bits & 0xFF
        flat[b, field + 1] = bits >> 8
    return W


def gpu_validate(qtype, W, M, K, offset=0):
    if offset:
        buf = torch.zeros(W.size + 16, dtype=torch.uint8, device="cuda")
        buf[offset:offset + W.size] = torch.from_numpy(W.reshape(-1)).cuda()
        result = torch.empty(2, dtype=torch.int64, device="cuda")
        gq.gq_validate(qtype, buf.data_ptr() + offset, M, K, result)
        torch.cuda.synchronize()
        r = result.cpu().tolist()
        first = r[1] & 0xFFFFFFFFFFFFFFFF
        return r[0], (None if first == 0xFFFFFFFFFFFFFFFF else first)
    return gq.validate(qtype, torch.from_numpy(np.array(W, copy=True)).cuda(), K, M)


@pytest.mark.parametrize("qtype", TYPES, ids=lambda t: NAMES[t])
@pytest.mark.parametrize("M,K,nbad", [(256, 1024, 0), (256, 1024, 1), (300, 4096, 37), (7, 96, 3), (1, 32, 1),
                                      (4096, 4096, 500)])
def test_validate_matches_oracle(qtype, M, K, nbad):
    W = planted(qtype, M, K, 16000 + M + K + nbad + qtype, nbad)
    got = gpu_validate(qtype, W, M, K)
    assert got == oracle.get().validate(qtype, W, M, K)
    assert got[0] == nbad


def test_q4_1_min_field():
    M, K = 500, 2048
    W = planted(1, M, K, 16100, 9, field=2)
    assert gpu_validate(1, W, M, K) == oracle.get().validate(1, W, M, K) and gpu_validate(1, W, M, K)[0] == 9
    # the same bytes read as Q4_0 would be other blocks entirely: only the typed reading counts


@pytest.mark.parametrize("offset", [1, 3, 8])
def test_unaligned_weights(offset):
    M, K = 129, 288
    W = planted(0, M, K, 16200 + offset, 5)
    assert gpu_validate(0, W, M, K, offset) == oracle.get().validate(0, W, M, K)


def test_full_size_and_last_block():
    """A 14336 x 4096 matrix with one bad block, the very last one."""
    M, K = 14336, 4096
    W = synth.q4_0_weights(M, K, seed=16300)
    W.reshape(-1, 18)[-1, 1] = 0x7E
    count, first = gpu_validate(0, W, M, K)
    assert (count, first) == (1, M * K // 32 - 1) == oracle.get().validate(0, W, M, K)


def test_empty_and_result_reset():
    result = torch.full((2,), 5, dtype=torch.int64, device="cuda")
    gq.gq_validate_q4_0(None, 0, 64, result)
    torch.cuda.synchronize()
    assert result.cpu().tolist() == [0, -1]        # (0, UINT64_MAX)
    # a second call on clean weights resets a previous result
    W = torch.from_numpy(synth.q4_0_weights(64, 256, seed=16400)).cuda()
    result.fill_(9)
    gq.gq_validate_q4_0(W, 64, 256, result)
    torch.cuda.synchronize()
    assert result.cpu().tolist() == [0, -1]
