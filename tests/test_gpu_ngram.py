"""GPU n-gram pool (sv_ngram_pool_*) against the oracle's pool, bit-exact,
over streams of steps with duplicates, evictions, invalid tokens and invalid
lookups; and the pool feeding sv_verify_greedy on the greedy workload's
logits ("Lookahead Decoding 完全拆解", sections "N-gram 池与身份判定" and the
verify branch)."""
import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    svpkg.build()
    torch.cuda.set_device(0)
    yield


# (the insert stages a step's keys in shared memory when W <= 32, N <= 33,
# cap <= 32 and eight warps' stages fit 48 KB: the first four shapes; the
# others take the direct path)
@pytest.mark.parametrize("B,V,N,cap,G,W,keys", [(5, 40, 4, 3, 4, 6, 3), (3, 1000, 5, 7, 7, 7, 2),
                                                 (2, 9, 2, 1, 2, 3, 9), (33, 32000, 5, 7, 7, 7, 4),
                                                 (3, 60, 33, 32, 6, 32, 3),
                                                 (4, 100, 40, 5, 3, 4, 2), (3, 50, 3, 40, 5, 5, 2),
                                                 (2, 200, 4, 4, 4, 40, 3)])
def test_pool_matches_oracle(B, V, N, cap, G, W, keys):
    rng = np.random.default_rng(B * 1000 + N)
    ref = oracle.NgramPool(B, V, N, cap)
    pool = svpkg.NgramPool(B, V, N, cap)
    for step in range(40):
        g = rng.integers(0, V, size=(B, W, N)).astype(np.int32)
        g[:, :, 0] = rng.integers(0, keys, size=(B, W))
        # repeats of earlier n-grams, and invalid tokens now and then
        if step % 3 == 1:
            g[:, 1] = g[:, 0]
        if step % 7 == 3:
            g[0, 0, -1] = V
            g[-1, -1, 1] = -5
        ref.insert(g)
        pool.insert(g)
        last = rng.integers(0, keys, size=B).astype(np.int32)
        if step % 11 == 5:
            last[0] = V
        rc, rn = ref.lookup(last, G)
        gc, gn = pool.lookup(last, G)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(gn.cpu().numpy(), rn)
        np.testing.assert_array_equal(gc.cpu().numpy(), rc)
    assert svpkg.get_status() == 0


def test_pool_feeds_greedy_verify():
    """Candidates from the pool, verified greedily on logits of the greedy
    workload's shape: the library's pool + verify equal the oracle's pool +
    verify; half the inserted n-grams continue with the rows' argmaxes so
    that candidates match."""
    cfg = sg.CONFIGS["cfg4_greedy_v32000_bf16"]
    B, G, N, V = cfg.B, cfg.G, cfg.N, cfg.V
    d = sg.greedy_inputs(cfg)
    # every candidate slot of a sequence sees the same rows, so that an argmax
    # continuation matches wherever the pool places it
    d["logits"][:] = d["logits"][:, :1]
    logits = sg.to_float(d["logits"], cfg.dtype)
    rng = np.random.default_rng(5)
    last = rng.integers(0, V, size=B).astype(np.int32)
    grams = rng.integers(0, V, size=(B, 2 * G, N)).astype(np.int32)
    grams[:, :, 0] = last[:, None]
    am = np.argmax(logits[:, 0, :N - 1], axis=-1)  # [B, N-1]
    for b in range(B):
        for w in range(0, 2 * G, 2):  # every other n-gram continues with the argmaxes, for a random length
            k = 1 + (w // 2) % (N - 1)
            grams[b, w, 1:1 + k] = am[b, :k]
    ref = oracle.NgramPool(B, V, N, G)
    ref.insert(grams)
    pool = svpkg.NgramPool(B, V, N, G)
    pool.insert(grams)
    rc, rn = ref.lookup(last, G)
    gc, gn = pool.lookup(last, G)
    ot, oa, _ = oracle.verify_greedy(d["logits"], rc)
    tt, ta = svpkg.verify_greedy(to_dev(d["logits"]), gc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gc.cpu().numpy(), rc)
    np.testing.assert_array_equal(ta.cpu().numpy(), oa)
    np.testing.assert_array_equal(tt.cpu().numpy(), ot)
    assert (oa > 0).any()


def test_pool_argument_errors():
    lib = svpkg.lib()
    assert lib.sv_ngram_pool_bytes(2, 10, 1, 3) == -1
    assert lib.sv_ngram_pool_bytes(2, 10, 3, 0) == -1
    assert lib.sv_ngram_pool_bytes(2, 10, 3, 2) == 256 + 2 * 10 * 2 * 2 * 4
    x = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = svpkg._ptr(x)
    assert lib.sv_ngram_pool_insert(None, 2, 10, 3, 2, p, 1, None) == -1
    assert lib.sv_ngram_pool_lookup(p, 2, 10, 3, 2, p, 0, p, p, None) == -1
    assert lib.sv_ngram_pool_insert(p, 0, 10, 3, 2, None, 1, None) == 0
