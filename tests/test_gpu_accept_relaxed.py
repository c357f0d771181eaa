"""eagle3_accept_relaxed (relaxed acceptance inside thinking blocks) against the oracle, bit-exact."""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu


def _case(seed, B, G, K, vocab, p_best=0.6):
    rng = np.random.default_rng(seed)
    ids = np.stack([np.stack([rng.choice(vocab, size=K, replace=False) for _ in range(G)]) for _ in range(B)])
    # descending log-probabilities with a few exact ties between neighbours
    gaps = rng.uniform(0.0, 0.5, size=(B, G, K)).astype(np.float32)
    gaps[rng.random((B, G, K)) < 0.1] = 0.0
    lp = (-np.cumsum(gaps, axis=2)).astype(np.float32)
    col = rng.integers(0, K, size=(B, G))
    draft = ids[np.arange(B)[:, None], np.arange(G)[None, :], col]
    draft = np.where(rng.random((B, G)) < p_best, ids[:, :, 0], draft)
    draft = np.where(rng.random((B, G)) < 0.05, vocab + 3, draft)      # a token outside every list
    think = rng.random(B) < 0.5
    return draft.astype(np.int32), ids.astype(np.int32), lp, think


@pytest.mark.parametrize("B,G,K,delta", [(1, 3, 10, 0.6), (37, 5, 10, 0.6), (300, 7, 4, 0.25), (64, 1, 1, 0.6),
                                         (257, 6, 16, 2.0), (9, 4, 10, 0.0)])
def test_accept_relaxed_matches_oracle(B, G, K, delta):
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    draft, ids, lp, think = _case(B * 131 + G * 7 + K, B, G, K, 50)
    for flags in (think, None):
        acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        hist = torch.full((G + 1,), -1, dtype=torch.int32, device="cuda")
        th = torch.from_numpy(flags.astype(np.uint8)).cuda() if flags is not None else None
        E.eagle3_accept_relaxed(torch.from_numpy(draft).cuda(), torch.from_numpy(ids).cuda(),
                                torch.from_numpy(lp).cuda(), th, B, G, K, delta, acc, hist)
        torch.cuda.synchronize()
        want, whist = O.accept_relaxed(draft, ids, lp, flags if flags is not None else np.zeros(B, bool), delta)
        np.testing.assert_array_equal(acc.cpu().numpy(), want)
        np.testing.assert_array_equal(hist.cpu().numpy(), whist)
