"""Sampled drafts (eagle3_sample) and residual acceptance (eagle3_accept_residual) against the oracle.

Tokens are compared exactly, except where the oracle's own decision moves when u or top_p is nudged by
1e-4: the GPU sums its fp32 weights in another order, so a draw within rounding of a CDF boundary may
land on either neighbour (the same rule as the near-tie rule of the argmax)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu
EPS = 1e-4


def _logits(seed, rows, V):
    rng = np.random.default_rng(seed)
    l = rng.normal(0.0, 2.0, size=(rows, V)).astype(np.float32)
    l[:, 7] = l[:, 3]                                   # exact ties
    l[0, :16] = l[0, 16:32]
    return l


def _allowed(l, T, k, p, u):
    out = set()
    for du in (-EPS, 0.0, EPS):
        for dp in ((-EPS, 0.0, EPS) if p < 1.0 else (0.0,)):
            out.add(O.sample_filtered(l, T, k, min(1.0, p + dp), min(max(u + du, 0.0), 1.0 - 1e-9))[0])
    return out


CASES = [(0.0, 0, 1.0), (0.7, 0, 1.0), (1.0, 50, 1.0), (0.8, 1024, 0.9), (1.3, 20, 0.5), (1.0, 1, 1.0)]


@pytest.mark.parametrize("V", [4096, 32000])
@pytest.mark.parametrize("T,k,p", CASES)
def test_sample_matches_oracle(V, T, k, p):
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    rows = 6
    l = _logits(V + k, rows, V)
    u = np.random.default_rng(V * 3 + k).random(rows).astype(np.float32)
    w = WL.workload("dsv3_b1", draft_vocab=V)
    d2t = WL.make_d2t(w).astype(np.int32)
    Vt = w.target_vocab
    tok = torch.zeros(rows, dtype=torch.int32, device="cuda")
    tp = torch.zeros(rows, dtype=torch.float32, device="cuda")
    probs = torch.full((rows, Vt), -1.0, dtype=torch.float32, device="cuda")
    E.eagle3_sample(torch.from_numpy(l).cuda(), rows, V, V, T, k, p, torch.from_numpy(u).cuda(),
                    torch.from_numpy(d2t).cuda(), Vt, tok, tp, probs, Vt, True)
    torch.cuda.synchronize()
    tok, tp, probs = tok.cpu().numpy(), tp.cpu().numpy(), probs.cpu().numpy()
    for r in range(rows):
        t_o, pr_o = O.sample_filtered(l[r], T, k, p, float(u[r]))
        g = int(tok[r])
        if g != t_o + d2t[t_o]:
            allowed = {a + int(d2t[a]) for a in _allowed(l[r], T, k, p, float(u[r]))}
            assert g in allowed, (r, g, t_o)
            continue
        # same token: its probability and the whole final distribution (mapped to target ids) agree
        assert abs(tp[r] - pr_o[t_o]) <= 1e-4 * max(pr_o[t_o], 1e-3), (r, tp[r], pr_o[t_o])
        keep_same = p >= 1.0 or len({tuple(np.flatnonzero(O.sample_filtered(l[r], T, k, q, 0.5)[1]))
                                     for q in (p - EPS, p, min(1.0, p + EPS))}) == 1
        if keep_same:
            want = np.zeros(Vt)
            want[np.arange(V) + d2t] = pr_o
            np.testing.assert_allclose(probs[r], want, atol=2e-6, rtol=1e-4)


def test_accept_residual_matches_oracle():
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    rng = np.random.default_rng(21)
    B, G, V = 24, 4, 777
    # draft distributions: sparse (top-k-like supports), target distributions: dense
    q = np.zeros((B, G, V), np.float32)
    for b in range(B):
        for i in range(G):
            sup = rng.choice(V, size=12, replace=False)
            q[b, i, sup] = rng.dirichlet(np.ones(12))
    p = rng.dirichlet(np.ones(V) * 0.3, size=(B, G + 1)).astype(np.float32)
    p[:3, :G] = q[:3]                                   # rows whose target equals the draft
    p[3, 0] = 0.0                                       # a row whose first target distribution is empty
    p[3, 0, 5] = 1.0
    draft = np.zeros((B, G), np.int32)
    for b in range(B):
        for i in range(G):
            draft[b, i] = rng.choice(V, p=q[b, i] / q[b, i].sum())
    ua = rng.random((B, G)).astype(np.float32)
    ur = rng.random((B, G)).astype(np.float32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    hist = torch.full((G + 1,), -1, dtype=torch.int32, device="cuda")
    E.eagle3_accept_residual(dev(draft), dev(q), dev(p), dev(ua), dev(ur), B, G, V, acc, nxt, hist)
    torch.cuda.synchronize()
    acc, nxt, hist = acc.cpu().numpy(), nxt.cpu().numpy(), hist.cpu().numpy()
    o_acc, o_nxt, o_hist = O.accept_residual(draft, q, p, ua, ur)
    np.testing.assert_array_equal(acc, o_acc)
    np.testing.assert_array_equal(hist, o_hist)
    assert np.all(acc[:3] == G)
    for b in range(B):
        if nxt[b] == o_nxt[b]:
            continue
        near = set()
        for du in (-1e-5, 1e-5):
            u2 = ur.copy()
            k = o_acc[b]
            u2[b, min(k, G - 1)] = np.clip(u2[b, min(k, G - 1)] + du, 0.0, 1.0 - 1e-9)
            near.add(int(O.accept_residual(draft[b:b + 1], q[b:b + 1], p[b:b + 1], ua[b:b + 1], u2[b:b + 1])[1][0]))
        assert nxt[b] in near, (b, nxt[b], o_nxt[b])


@pytest.mark.parametrize("k", [5, 50, 1000])
def test_sample_top_k_boundary_on_ties(k):
    # integer-valued logits: the top_k boundary falls inside a group of equal values, where the lower
    # indices must be the ones kept
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    rows, V = 4, 4096
    rng = np.random.default_rng(k)
    l = np.round(rng.normal(0.0, 1.5, size=(rows, V))).astype(np.float32)
    u = rng.random(rows).astype(np.float32)
    tok = torch.zeros(rows, dtype=torch.int32, device="cuda")
    probs = torch.zeros((rows, V), dtype=torch.float32, device="cuda")
    E.eagle3_sample(torch.from_numpy(l).cuda(), rows, V, V, 1.0, k, 1.0, torch.from_numpy(u).cuda(), None, 0, tok,
                    None, probs, V, False)
    torch.cuda.synchronize()
    tok, probs = tok.cpu().numpy(), probs.cpu().numpy()
    for r in range(rows):
        t_o, pr_o = O.sample_filtered(l[r], 1.0, k, 1.0, float(u[r]))
        np.testing.assert_array_equal(probs[r] > 0, pr_o > 0)      # the same kept set, ties included
        if tok[r] != t_o:
            assert tok[r] in _allowed(l[r], 1.0, k, 1.0, float(u[r])), (r, tok[r], t_o)


@pytest.mark.parametrize("seed,offset,n", [(0, 0, 1), (7, 0, 10001), (0xDEADBEEFCAFEBABE, 12345, 4099),
                                           (3, (1 << 64) - 3, 33)])
def test_philox_uniforms_match_oracle(seed, offset, n):
    # bit-exact against the oracle's statement of the stream; the last case carries into counter word 1
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    out = torch.full((n + 5,), -1.0, dtype=torch.float32, device="cuda")
    E.eagle3_philox_uniforms(seed, offset, n, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got[:n].astype(np.float64), O.philox_uniforms(seed, offset, n))
    assert np.all(got[n:] == -1.0)                     # nothing past n is written


def _typical_case(seed, B, G, V, conc):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(V) * conc, size=(B, G)).astype(np.float32)
    best = np.argmax(p, axis=2)
    draft = np.where(rng.random((B, G)) < 0.7, best, rng.integers(0, V, size=(B, G)))
    draft[0, :] = best[0, :]                          # a row that accepts through its whole length
    draft[1, 0] = V + 5                               # an id outside the vocabulary
    return draft.astype(np.int32), p


@pytest.mark.parametrize("B,G,V,conc,eps,dlt", [(37, 5, 777, 0.3, 0.09, 0.3), (9, 7, 32000, 0.05, 0.09, 0.3),
                                                (64, 3, 129, 2.0, 0.3, 0.9), (5, 2, 1000, 0.01, 0.0, 0.0)])
def test_accept_typical_matches_oracle(B, G, V, conc, eps, dlt):
    # the entropy is an fp32 sum on the GPU and an fp64 one in the oracle: where a probability sits within
    # 1e-4 (relative) of its threshold either decision is accepted, i.e. the GPU length lies between the
    # oracle's lengths with both thresholds scaled by 1 + 1e-4 and by 1 - 1e-4
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    draft, p = _typical_case(B * 7 + V, B, G, V, conc)
    acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    hist = torch.full((G + 1,), -1, dtype=torch.int32, device="cuda")
    E.eagle3_accept_typical(torch.from_numpy(draft).cuda(), torch.from_numpy(p).cuda(), B, G, V, eps, dlt, acc, hist)
    torch.cuda.synchronize()
    acc, hist = acc.cpu().numpy(), hist.cpu().numpy()
    want, _ = O.accept_typical(draft, p, np.float32(eps), np.float32(dlt))
    lo, _ = O.accept_typical(draft, p, np.float32(eps) * (1 + 1e-4), np.float32(dlt) * (1 + 1e-4))
    hi, _ = O.accept_typical(draft, p, np.float32(eps) * (1 - 1e-4), np.float32(dlt) * (1 - 1e-4))
    assert np.all((acc >= lo) & (acc <= hi)), (acc, want)
    assert np.mean(acc == want) >= 0.9
    np.testing.assert_array_equal(hist, np.bincount(acc, minlength=G + 1))
    assert acc[0] == want[0] and acc[1] == 0


@pytest.mark.parametrize("V", [5, 100, 8191, 129280])
@pytest.mark.parametrize("T,k,p", [(0.0, 0, 1.0), (0.9, 0, 1.0), (1.0, 50, 0.9), (0.6, 1024, 1.0)])
def test_sample_slices_without_d2t(V, T, k, p):
    # the row is split over the CTAs of a cluster: fewer tokens than CTAs (5), slices of 13 (100), a
    # ragged last slice (8191) and the full target vocabulary (129280); probabilities in draft ids
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    build.build()
    rows = 3
    l = _logits(V * 7 + k, rows, max(V, 32))[:, :V].copy()
    u = np.random.default_rng(V + 11).random(rows).astype(np.float32)
    u[0] = 0.0                                          # the first kept token
    tok = torch.zeros(rows, dtype=torch.int32, device="cuda")
    tp = torch.zeros(rows, dtype=torch.float32, device="cuda")
    probs = torch.full((rows, V), -1.0, dtype=torch.float32, device="cuda")
    E.eagle3_sample(torch.from_numpy(l).cuda(), rows, V, V, T, k, p, torch.from_numpy(u).cuda(), None, 0, tok,
                    tp, probs, V, False)
    torch.cuda.synchronize()
    tok, tp, probs = tok.cpu().numpy(), tp.cpu().numpy(), probs.cpu().numpy()
    for r in range(rows):
        t_o, pr_o = O.sample_filtered(l[r], T, k, p, float(u[r]))
        if tok[r] != t_o:
            assert tok[r] in _allowed(l[r], T, k, p, float(u[r])), (r, tok[r], t_o)
            continue
        assert abs(tp[r] - pr_o[t_o]) <= 1e-4 * max(pr_o[t_o], 1e-3), (r, tp[r], pr_o[t_o])
        keep_same = p >= 1.0 or len({tuple(np.flatnonzero(O.sample_filtered(l[r], T, k, q, 0.5)[1]))
                                     for q in (p - EPS, p, min(1.0, p + EPS))}) == 1
        if keep_same:
            np.testing.assert_allclose(probs[r], pr_o, atol=2e-6, rtol=1e-4)
