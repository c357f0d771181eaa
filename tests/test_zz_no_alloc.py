"""eagle3_linear_noalloc against the existing handle-based entry point eagle3_linear, through the C ABI.

eagle3_linear_noalloc serves callers that cannot allocate device memory on their call path (a runtime
whose HBM is all promised to its own pool, or a loop that must not reach cudaMalloc / cudaFree): it keeps
its split-K scratch in a fixed array inside the library instead of a handle's workspace.

Named to be collected last: it must pass both alone in a fresh process (where its first call does the
per-device scratch lookup) and after every other GPU test has run in the same process.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu

TOL = 1e-5   # max |a - b| / max |b|: both sides accumulate the same bf16 products in fp32


@pytest.fixture(scope="module")
def head():
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    build.build()
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048, target_vocab=8192,
                    draft_vocab=4096, batch=4, ctx=(64, 64), seed=91)
    h = HN.DeviceHead(w, WL.make_weights(w))
    yield h
    h.close()


def _inputs(M, N, K, tag):
    x = WL.f32_to_bf16_bits(WL.normal((M, K), 1.0, 7, f"noalloc.x.{tag}.{M}.{K}"))
    w = WL.f32_to_bf16_bits(WL.normal((N, K), 0.02, 7, f"noalloc.w.{tag}.{N}.{K}"))
    return x, w


def _rel(a, b):
    a = a.double()
    b = b.double()
    return float((a - b).abs().max() / b.abs().max())


# (M, N, K): row counts in the existing entry's GEMV and tensor-core ranges, a K short enough for a
# single split (no scratch use), and M * N exactly at the scratch limit (two splits)
SHAPES = [(1, 2112, 1024), (8, 448, 1088), (24, 448, 1088), (200, 2112, 1024), (64, 256, 128),
          (256, 8192, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_noalloc_matches_linear_on_two_calls_in_a_row(head, M, N, K):
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    assert M * N <= E.NOALLOC_SCRATCH_BYTES // 8
    host = [_inputs(M, N, K, "a"), _inputs(M, N, K, "b")]
    dev = [(HN.to_device(x), HN.to_device(w)) for x, w in host]
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    # two calls back to back on one stream, with different operands, before any synchronisation: the
    # second reuses the scratch the first left behind
    for (xd, wd), y in zip(dev, ys):
        E.eagle3_linear_noalloc(xd, wd, y, M, N, K)
    refs = []
    for xd, wd in dev:
        r = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        E.eagle3_linear(head.handle, xd, wd, r, M, N, K)
        refs.append(r)
    torch.cuda.synchronize()
    assert head.error_word() == 0
    for y, r in zip(ys, refs):
        assert bool(torch.isfinite(y).all())
        err = _rel(y.cpu(), r.cpu())
        assert err < TOL, (M, N, K, err)
    # the first result against the oracle's fp64 product as well
    x, w = host[0]
    ref = O.linear(WL.bf16_to_f32(x), WL.bf16_to_f32(w))
    got = ys[0].cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() / np.abs(ref).max() < TOL


def test_noalloc_rejects_sizes_beyond_its_scratch(head):
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    limit = E.NOALLOC_SCRATCH_BYTES // 8
    M, N, K = 257, 8192, 256          # M * N = limit + 8192
    assert M * N > limit
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(E.Eagle3Error) as ei:
        E.eagle3_linear_noalloc(x, w, y, M, N, K)
    assert ei.value.status == E.ERR_SCRATCH_LIMIT
    with pytest.raises(E.Eagle3Error) as ei:
        E.eagle3_linear_noalloc(x, w, y, 4, N, 200)   # K not a multiple of 64
    assert ei.value.status == E.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((y == 0).all())
