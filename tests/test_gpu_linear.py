"""GPU-vs-oracle parity of the head's linear-layer engine (weight-streaming GEMV for few rows, tcgen05
GEMM above eight rows) through the C ABI entry point eagle3_linear."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def head():
    from eagle_speculative_decoding_eagle3_gb300 import build
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    build.build()
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048, target_vocab=8192,
                    draft_vocab=4096, batch=4, ctx=(64, 64), seed=90)
    h = HN.DeviceHead(w, WL.make_weights(w))
    yield h
    h.close()


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 24, 64, 200, 256, 300])
@pytest.mark.parametrize("N,K", [(448, 1088), (2112, 1024), (2112, 14336)])
def test_linear_matches_oracle(head, M, N, K):
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    x = WL.f32_to_bf16_bits(WL.normal((M, K), 1.0, 5, f"lin.x.{M}.{K}"))
    w = WL.f32_to_bf16_bits(WL.normal((N, K), 0.02, 5, f"lin.w.{N}.{K}"))
    xd, wd = HN.to_device(x), HN.to_device(w)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    E.eagle3_linear(head.handle, xd, wd, y, M, N, K)
    torch.cuda.synchronize()
    assert head.error_word() == 0
    ref = O.linear(WL.bf16_to_f32(x), WL.bf16_to_f32(w))
    err = row_rel_err(y.cpu().numpy(), ref)      # per row: ||g - o||_inf / ||o||_inf
    assert err < 1e-5, err


@pytest.mark.parametrize("M", [2048, 2100])
def test_linear_pair_tiles_match_oracle(head, M):
    # enough 256 x 256 tiles that the tensor-core engine pairs two 128-row weight tiles per CTA; the
    # last pair has a partial first tile and an empty second one, and M ends inside a token tile
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    N, K = 10048, 1024
    x = WL.f32_to_bf16_bits(WL.normal((M, K), 1.0, 6, f"linp.x.{M}"))
    w = WL.f32_to_bf16_bits(WL.normal((N, K), 0.02, 6, "linp.w"))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    E.eagle3_linear(head.handle, HN.to_device(x), HN.to_device(w), y, M, N, K)
    torch.cuda.synchronize()
    assert head.error_word() == 0
    ref = O.linear(WL.bf16_to_f32(x), WL.bf16_to_f32(w))
    err = row_rel_err(y.cpu().numpy(), ref)      # per row: ||g - o||_inf / ||o||_inf
    assert err < 1e-5, err
