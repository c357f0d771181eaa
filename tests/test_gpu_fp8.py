"""FP8 E4M3 draft weights ("EAGLE head deep dive", deployment: the drafter's post-training quantization
to FP8) through the C ABI: the device quantizer against the oracle's per-row rule (bit-exact codes and
scales), and whole drafting rounds of FP8 heads against the oracle running on its own quantization of
the same weights (the bf16 tolerances: the FP8 kernels widen the codes exactly and accumulate in fp32)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL

from parity import TOL_BF16, check_round, run_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from eagle_speculative_decoding_eagle3_gb300 import build
    build.build()


def _quantize_on_gpu(W, dtype):
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    t = HN.to_device(WL.f32_to_bf16_bits(W) if dtype == "bf16" else W.astype(np.float32))
    codes = torch.full(W.shape, 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((W.shape[0],), -1.0, dtype=torch.float32, device="cuda")
    E.eagle3_quantize_e4m3(t, E.BF16 if dtype == "bf16" else E.F32, W.shape[0], W.shape[1], codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("N,K,dtype", [(5, 40, "f32"), (37, 7168, "bf16"), (3, 1001, "f32"), (300, 2048, "bf16"),
                                       (64, 18432, "bf16")])
def test_quantize_e4m3_bit_exact(N, K, dtype):
    W = WL.normal((N, K), 0.02, 11, f"fp8.q.{N}.{K}").astype(np.float32)
    if dtype == "bf16":
        W = WL.bf16_to_f32(WL.f32_to_bf16_bits(W))
    W[min(2, N - 1)] = 0.0                                     # an all-zero row: scale 1, zero codes
    if N >= 5 and K >= 40:
        # a row whose maximum is 448 (scale 1): exact midpoints between codes round to the even code,
        # and signed zeros and values below half the smallest subnormal keep their sign
        W[0, :10] = [448.0, 1.0625, 1.1875, -1.0625, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -10, 0.4375, 300.0]
        W[0, 10:] = 0.5
    codes, scales = _quantize_on_gpu(W, dtype)
    ref_codes, ref_scales, _ = O.quantize_rows_e4m3(W)
    np.testing.assert_array_equal(scales.view(np.uint32), ref_scales.view(np.uint32))
    np.testing.assert_array_equal(codes, ref_codes)


def _narrow(**kw):
    base = dict(hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048, target_vocab=8192, draft_vocab=4096)
    base.update(kw)
    return WL.workload("dsv3_b1", **base)


def test_fp8_round_gemv_and_tensor_core_extend():
    # 3 sequences x 3 new rows: the extend (9 rows) expands the FP8 matrices to bf16 for the tensor-core
    # GEMM; the decode steps (3 rows) stream the E4M3 codes through the GEMV kernels
    w = _narrow(batch=3, ctx=(100, 700), t_new=3, gamma=4, accept_p=(0.7,) * 4, seed=83)
    gpu, orc, seqs, paged = run_round(w, fp8=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_fp8_round_all_gemv():
    # 2 sequences x 3 new rows: every call, the extend's fc over the bf16 aux states included, stays
    # on the FP8 GEMV path
    w = _narrow(batch=2, ctx=(40, 300), t_new=3, gamma=3, accept_p=(0.7,) * 3, seed=84)
    gpu, orc, seqs, paged = run_round(w, fp8=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_fp8_round_tensor_core_decode():
    # 24 sequences: every decode step (24 rows) also takes the expanded tensor-core path
    w = _narrow(batch=24, ctx=(30, 700), t_new=2, gamma=3, accept_p=(0.7,) * 3, seed=85)
    gpu, orc, seqs, paged = run_round(w, fp8=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_fp8_dsv3_b1_full_size_round():
    # the batch-1 DeepseekV3-shaped workload at full size with FP8 projection matrices, as the
    # benchmark's FP8 mode runs it
    w = WL.workload("dsv3_b1")
    gpu, orc, seqs, paged = run_round(w, fp8=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


# ---------------------------------------------------------------- NVFP4
def _quantize_nvfp4_on_gpu(W, dtype):
    from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E
    from eagle_speculative_decoding_eagle3_gb300 import harness as HN
    t = HN.to_device(WL.f32_to_bf16_bits(W) if dtype == "bf16" else W.astype(np.float32))
    N, K = W.shape
    codes = torch.full((N, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
    block = torch.full((N, K // 16), 0xCD, dtype=torch.uint8, device="cuda")
    g = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    E.eagle3_quantize_nvfp4(t, E.BF16 if dtype == "bf16" else E.F32, N, K, codes, block, g)
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    unpacked = np.empty((N, K), dtype=np.uint8)
    unpacked[:, 0::2] = c & 0xF                      # the even element in the low nibble
    unpacked[:, 1::2] = c >> 4
    return unpacked, block.cpu().numpy(), g.cpu().numpy()


@pytest.mark.parametrize("N,K,dtype", [(5, 64, "f32"), (37, 7168, "bf16"), (300, 2048, "bf16"), (64, 18432, "bf16")])
def test_quantize_nvfp4_bit_exact(N, K, dtype):
    W = WL.normal((N, K), 0.02, 12, f"fp4.q.{N}.{K}").astype(np.float32)
    if dtype == "bf16":
        W = WL.bf16_to_f32(WL.f32_to_bf16_bits(W))
    W[min(2, N - 1), 16:32] = 0.0                              # an all-zero block
    W[0, :16] = np.float32(2.0 ** -40)                         # a block whose E4M3 scale underflows to 0
    if N >= 5:
        # matrix maximum 2688 makes g = 1; a block with maximum 6 then has scale code E4M3(1) and e_b = 1,
        # so its values are the exact E2M1 midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 (both signs),
        # which must round to the even code
        W[3, 0] = np.float32(2688.0)
        W[4, 32:48] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, 0],
                               dtype=np.float32)
    codes, block, g = _quantize_nvfp4_on_gpu(W, dtype)
    ref_codes, ref_block, ref_g, _ = O.quantize_nvfp4(W)
    assert np.float32(g[0]).view(np.uint32) == np.float32(ref_g).view(np.uint32)
    np.testing.assert_array_equal(block, ref_block)
    np.testing.assert_array_equal(codes, ref_codes)


def test_nvfp4_round_gemv_and_tensor_core_extend():
    w = _narrow(batch=3, ctx=(100, 700), t_new=3, gamma=4, accept_p=(0.7,) * 4, seed=86)
    gpu, orc, seqs, paged = run_round(w, nvfp4=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_nvfp4_round_all_gemv():
    w = _narrow(batch=2, ctx=(40, 300), t_new=3, gamma=3, accept_p=(0.7,) * 3, seed=87)
    gpu, orc, seqs, paged = run_round(w, nvfp4=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_nvfp4_round_tensor_core_decode():
    w = _narrow(batch=24, ctx=(30, 700), t_new=2, gamma=3, accept_p=(0.7,) * 3, seed=88)
    gpu, orc, seqs, paged = run_round(w, seqs=[0, 11, 23], nvfp4=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_nvfp4_dsv3_b1_full_size_round():
    w = WL.workload("dsv3_b1")
    gpu, orc, seqs, paged = run_round(w, nvfp4=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))
