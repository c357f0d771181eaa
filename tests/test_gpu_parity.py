"""GPU-vs-oracle parity of whole drafting rounds (extend + gamma-1 decode steps + acceptance),
through the C ABI, on seeded inputs."""
import pytest

import workloads as WL

from parity import TOL_BF16, TOL_F32, check_round, run_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from eagle_speculative_decoding_eagle3_gb300 import build
    build.build()


def test_tiny_f32_round():
    w = WL.workload("tiny_f32")
    gpu, orc, seqs, paged = run_round(w)
    rep = check_round(w, gpu, orc, seqs, paged, TOL_F32)
    print(rep)


def test_tiny_f32_ragged_and_page_crossing():
    # ragged contexts, a page boundary inside the new rows, 5 sequences, longer round
    w = WL.workload("tiny_f32", batch=5, ctx=(1, 45), t_new=7, gamma=5, accept_p=(0.7,) * 5, seed=77)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32))


def test_tiny_f32_empty_cache_no_d2t():
    # extend from an empty cache (causal attention among the new rows only), identity vocab map
    w = WL.workload("tiny_f32", ctx=(0, 0), t_new=9, draft_vocab=2048, d2t=None, seed=78)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32))


def test_tiny_f32_single_split():
    # contexts short enough (max 28 slots) that attention runs one split and writes o_lat itself
    w = WL.workload("tiny_f32", batch=3, ctx=(3, 20), t_new=5, gamma=3, seed=80)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32))


def test_mla_shaped_bf16_round():
    # bf16 storage with the DeepseekV3 latent geometry (kv_lora 512, rope 64, nope 128, v 128) on a
    # narrow hidden size; several tiles of context with ragged lengths
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048,
                    target_vocab=8192, draft_vocab=4096, batch=3, ctx=(100, 700), t_new=3, gamma=4,
                    accept_p=(0.7,) * 4, seed=79)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


# 128 heads with the DeepseekV3 latent geometry: the tcgen05 latent attention (a CTA pair per row and
# split, scores split over K across the pair) on a narrow hidden size
MLA128 = dict(hidden=1024, n_heads=128, q_lora_rank=256, intermediate=2048, target_vocab=8192, draft_vocab=4096)


@pytest.mark.parametrize("over", [
    # GEMV decode (3 rows, mma.sync attention), tensor-core extend (18 rows, tcgen05 attention); ragged
    # contexts over several splits and pages
    dict(batch=3, ctx=(100, 700), t_new=6, gamma=4, accept_p=(0.7,) * 4, seed=85),
    # every call on the tensor-core path (24 and 48 rows)
    dict(batch=24, ctx=(30, 700), t_new=2, gamma=3, accept_p=(0.7,) * 3, seed=86),
    # contexts short enough for a single split (o_lat written by the attention kernel itself), 20 rows
    dict(batch=4, ctx=(3, 20), t_new=5, gamma=3, accept_p=(0.7,) * 3, seed=87),
    # extend on an empty cache: causal attention among the new rows only (18 rows)
    dict(batch=2, ctx=(0, 0), t_new=9, gamma=3, accept_p=(0.7,) * 3, seed=88),
    # one sequence: the decode steps divide 2300+ slots over 76 splits of one 32-slot tile (72 of them
    # live), merged with the value projection past the plain merge's 64 splits
    dict(batch=1, ctx=(2300, 2300), t_new=3, gamma=3, accept_p=(0.7,) * 3, seed=89),
])
def test_mla_128_heads_tensor_core_attention(over):
    w = WL.workload("dsv3_b1", **MLA128, **over)
    gpu, orc, seqs, paged = run_round(w, absorbed=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_dsv3_b1_full_size_round():
    # the batch-1 DeepseekV3-shaped workload at full size (4096-token cache, 32000-entry draft vocab
    # with d2t), as the benchmark runs it; the oracle follows the unabsorbed definition
    w = WL.workload("dsv3_b1")
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_mla_shaped_bf16_tensor_core_rounds():
    # 24 sequences: the extend (48 rows) and every decode step (24 rows) take the tcgen05 path
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048,
                    target_vocab=8192, draft_vocab=4096, batch=24, ctx=(30, 700), t_new=2, gamma=3,
                    accept_p=(0.7,) * 3, seed=80)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


@pytest.mark.parametrize("batch", [6, 24])
def test_persistent_lm_head_ragged_vocabulary(batch):
    # a 20,100-entry draft vocabulary: 157 full 128-row weight tiles and a ragged one, more tiles than SMs,
    # so the lm_head's argmax runs on the persistent tcgen05 GEMM (at 6 rows per decode step too)
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048,
                    target_vocab=40000, draft_vocab=20100, batch=batch, ctx=(30, 300), t_new=2, gamma=3,
                    accept_p=(0.7,) * 3, seed=90 + batch)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_dsv3_extend_rows_tensor_core():
    # full DeepseekV3 head dimensions, 2 sequences x 256 new rows on an empty cache (causal extend)
    w = WL.workload("dsv3_extend", batch=2, t_new=256, gamma=2, accept_p=(0.7, 0.7))
    gpu, orc, seqs, paged = run_round(w, absorbed=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_mla_shaped_long_extend_unabsorbed():
    # 2 sequences x 600 new rows over ragged cached prefixes (0..50 slots): the extend takes the
    # unabsorbed path (gathered and expanded keys/values, flash-attention tiles); the last query tile of
    # each sequence is partial and the last key tile runs past the configured context
    w = WL.workload("dsv3_b1", hidden=1024, n_heads=8, q_lora_rank=256, intermediate=2048,
                    target_vocab=8192, draft_vocab=4096, batch=2, ctx=(0, 50), t_new=600, gamma=2,
                    accept_p=(0.7, 0.7), seed=81)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_dsv3_long_extend_over_prefix_sampled():
    # full DeepseekV3 dimensions, 2 sequences x 1024 new rows over cached prefixes of 100..300 slots
    # (unabsorbed extend path); the oracle checks sequence 1
    w = WL.workload("dsv3_extend", batch=2, t_new=1024, ctx=(100, 300), gamma=2, accept_p=(0.7, 0.7), seed=82)
    gpu, orc, seqs, paged = run_round(w, seqs=[1], absorbed=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_dsv3_b64_full_size_sampled():
    # batch 64, ragged contexts U[1024, 8192], full 129280-entry vocab without d2t, gamma 5; the GPU runs
    # the whole batch on the tensor-core path, the oracle checks two sampled sequences (sequences are
    # independent)
    w = WL.workload("dsv3_b64")
    gpu, orc, seqs, paged = run_round(w, seqs=[5, 42], absorbed=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_dsv3_b256_full_size_sampled():
    # batch 256, contexts U[4096, 16384], gamma 7, 32000-entry draft vocab with d2t
    w = WL.workload("dsv3_b256")
    gpu, orc, seqs, paged = run_round(w, seqs=[0, 131], absorbed=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_dsv3_extend_full_size_sampled():
    # 8 sequences x 2048 new rows on an empty cache (causal extend at M = 16384 rows)
    w = WL.workload("dsv3_extend")
    gpu, orc, seqs, paged = run_round(w, seqs=[3], absorbed=True)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))
