"""The Llama-style MHA draft head ("Eagle3 DeepseekV3 in MAX" §11: LlamaForCausalLMEagle3 on a DeepseekV3
target, its own one-layer bf16 key/value cache) against the oracle: whole drafting rounds (extend +
gamma - 1 decode steps + acceptance) through the C ABI, compared element by element under the rules
of the MLA head's parity tests (hidden states, logits and appended cache rows within the tolerance,
tokens under the near-tie rule, acceptance bit-exact)."""
import pytest

import workloads as WL

from parity import TOL_BF16, TOL_F32, check_round, run_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from eagle_speculative_decoding_eagle3_gb300 import build
    build.build()


def _narrow(**kw):
    base = dict(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, intermediate=2048, target_vocab=8192,
                draft_vocab=4096)
    base.update(kw)
    return WL.workload("mha_b1", **base)


def test_mha_tiny_f32_round():
    # fp32 storage and arithmetic, 2-way fc, 4 query heads per key/value head, head_dim 32
    w = WL.workload("mha_tiny_f32")
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32))


def test_mha_tiny_f32_ragged_and_page_crossing():
    # 5 sequences with contexts 1..45, 7 new rows crossing 16-slot pages, 5 draft tokens
    w = WL.workload("mha_tiny_f32", batch=5, ctx=(1, 45), t_new=7, gamma=5, accept_p=(0.7,) * 5, seed=1012)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32))


def test_mha_tiny_f32_empty_cache_one_kv_head_per_query_head():
    # extend from an empty cache; n_kv_heads == n_heads (plain multi-head attention)
    w = WL.workload("mha_tiny_f32", n_kv_heads=8, ctx=(0, 0), t_new=9, seed=1013)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_F32))


def test_mha_bf16_round_gemv_decode_tensor_core_extend():
    # bf16 with head_dim 128: the extend (9 rows) takes the tensor-core projections, the decode steps
    # (3 rows) the GEMV path; contexts 100..700 split over several 128-slot chunks
    w = _narrow(batch=3, ctx=(100, 700), t_new=3, gamma=4, accept_p=(0.7,) * 4, seed=1014)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_mha_bf16_two_way_fc_seven_query_heads_per_kv_head():
    # fc over two aux states ([H, 2H]), 14 heads on 2 key/value heads, head_dim 64
    w = _narrow(n_heads=14, head_dim=64, hidden=896, fc_inputs=2, batch=2, ctx=(30, 300), t_new=2, gamma=3,
                accept_p=(0.7,) * 3, seed=1015)
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_mha_bf16_tensor_core_rounds():
    # 24 sequences: the extend (48 rows) and every decode step (24 rows) take the tensor-core path
    w = _narrow(batch=24, ctx=(30, 700), t_new=2, gamma=3, accept_p=(0.7,) * 3, seed=1016)
    gpu, orc, seqs, paged = run_round(w, seqs=[0, 7, 23])
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))


def test_mha_b1_full_size_round():
    # the batch-1 workload at full size: hidden 7168, 56 heads on 8 key/value heads, 4096-token cache,
    # 32000-entry draft vocabulary with d2t, as the benchmark runs it
    w = WL.workload("mha_b1")
    gpu, orc, seqs, paged = run_round(w)
    print(check_round(w, gpu, orc, seqs, paged, TOL_BF16))
