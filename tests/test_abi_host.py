"""Host-only checks of the C ABI: the library builds, loads, exports every declared entry point,
and rejects bad arguments before touching a GPU."""
import ctypes as C
import os
import re

import pytest

from eagle_speculative_decoding_eagle3_gb300 import build as B
from eagle_speculative_decoding_eagle3_gb300 import eagle3 as E

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return E._lib()


def declared_functions():
    names = []
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, f)).read()
            names += re.findall(r"EAGLE3_API\s+[\w\s\*]+?\b(eagle3_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert E.eagle3_status_string(0) == "ok"
    assert "CUDA" in E.eagle3_status_string(E.ERR_CUDA)
    assert E.eagle3_status_string(99) == "unknown status"


def _dsv3_config(**kw):
    base = dict(hidden=7168, n_heads=128, q_lora_rank=1536, kv_lora_rank=512, qk_nope_dim=128, qk_rope_dim=64,
                v_head_dim=128, intermediate=18432, target_vocab=129280, draft_vocab=32000, max_batch=1,
                max_tokens_per_extend=1, max_ctx=4100, page_size=64, max_pages_per_seq=65, yarn_factor=40.0,
                dtype=E.BF16)
    base.update(kw)
    return E.make_config(**base)


def test_workspace_bytes_and_config_checks(lib):
    n = E.eagle3_draft_workspace_bytes(_dsv3_config())
    assert 0 < n < 1 << 30
    # bigger batches need more workspace
    assert E.eagle3_draft_workspace_bytes(_dsv3_config(max_batch=256, max_tokens_per_extend=256)) > n
    bad = [dict(hidden=0), dict(qk_rope_dim=63), dict(rope_interleave=0), dict(dtype=7), dict(hidden=7164),
           dict(kv_lora_rank=256), dict(draft_vocab=200000), dict(max_ctx=10_000), dict(rms_eps=0.0)]
    for kw in bad:
        with pytest.raises(E.Eagle3Error) as ei:
            E.eagle3_draft_workspace_bytes(_dsv3_config(**kw))
        assert ei.value.status in (E.ERR_INVALID_ARG, E.ERR_UNSUPPORTED), kw


def test_null_arguments_are_rejected_without_a_gpu(lib):
    h = C.c_void_p()
    assert lib.eagle3_draft_create(None, None, C.byref(h)) == E.ERR_INVALID_ARG
    cfg = _dsv3_config()
    w = E.eagle3_weights_t()   # all null
    assert lib.eagle3_draft_create(C.byref(cfg), C.byref(w), C.byref(h)) == E.ERR_INVALID_ARG
    assert h.value is None
    kv = E.eagle3_kv_t()
    aux = (C.c_void_p * 3)()
    assert lib.eagle3_draft_extend(None, aux, None, None, None, 1, 1, C.byref(kv), None, None, None) == \
        E.ERR_INVALID_ARG
    assert lib.eagle3_draft_decode(None, 3, None, C.byref(kv), None, None, None, None) == E.ERR_INVALID_ARG
    assert lib.eagle3_accept(None, None, 1, 1, None, None, None) == E.ERR_INVALID_ARG
    assert lib.eagle3_draft_destroy(None) == E.OK


def test_accept_relaxed_rejects_bad_arguments(lib):
    # argument checks happen on the host before any launch
    for kw in [dict(draft=None), dict(k=0), dict(k=2000), dict(delta=-0.1), dict(batch=0), dict(gamma=0)]:
        args = dict(draft=16, ids=16, lp=16, think=None, batch=2, gamma=3, k=4, delta=0.6, acc=16)
        args.update(kw)
        with pytest.raises(E.Eagle3Error) as ei:
            E.eagle3_accept_relaxed(args["draft"], args["ids"], args["lp"], args["think"], args["batch"],
                                    args["gamma"], args["k"], args["delta"], args["acc"])
        assert ei.value.status == E.ERR_INVALID_ARG, kw


def test_typical_acceptance_and_uniforms_reject_bad_arguments(lib):
    for kw in [dict(draft=None), dict(probs=None), dict(batch=0), dict(gamma=0), dict(V=0), dict(eps=-0.1),
               dict(dlt=float("nan")), dict(acc=None)]:
        args = dict(draft=16, probs=16, batch=2, gamma=3, V=10, eps=0.09, dlt=0.3, acc=16)
        args.update(kw)
        with pytest.raises(E.Eagle3Error) as ei:
            E.eagle3_accept_typical(args["draft"], args["probs"], args["batch"], args["gamma"], args["V"], args["eps"],
                                    args["dlt"], args["acc"])
        assert ei.value.status == E.ERR_INVALID_ARG, kw
    with pytest.raises(E.Eagle3Error) as ei:
        E.eagle3_philox_uniforms(1, 0, -1, 16)
    assert ei.value.status == E.ERR_INVALID_ARG
    with pytest.raises(E.Eagle3Error) as ei:
        E.eagle3_philox_uniforms(1, 0, 8, None)
    assert ei.value.status == E.ERR_INVALID_ARG
    E.eagle3_philox_uniforms(1, 0, 0, None)   # nothing to draw: no launch, no GPU needed


def test_fp8_weight_format_checks_without_a_gpu(lib):
    # the format must be known, FP8 needs bf16 storage, and extends above the GEMV rows reserve the
    # bf16 expansion of the largest FP8 matrix pair (gate | up: 2 x 18432 x 7168 elements)
    for kw in [dict(weight_format=3), dict(weight_format=E.WEIGHTS_FP8, dtype=E.F32),
               dict(weight_format=E.WEIGHTS_FP8, hidden=7160),           # FP8 rows: K a multiple of 16
               dict(weight_format=E.WEIGHTS_NVFP4, intermediate=18448),  # NVFP4 rows: K a multiple of 32
               dict(weight_format=E.WEIGHTS_NVFP4, dtype=E.F32)]:
        with pytest.raises(E.Eagle3Error) as ei:
            E.eagle3_draft_workspace_bytes(_dsv3_config(**kw))
        assert ei.value.status in (E.ERR_INVALID_ARG, E.ERR_UNSUPPORTED), kw
    small = E.eagle3_draft_workspace_bytes(_dsv3_config(weight_format=E.WEIGHTS_FP8))
    assert small == E.eagle3_draft_workspace_bytes(_dsv3_config())
    big = dict(max_batch=64, max_tokens_per_extend=64)
    extra = E.eagle3_draft_workspace_bytes(_dsv3_config(weight_format=E.WEIGHTS_FP8, **big)) - \
        E.eagle3_draft_workspace_bytes(_dsv3_config(**big))
    assert 0 <= extra - 2 * 18432 * 7168 * 2 < 256
    # an FP8 head without its row scales is rejected before any CUDA call
    h = C.c_void_p()
    cfg = _dsv3_config(weight_format=E.WEIGHTS_FP8)
    w = E.eagle3_weights_t()
    for n in E.WEIGHT_NAMES:
        setattr(w, n, 256)
    assert lib.eagle3_draft_create(C.byref(cfg), C.byref(w), C.byref(h)) == E.ERR_INVALID_ARG
    assert h.value is None
    # the quantizer checks its arguments on the host
    assert lib.eagle3_quantize_e4m3(None, E.BF16, 4, 8, None, None, None) == E.ERR_INVALID_ARG
    assert lib.eagle3_quantize_e4m3(256, E.BF16, 0, 8, 256, 256, None) == E.ERR_INVALID_ARG
    assert lib.eagle3_quantize_e4m3(256, 7, 4, 8, 256, 256, None) == E.ERR_UNSUPPORTED
    # NVFP4: valid for the DeepseekV3 head's sizes; the quantizer wants K a multiple of 32
    assert E.eagle3_draft_workspace_bytes(_dsv3_config(weight_format=E.WEIGHTS_NVFP4, intermediate=18432)) > 0
    assert E.eagle3_draft_workspace_bytes(_dsv3_config(weight_format=E.WEIGHTS_FP8, intermediate=18448)) > 0
    assert lib.eagle3_quantize_nvfp4(None, E.BF16, 4, 32, None, None, None, None) == E.ERR_INVALID_ARG
    assert lib.eagle3_quantize_nvfp4(256, E.BF16, 4, 48, 256, 256, 256, None) == E.ERR_UNSUPPORTED
    assert lib.eagle3_quantize_nvfp4(256, 7, 4, 64, 256, 256, 256, None) == E.ERR_UNSUPPORTED
    # an NVFP4 head needs its matrix scales as well as the block scales
    cfg = _dsv3_config(weight_format=E.WEIGHTS_NVFP4)
    w = E.eagle3_weights_t()
    for n in E.WEIGHT_NAMES:
        setattr(w, n, 256)
    for n in E.FP8_WEIGHT_NAMES:
        setattr(w, n + "_scale", 256)
    assert lib.eagle3_draft_create(C.byref(cfg), C.byref(w), C.byref(h)) == E.ERR_INVALID_ARG


def _mha_config(**kw):
    base = dict(hidden=7168, n_heads=56, n_kv_heads=8, head_dim=128, intermediate=18432, target_vocab=129280,
                draft_vocab=32000, max_batch=1, max_tokens_per_extend=1, max_ctx=4100, page_size=64,
                max_pages_per_seq=65, yarn_factor=40.0, dtype=E.BF16, attention=E.ATTN_MHA, fc_inputs=3)
    base.update(kw)
    return E.make_config(**base)


def test_mha_config_checks_without_a_gpu(lib):
    # the MHA head ignores the MLA sizes (zero here) and checks its own
    n = E.eagle3_draft_workspace_bytes(_mha_config())
    assert 0 < n < 1 << 30
    assert E.eagle3_draft_workspace_bytes(_mha_config(fc_inputs=2)) > 0
    bad = [dict(attention=2), dict(n_kv_heads=0), dict(n_kv_heads=5), dict(n_heads=12, n_kv_heads=4),
           dict(head_dim=96), dict(weight_format=E.WEIGHTS_FP8), dict(fc_inputs=1), dict(hidden=7164),
           dict(max_ctx=10_000)]
    for kw in bad:
        with pytest.raises(E.Eagle3Error) as ei:
            E.eagle3_draft_workspace_bytes(_mha_config(**kw))
        assert ei.value.status in (E.ERR_INVALID_ARG, E.ERR_UNSUPPORTED), kw
    # a 2-way fc belongs to the MHA head only
    with pytest.raises(E.Eagle3Error):
        E.eagle3_draft_workspace_bytes(_dsv3_config(fc_inputs=2))
    # an MHA head without its q/k/v projections is rejected before any CUDA call, whatever its MLA
    # fields hold
    h = C.c_void_p()
    cfg = _mha_config()
    w = E.eagle3_weights_t()
    for nm in E.WEIGHT_NAMES:
        setattr(w, nm, 256)
    assert lib.eagle3_draft_create(C.byref(cfg), C.byref(w), C.byref(h)) == E.ERR_INVALID_ARG
    assert h.value is None


def test_sample_rejects_bad_arguments(lib):
    # one cluster of 8 CTAs per row along the grid's y dimension: rows past 65535 are refused on the host,
    # as are rows or vocabularies outside range and inconsistent filters (no launch, no GPU needed)
    base = dict(logits=16, rows=2, V=100, ld=100, T=0.8, k=50, p=0.9, u=16, tokens=16)
    for kw in [dict(logits=None), dict(u=None), dict(tokens=None), dict(rows=0), dict(rows=65536), dict(V=0),
               dict(V=131073, ld=131073), dict(ld=99), dict(k=1025), dict(k=-1), dict(p=0.0), dict(p=1.5),
               dict(k=0, p=0.5), dict(T=-1.0)]:
        args = dict(base)
        args.update(kw)
        with pytest.raises(E.Eagle3Error) as ei:
            E.eagle3_sample(args["logits"], args["rows"], args["V"], args["ld"], args["T"], args["k"], args["p"],
                            args["u"], None, 0, args["tokens"])
        assert ei.value.status == E.ERR_INVALID_ARG, kw
