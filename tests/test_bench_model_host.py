"""Host checks of the benchmark's algorithmic bytes and FLOP models (what the roofline fractions divide by)."""
import bench
import workloads as WL


def _tot(model):
    return sum(b * n for b, n in model.values())


def test_weight_bytes_of_the_projection_layers_follow_the_storage_format():
    w = WL.workload("dsv3_b1")
    L = WL.context_lengths(w)
    bf16 = bench.algorithmic_bytes(w, L)
    fp8 = bench.algorithmic_bytes(w, L, fp8=True)
    fp4 = bench.algorithmic_bytes(w, L, nvfp4=True)
    H, I, V = w.hidden, w.intermediate, w.draft_vocab
    # gate | up at batch 1: both weight matrices once plus the activations
    act = H * 4 + I * 4
    assert bf16["gate_up_silu"][0] == 2 * I * H * 2 + act
    assert fp8["gate_up_silu"][0] == 2 * I * (H + 4) + act                  # one byte each + a row scale
    assert fp4["gate_up_silu"][0] == 2 * I * H * (0.5 + 1 / 16) + act      # half a byte + a scale per 16
    assert bf16["lm_head_argmax"][0] == V * H * 2 + H * 4
    # kv_b (absorb, unabsorb) and the latent rows stay bf16 in every format
    for k in ("absorb", "unabsorb", "attention"):
        assert fp8[k] == bf16[k] == fp4[k]
    assert 0.49 < _tot(fp8) / _tot(bf16) < 0.52
    assert 0.27 < _tot(fp4) / _tot(bf16) < 0.30


def test_mha_model_counts_its_own_projections_and_cache_rows():
    w = WL.workload("mha_b1")
    L = WL.context_lengths(w)
    m = bench.algorithmic_bytes(w, L)
    f = bench.algorithmic_flops(w, L)
    H, nh, nkv, d = w.hidden, w.n_heads, w.n_kv_heads, w.head_dim
    assert "absorb" not in m and "unabsorb" not in m
    # q_proj under "q_b", k | v under "q_a_kv_a" (bf16 weights at 2H input)
    assert m["q_b"][0] == nh * d * 2 * H * 2 + 2 * H * 4 + nh * d * 4
    assert m["q_a_kv_a"][0] == 2 * nkv * d * 2 * H * 2 + 2 * H * 4 + 2 * nkv * d * 4
    # attention reads each live [k | v] row once per launch: 2 n_kv d bf16 values per slot
    assert m["attention"][1] == w.gamma
    assert m["attention"][0] * w.gamma == sum((int(l) + w.t_new + s) * 2 * nkv * d * 2 for l in L for s in range(w.gamma))
    # FLOPs: 2 per multiply-add, score and value per (row, head, visible slot)
    assert f["q_b"][0] == 2.0 * 2 * H * nh * d
    visible = sum(sum(int(l) + j + 1 for j in range(w.t_new)) for l in L)
    ext = 2.0 * nh * 2 * d * visible
    dec = [2.0 * nh * 2 * d * sum(int(l) + w.t_new + s for l in L) for s in range(1, w.gamma)]
    assert abs(f["attention"][0] * f["attention"][1] - (ext + sum(dec))) < 1e-6 * (ext + sum(dec))


def test_packed_views_keep_dtype_shape_and_bytes():
    # the end-to-end step's packed input buffer: typed views at 256-byte aligned offsets of one byte buffer
    import torch
    parts = [torch.arange(12, dtype=torch.bfloat16).view(3, 4), torch.arange(5, dtype=torch.int32),
             torch.rand(2, 3, 7, dtype=torch.float32)]
    offs, n = [], 0
    for t in parts:
        offs.append(n)
        n += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.zeros(n, dtype=torch.uint8)
    views = [bench.slice_as(buf, o, t) for o, t in zip(offs, parts)]
    for v, t in zip(views, parts):
        v.copy_(t)
    for o, v, t in zip(offs, views, parts):
        assert o % 256 == 0 and v.dtype == t.dtype and v.shape == t.shape
        assert torch.equal(v, t)
        assert v.data_ptr() == buf.data_ptr() + o
