"""The work counts behind bench.py's roofline fractions, pinned to numbers the
pages print: the SmolLM2-135M configuration and its 134,515,008-parameter
total (tests/golden/smollm2_135m_facts.json).  No GPU is involved."""
import json
import os

import numpy as np

import bench
from llama_decoder_forward_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLDEN, "smollm2_135m_facts.json")))


def _linear_weights_per_block(wl):
    """Weights of the four projections of one block, counted from the total the
    page prints: (total - embedding - final norm) / layers - the two norms."""
    per_block = (FACTS["param_total"] - wl.vocab * wl.hidden - wl.hidden) // wl.n_layers
    return per_block - 2 * wl.hidden


def test_workload_is_the_page_config():
    wl = synth.WORKLOADS["smollm2_model_b8_t2048"]
    c = FACTS["config"]
    assert (wl.hidden, wl.intermediate, wl.n_layers, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.vocab,
            wl.max_pos, wl.rms_eps, wl.rope_theta) == (
        c["hidden_size"], c["intermediate_size"], c["num_hidden_layers"], c["num_attention_heads"],
        c["num_key_value_heads"], c["head_dim"], c["vocab_size"], c["max_position_embeddings"],
        c["rms_norm_eps"], c["rope_theta"])


def test_prefill_flops_follow_the_parameter_total():
    # a dense product costs 2 FLOP per weight per token; attention is counted
    # causal-exact: QK^T and PV over the T(T+1)/2 visible pairs per head
    wl = synth.WORKLOADS["smollm2_model_b8_t2048"]
    M = wl.B * wl.T
    per = bench.prefill_flops_per_launch(wl)
    linear = per["qkv_gemm_rope"] + per["o_gemm_residual"] + per["gateup_gemm_swiglu"] + per["down_gemm_residual"]
    assert linear == 2 * M * _linear_weights_per_block(wl)
    assert per["lm_head_gemm"] == 2 * M * wl.vocab * wl.hidden
    pairs = wl.B * wl.n_heads * wl.T * (wl.T + 1) // 2
    assert per["flash_attention"] == pairs * 2 * 2 * wl.head_dim
    total = bench.prefill_flops_total(wl)
    assert total == wl.n_layers * (linear + per["flash_attention"]) + per["lm_head_gemm"]
    assert abs(total / 5.567e12 - 1) < 1e-3            # the per-forward figure quoted with the workload


def test_decode_bytes_follow_the_parameter_total():
    # every weight read once (bf16: 2 bytes per parameter), each cached key and
    # value of the prefix once, the new K/V written, the logits written
    wl = synth.WORKLOADS["smollm2_decode_b64_cache4096"]
    zero = np.zeros(wl.B, dtype=np.int64)
    step0, attn0 = bench.decode_bytes(wl, zero)
    new_kv = 2 * wl.n_layers * wl.B * wl.n_kv_heads * wl.head_dim * 2
    logits = wl.B * wl.vocab * 2
    assert step0 == 2 * FACTS["param_total"] + new_kv + logits
    lengths = np.arange(wl.B, dtype=np.int64) * 61 + 1024
    step, attn = bench.decode_bytes(wl, lengths)
    # 768 bytes per cached token per layer: K and V, 3 kv heads x 64 dims, bf16
    assert step - step0 == int(lengths.sum()) * wl.n_layers * 768
    # one attention launch reads one layer's prefix plus the new key/value of each sequence
    assert attn == int((lengths + 1).sum()) * 768 and attn0 == wl.B * 768


def test_block_workload_flops():
    # one unpadded SmolLM2 block step costs exactly one layer of the prefill count
    wl = synth.WORKLOADS["smollm2_block_b1_t128"]
    per = bench.prefill_flops_per_launch(wl)
    layer = sum(v for k, v in per.items() if k != "lm_head_gemm")
    flops, tokens = bench.block_flops(wl)
    assert (flops, tokens) == (layer, wl.B * wl.T)
    # left padding: only valid tokens count, each sequence's attention over its own length
    wl3 = synth.WORKLOADS["slm125m_block_leftpad_b16_t1024"]
    lengths = np.array([128, 1024] + [500] * (wl3.B - 2))
    f3, n3 = bench.block_flops(wl3, lengths)
    assert n3 == lengths.sum()
    lin = 2 * ((wl3.n_heads + 2 * wl3.n_kv_heads) * wl3.head_dim * wl3.hidden
               + wl3.hidden * wl3.n_heads * wl3.head_dim + 3 * wl3.intermediate * wl3.hidden)
    assert lin == 12_582_912                          # the per-token figure quoted with the workload
    attn = sum(4 * wl3.head_dim * wl3.n_heads * L * (L + 1) // 2 for L in lengths)
    assert f3 == lin * n3 + attn
    full, _ = bench.block_flops(wl3)
    assert full > f3
