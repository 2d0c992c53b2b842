"""Pins for the fp64 oracle: it is checked against things other than itself.

Each test names what fixes the expected value: a number the pages print, a
closed form, an invariant of the mathematics, a torch library routine, or a
scalar brute-force restatement (tests/bruteforce.py) on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import bruteforce as bf
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)

TINY = O.Config(hidden=8, n_heads=2, n_kv_heads=1, head_dim=4, intermediate=6, n_layers=2,
                vocab=11, max_pos=64, rms_eps=1e-5, rope_theta=100.0)


def tiny_weights(cfg, rng, std=0.4):
    d, hd = cfg.hidden, cfg.head_dim
    shapes = dict(wq=(cfg.n_heads * hd, d), wk=(cfg.n_kv_heads * hd, d), wv=(cfg.n_kv_heads * hd, d),
                  wo=(d, cfg.n_heads * hd), wgate=(cfg.intermediate, d), wup=(cfg.intermediate, d),
                  wdown=(d, cfg.intermediate))
    w = {k: rng.normal(0, std, s) for k, s in shapes.items()}
    w["attn_norm"] = 1 + rng.normal(0, 0.1, d)
    w["mlp_norm"] = 1 + rng.normal(0, 0.1, d)
    return w


def as_block(w):
    return O.BlockWeights(**{k: np.asarray(v) for k, v in w.items()})


def nested(a):
    return np.asarray(a).tolist()


# ---------------------------------------------------------------- page facts

def test_param_total_matches_page():
    facts = json.load(open(os.path.join(GOLDEN, "smollm2_135m_facts.json")))
    c = facts["config"]
    cfg = O.Config(hidden=c["hidden_size"], n_heads=c["num_attention_heads"],
                   n_kv_heads=c["num_key_value_heads"], head_dim=c["head_dim"],
                   intermediate=c["intermediate_size"], n_layers=c["num_hidden_layers"],
                   vocab=c["vocab_size"], max_pos=c["max_position_embeddings"],
                   rms_eps=c["rms_norm_eps"], rope_theta=float(c["rope_theta"]))
    assert cfg == O.SMOLLM2_135M
    assert cfg.hidden == cfg.n_heads * cfg.head_dim
    assert O.param_count(cfg, tied=c["tie_word_embeddings"]) == facts["param_total"]
    # an untied head would add exactly one more V x d matrix
    assert O.param_count(cfg, tied=False) == facts["param_total"] + cfg.vocab * cfg.hidden


def test_logits_shapes_match_page():
    facts = json.load(open(os.path.join(GOLDEN, "smollm2_135m_facts.json")))
    rng = np.random.default_rng(0)
    for (ids_shape, logits_shape) in facts["logits_shapes"]:
        # same shapes with a tiny stand-in vocabulary/depth; the vocab axis is checked symbolically
        cfg = TINY
        layers = [as_block(tiny_weights(cfg, rng))]
        embed = rng.normal(0, 0.3, (cfg.vocab, cfg.hidden))
        ids = rng.integers(0, cfg.vocab, ids_shape)
        out = O.model_forward(cfg, layers, embed, np.ones(cfg.hidden), ids)
        assert out.shape == tuple(ids_shape) + (cfg.vocab,)
        assert logits_shape[-1] == O.SMOLLM2_135M.vocab and list(logits_shape[:2]) == list(ids_shape)


def test_max_position_guard():
    cfg = O.Config(**{**TINY.__dict__, "max_pos": 4})
    rng = np.random.default_rng(0)
    layers = [as_block(tiny_weights(cfg, rng))]
    embed = rng.normal(0, 0.3, (cfg.vocab, cfg.hidden))
    with pytest.raises(ValueError):
        O.model_forward(cfg, layers, embed, np.ones(cfg.hidden), np.zeros((1, 5), dtype=int))


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_forms():
    # constant vector c: every output is w_i * c / sqrt(c^2 + eps)
    c, eps = 3.0, 1e-5
    w = np.array([1.0, 2.0, -0.5, 4.0])
    y = O.rms_norm(np.full(4, c), w, eps)
    np.testing.assert_allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-15)
    # [1,2,3,4], w=1, eps=0: mean square 7.5
    y = O.rms_norm(np.array([1.0, 2, 3, 4]), np.ones(4), 0.0)
    np.testing.assert_allclose(y, np.array([1, 2, 3, 4]) / math.sqrt(7.5), rtol=1e-15)
    # w = 1, eps = 0 gives unit root-mean-square output, scale-invariant input
    x = RNG.normal(0, 5, (7, 33))
    y = O.rms_norm(x, np.ones(33), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(10 * x, np.ones(33), 0.0), y, rtol=1e-13)


def test_rmsnorm_vs_torch_library():
    x = RNG.normal(0, 1, (5, 24))
    w = 1 + RNG.normal(0, 0.1, 24)
    ref = F.rms_norm(torch.tensor(x), (24,), torch.tensor(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- RoPE

def test_rope_inv_freq_closed_form():
    f = O.rope_inv_freq(64, 1e4)
    assert f[0] == 1.0
    np.testing.assert_allclose(f[16], 1e4 ** -0.5, rtol=1e-15)   # i = hd/4 -> theta^(-1/2)
    # the first model.py's form base^(-i/half) is the same number
    half = 32
    np.testing.assert_allclose(f, 1.0 / (1e4 ** (np.arange(half) / half)), rtol=1e-14)
    assert np.all(np.diff(f) < 0)


def test_rope_position_zero_is_identity():
    x = RNG.normal(0, 1, (3, 5, 64))
    np.testing.assert_array_equal(O.apply_rope(x, np.zeros((3, 5), dtype=int), 1e5), x)


def test_rope_preserves_norm_of_each_pair():
    x = RNG.normal(0, 1, (4, 64))
    pos = np.array([0, 7, 300, 8191])
    y = O.apply_rope(x, pos, 1e5)
    pair = lambda a: a[..., :32] ** 2 + a[..., 32:] ** 2
    np.testing.assert_allclose(pair(y), pair(x), rtol=1e-12)


def test_rope_relative_position_invariance():
    q = RNG.normal(0, 1, 64)
    k = RNG.normal(0, 1, 64)
    for m, n, delta in [(5, 2, 11), (100, 3, 1000), (0, 0, 4096)]:
        a = O.apply_rope(q, np.array(m), 1e5) @ O.apply_rope(k, np.array(n), 1e5)
        b = O.apply_rope(q, np.array(m + delta), 1e5) @ O.apply_rope(k, np.array(n + delta), 1e5)
        assert abs(a - b) < 1e-11 * (1 + abs(a))


def test_rope_equals_complex_rotation():
    x = RNG.normal(0, 1, 8)
    for pos in (1, 3, 250):
        y = O.apply_rope(x, np.array(pos), 10.0)
        ref = bf.rotate(list(x), pos, 10.0)
        np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)
    # explicit 2x2 rotation of the first pair at pos 1, freq 1: angle = 1 rad
    e = np.zeros(8); e[0] = 1.0
    y = O.apply_rope(e, np.array(1), 10.0)
    np.testing.assert_allclose([y[0], y[4]], [math.cos(1.0), math.sin(1.0)], rtol=1e-15)


# ---------------------------------------------------------------- SiLU

def test_silu_vs_torch_and_limits():
    z = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(O.silu(z), F.silu(torch.tensor(z)).numpy(), rtol=1e-14, atol=1e-300)
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(40.0) - 40.0) < 1e-15 * 40 * 10
    assert abs(O.silu(-40.0)) < 1e-15


# ---------------------------------------------------------------- attention

def _rand_qkv(B, H, KV, T, hd, rng):
    return (rng.normal(0, 1, (B, H, T, hd)), rng.normal(0, 1, (B, KV, T, hd)),
            rng.normal(0, 1, (B, KV, T, hd)))


def test_attention_vs_bruteforce_loops():
    rng = np.random.default_rng(7)
    B, H, KV, T, hd = 2, 6, 2, 7, 4
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    vs = [0, 3]
    o = O.gqa_attention(q, k, v, vs)
    for b in range(B):
        for h in range(H):
            kvh = h // (H // KV)
            for t in range(T):
                keys = [j for j in range(T) if vs[b] <= j <= t]
                if not keys:
                    np.testing.assert_array_equal(o[b, h, t], 0.0)
                    continue
                s = [sum(q[b, h, t, c] * k[b, kvh, j, c] for c in range(hd)) / math.sqrt(hd) for j in keys]
                e = [math.exp(x) for x in s]
                ref = [sum(e[a] * v[b, kvh, j, c] for a, j in enumerate(keys)) / sum(e) for c in range(hd)]
                np.testing.assert_allclose(o[b, h, t], ref, rtol=1e-12, atol=1e-13)


def test_attention_vs_torch_sdpa():
    rng = np.random.default_rng(8)
    B, H, KV, T, hd = 2, 9, 3, 33, 16
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    g = H // KV
    kt = torch.tensor(k).repeat_interleave(g, dim=1)
    vt = torch.tensor(v).repeat_interleave(g, dim=1)
    ref = F.scaled_dot_product_attention(torch.tensor(q), kt, vt, is_causal=True).numpy()
    np.testing.assert_allclose(O.gqa_attention(q, k, v), ref, rtol=1e-11, atol=1e-12)


def test_attention_causality():
    rng = np.random.default_rng(9)
    B, H, KV, T, hd = 1, 4, 2, 12, 8
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    base = O.gqa_attention(q, k, v)
    t = 6
    k2, v2, q2 = k.copy(), v.copy(), q.copy()
    k2[:, :, t + 1] += 3.0
    v2[:, :, t + 1] -= 2.0
    q2[:, :, t + 1] *= -1
    pert = O.gqa_attention(q2, k2, v2)
    np.testing.assert_array_equal(pert[:, :, :t + 1], base[:, :, :t + 1])
    assert not np.allclose(pert[:, :, t + 1], base[:, :, t + 1])


# ---------------------------------------------------------------- block / model

def test_block_vs_bruteforce_loops():
    rng = np.random.default_rng(11)
    w = tiny_weights(TINY, rng)
    x = rng.normal(0, 1, (2, 5, TINY.hidden))
    for vs in (None, [0, 2]):
        out = O.block_forward(TINY, as_block(w), x, vs)
        ref = np.array(bf.block(TINY, {k: nested(a) for k, a in w.items()}, nested(x), vs))
        rows = slice(None) if vs is None else None
        if vs is None:
            np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
        else:
            for b in range(2):
                np.testing.assert_allclose(out[b, vs[b]:], ref[b, vs[b]:], rtol=1e-11, atol=1e-12)


def test_block_gqa_with_groups_of_three():
    cfg = O.Config(hidden=12, n_heads=6, n_kv_heads=2, head_dim=2, intermediate=5, n_layers=1,
                   vocab=5, max_pos=64, rms_eps=1e-6, rope_theta=1e4)
    rng = np.random.default_rng(12)
    w = tiny_weights(cfg, rng)
    x = rng.normal(0, 1, (1, 4, cfg.hidden))
    out = O.block_forward(cfg, as_block(w), x)
    ref = np.array(bf.block(cfg, {k: nested(a) for k, a in w.items()}, nested(x)))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_gqa_equals_mha_with_duplicated_kv_weights():
    cfg = O.Config(hidden=24, n_heads=6, n_kv_heads=2, head_dim=4, intermediate=10, n_layers=1,
                   vocab=5, max_pos=64, rms_eps=1e-5, rope_theta=1e4)
    rng = np.random.default_rng(13)
    w = tiny_weights(cfg, rng)
    x = rng.normal(0, 1, (2, 9, cfg.hidden))
    g = cfg.n_heads // cfg.n_kv_heads
    hd = cfg.head_dim
    dup = lambda m: np.concatenate([m[(h // g) * hd:(h // g + 1) * hd] for h in range(cfg.n_heads)])
    w_mha = dict(w, wk=dup(w["wk"]), wv=dup(w["wv"]))
    cfg_mha = O.Config(**{**cfg.__dict__, "n_kv_heads": cfg.n_heads})
    np.testing.assert_allclose(O.block_forward(cfg, as_block(w), x),
                               O.block_forward(cfg_mha, as_block(w_mha), x), rtol=1e-13, atol=1e-13)


def test_block_decomposition_identity():
    rng = np.random.default_rng(14)
    w = tiny_weights(TINY, rng)
    x = rng.normal(0, 1, (2, 6, TINY.hidden))
    taps = {}
    out = O.block_forward(TINY, as_block(w), x, taps=taps)
    np.testing.assert_array_equal(taps["layer_input"] + taps["attention_output"] + taps["mlp_output"], out)
    np.testing.assert_array_equal(taps["layer_mid"], taps["layer_input"] + taps["attention_output"])


def test_block_causality():
    rng = np.random.default_rng(15)
    w = tiny_weights(TINY, rng)
    x = rng.normal(0, 1, (1, 8, TINY.hidden))
    base = O.block_forward(TINY, as_block(w), x)
    x2 = x.copy()
    x2[0, 5] += 1.0
    pert = O.block_forward(TINY, as_block(w), x2)
    np.testing.assert_array_equal(pert[0, :5], base[0, :5])
    assert not np.allclose(pert[0, 5], base[0, 5])


def test_left_padding_equals_unpadded_run():
    cfg = O.Config(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=12, n_layers=1,
                   vocab=5, max_pos=64, rms_eps=1e-5, rope_theta=1e4)
    rng = np.random.default_rng(16)
    w = as_block(tiny_weights(cfg, rng))
    T, lens = 10, [10, 4, 7]
    x = rng.normal(0, 1, (3, T, cfg.hidden))
    vs = [T - L for L in lens]
    padded = O.block_forward(cfg, w, x, vs)
    for b, L in enumerate(lens):
        alone = O.block_forward(cfg, w, x[b:b + 1, T - L:])
        np.testing.assert_allclose(padded[b, T - L:], alone[0], rtol=1e-13, atol=1e-13)
        # padding rows keep their residual input plus the MLP of it: attention output is 0
        taps = {}
        O.block_forward(cfg, w, x[b:b + 1], [T - L], taps=taps)
        np.testing.assert_array_equal(taps["attention_head_outputs"][0, :T - L], 0.0)


def test_model_vs_bruteforce_loops():
    rng = np.random.default_rng(17)
    layers_raw = [tiny_weights(TINY, rng) for _ in range(2)]
    embed = rng.normal(0, 0.5, (TINY.vocab, TINY.hidden))
    fnorm = 1 + rng.normal(0, 0.1, TINY.hidden)
    ids = rng.integers(0, TINY.vocab, (2, 4))
    out = O.model_forward(TINY, [as_block(w) for w in layers_raw], embed, fnorm, ids)
    ref = np.array(bf.model(TINY, [{k: nested(a) for k, a in w.items()} for w in layers_raw],
                            nested(embed), nested(fnorm), nested(ids)))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_tied_head_uses_embedding_table():
    rng = np.random.default_rng(18)
    layers = [as_block(tiny_weights(TINY, rng))]
    embed = rng.normal(0, 0.5, (TINY.vocab, TINY.hidden))
    fnorm = 1 + rng.normal(0, 0.1, TINY.hidden)
    ids = rng.integers(0, TINY.vocab, (1, 3))
    taps = {}
    logits = O.model_forward(TINY, layers, embed, fnorm, ids, taps=taps)
    # scaling row r of the table scales column r of the logits of the last layer's output only via
    # the head (the embedding of ids not equal to r is untouched)
    r = [i for i in range(TINY.vocab) if i not in ids[0]][0]
    embed2 = embed.copy(); embed2[r] *= 2.0
    logits2 = O.model_forward(TINY, layers, embed2, fnorm, ids)
    np.testing.assert_allclose(logits2[..., r], 2.0 * logits[..., r], rtol=1e-13)
    others = [i for i in range(TINY.vocab) if i != r]
    np.testing.assert_array_equal(logits2[..., others], logits[..., others])


# ---------------------------------------------------------------- decode

def _prefill_cache(cfg, layers, embed, ids):
    """Post-RoPE K and V of every layer for a prefill of ids [B, T]."""
    x = embed[ids]
    ks, vs = [], []
    for l, w in enumerate(layers):
        taps = {}
        x = O.block_forward(cfg, w, x, taps=taps, layer=l)
        ks.append(taps["attention_keys"])
        vs.append(taps["attention_values"])
    return np.stack(ks), np.stack(vs)   # [L, B, KV, T, hd]


def test_decode_matches_last_row_of_prefill():
    cfg = O.Config(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=12, n_layers=3,
                   vocab=13, max_pos=64, rms_eps=1e-5, rope_theta=1e4)
    rng = np.random.default_rng(19)
    layers = [as_block(tiny_weights(cfg, rng)) for _ in range(cfg.n_layers)]
    embed = rng.normal(0, 0.5, (cfg.vocab, cfg.hidden))
    fnorm = 1 + rng.normal(0, 0.1, cfg.hidden)
    lens = [5, 9]
    S = 12
    seqs = [rng.integers(0, cfg.vocab, L + 1) for L in lens]
    k_cache = np.zeros((cfg.n_layers, 2, cfg.n_kv_heads, S, cfg.head_dim))
    v_cache = np.zeros_like(k_cache)
    for b, L in enumerate(lens):
        k, v = _prefill_cache(cfg, layers, embed, seqs[b][None, :L])
        k_cache[:, b, :, :L] = k[:, 0]
        v_cache[:, b, :, :L] = v[:, 0]
        k_cache[:, b, :, L:] = 99.0        # slots past the length must not be read
        v_cache[:, b, :, L:] = -99.0
    ids = np.array([s[-1] for s in seqs])
    logits, k_new, v_new = O.decode_step(cfg, layers, embed, fnorm, ids, lens, k_cache, v_cache)
    for b, L in enumerate(lens):
        full = O.model_forward(cfg, layers, embed, fnorm, seqs[b][None])
        np.testing.assert_allclose(logits[b], full[0, -1], rtol=1e-11, atol=1e-12)
        k, v = _prefill_cache(cfg, layers, embed, seqs[b][None])
        np.testing.assert_allclose(k_new[:, b], k[:, 0, :, L], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(v_new[:, b], v[:, 0, :, L], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- SmolLM3 variants:
# NoPE blocks and sliding windows ("SmolLM3", nnterp encyclopedia: "Every fourth
# block has no rotary", "On a NoPE block the queries and keys are the
# projections", "A sliding window the 3B checkpoints leave off")

def _with(cfg, **kw):
    return O.Config(**{**cfg.__dict__, **kw})


def test_block_kind_defaults_and_lists():
    assert O.block_kind(TINY, 0) == (True, 0) and O.block_kind(TINY, 1) == (True, 0)
    cfg = _with(TINY, no_rope_layers=(1, 0), sliding_window=(0, 128))
    assert O.block_kind(cfg, 0) == (True, 0)
    assert O.block_kind(cfg, 1) == (False, 128)


def test_nope_and_window_block_vs_bruteforce_loops():
    rng = np.random.default_rng(21)
    w = tiny_weights(TINY, rng)
    x = rng.normal(0, 1, (2, 9, TINY.hidden))
    wn = {k: nested(a) for k, a in w.items()}
    for rope, window in ((False, 0), (True, 3), (False, 4), (True, 1)):
        cfg = _with(TINY, no_rope_layers=(int(rope), 1), sliding_window=(window, 0))
        for vs in (None, [0, 3]):
            out = O.block_forward(cfg, as_block(w), x, vs, layer=0)
            ref = np.array(bf.block(TINY, wn, nested(x), vs, rope=rope, window=window))
            for b in range(2):
                v0 = 0 if vs is None else vs[b]
                np.testing.assert_allclose(out[b, v0:], ref[b, v0:], rtol=1e-11, atol=1e-12)


def test_nope_queries_are_the_projections():
    # on a NoPE block the attention's queries and keys equal the projections split
    # into heads at every position; on a rotary block only at position 0
    rng = np.random.default_rng(22)
    w = tiny_weights(TINY, rng)
    x = rng.normal(0, 1, (1, 6, TINY.hidden))
    cfg = _with(TINY, no_rope_layers=(1, 0))
    t_rot, t_nope = {}, {}
    O.block_forward(cfg, as_block(w), x, taps=t_rot, layer=0)
    O.block_forward(cfg, as_block(w), x, taps=t_nope, layer=1)
    np.testing.assert_array_equal(t_rot["attention_norm_output"], t_nope["attention_norm_output"])
    raw_q = np.matmul(t_nope["attention_norm_output"], np.asarray(w["wq"]).T)
    raw_q = raw_q.reshape(1, 6, TINY.n_heads, TINY.head_dim).transpose(0, 2, 1, 3)
    np.testing.assert_array_equal(t_nope["attention_queries"], raw_q)
    np.testing.assert_array_equal(t_rot["attention_queries"][:, :, 0], raw_q[:, :, 0])
    assert not np.allclose(t_rot["attention_queries"][:, :, 1:], raw_q[:, :, 1:])


def test_nope_last_row_ignores_the_order_of_earlier_tokens():
    # without the rotary a score depends on the two tokens' contents alone, so
    # the last query (which sees every key) is unchanged by permuting the keys
    # before it; with the rotary it changes
    cfg = O.Config(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=12, n_layers=2,
                   vocab=5, max_pos=64, rms_eps=1e-5, rope_theta=10.0, no_rope_layers=(1, 0))
    rng = np.random.default_rng(23)
    w = as_block(tiny_weights(cfg, rng))
    T = 8
    x = rng.normal(0, 1, (1, T, cfg.hidden))
    perm = np.concatenate([rng.permutation(T - 1), [T - 1]])
    xp = x[:, perm]
    nope = O.block_forward(cfg, w, x, layer=1)[0, -1]
    nope_p = O.block_forward(cfg, w, xp, layer=1)[0, -1]
    np.testing.assert_allclose(nope_p, nope, rtol=1e-12, atol=1e-12)
    rot = O.block_forward(cfg, w, x, layer=0)[0, -1]
    rot_p = O.block_forward(cfg, w, xp, layer=0)[0, -1]
    assert np.max(np.abs(rot_p - rot)) > 1e-6


def test_window_not_shorter_than_sequence_is_full_causal():
    rng = np.random.default_rng(24)
    B, H, KV, T, hd = 2, 6, 2, 11, 4
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    full = O.gqa_attention(q, k, v, [0, 4])
    for wdw in (T, T + 5):
        np.testing.assert_array_equal(O.gqa_attention(q, k, v, [0, 4], window=wdw), full)
    assert not np.allclose(O.gqa_attention(q, k, v, [0, 4], window=T - 1), full)


def test_window_of_one_returns_own_value():
    # a single visible key gets softmax weight exactly 1
    rng = np.random.default_rng(25)
    B, H, KV, T, hd = 2, 6, 3, 9, 8
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    o = O.gqa_attention(q, k, v, window=1)
    g = H // KV
    for h in range(H):
        np.testing.assert_array_equal(o[:, h], v[:, h // g])


def test_window_vs_torch_sdpa_band_mask():
    rng = np.random.default_rng(26)
    B, H, KV, T, hd = 2, 8, 2, 40, 16
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    g = H // KV
    kt = torch.tensor(k).repeat_interleave(g, dim=1)
    vt = torch.tensor(v).repeat_interleave(g, dim=1)
    for wdw in (1, 5, 16, 39):
        ones = torch.ones(T, T, dtype=torch.bool)
        band = torch.tril(ones) & ~torch.tril(ones, diagonal=-wdw)
        ref = F.scaled_dot_product_attention(torch.tensor(q), kt, vt, attn_mask=band).numpy()
        np.testing.assert_allclose(O.gqa_attention(q, k, v, window=wdw), ref, rtol=1e-11, atol=1e-12)


def test_window_locality_of_a_block():
    # with window w, block output row t depends on input rows t-w+1 .. t only
    wdw = 3
    cfg = _with(TINY, sliding_window=(wdw, 0))
    rng = np.random.default_rng(27)
    w = as_block(tiny_weights(TINY, rng))
    x = rng.normal(0, 1, (1, 12, TINY.hidden))
    base = O.block_forward(cfg, w, x, layer=0)
    j0 = 4
    x2 = x.copy()
    x2[0, j0] += 1.5
    pert = O.block_forward(cfg, w, x2, layer=0)
    np.testing.assert_array_equal(pert[0, :j0], base[0, :j0])
    np.testing.assert_array_equal(pert[0, j0 + wdw:], base[0, j0 + wdw:])
    for t in range(j0, j0 + wdw):
        assert not np.allclose(pert[0, t], base[0, t])


def test_model_with_nope_and_window_vs_bruteforce_loops():
    rng = np.random.default_rng(28)
    cfg = _with(TINY, no_rope_layers=(1, 0), sliding_window=(0, 2))
    layers_raw = [tiny_weights(TINY, rng) for _ in range(2)]
    embed = rng.normal(0, 0.5, (TINY.vocab, TINY.hidden))
    fnorm = 1 + rng.normal(0, 0.1, TINY.hidden)
    ids = rng.integers(0, TINY.vocab, (2, 5))
    out = O.model_forward(cfg, [as_block(w) for w in layers_raw], embed, fnorm, ids)
    ref = np.array(bf.model(TINY, [{k: nested(a) for k, a in w.items()} for w in layers_raw],
                            nested(embed), nested(fnorm), nested(ids), kinds=[(True, 0), (False, 2)]))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_decode_with_nope_and_windows_matches_last_row_of_prefill():
    cfg = O.Config(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=12, n_layers=3,
                   vocab=13, max_pos=64, rms_eps=1e-5, rope_theta=1e4,
                   no_rope_layers=(1, 0, 0), sliding_window=(0, 3, 7))
    rng = np.random.default_rng(29)
    layers = [as_block(tiny_weights(cfg, rng)) for _ in range(cfg.n_layers)]
    embed = rng.normal(0, 0.5, (cfg.vocab, cfg.hidden))
    fnorm = 1 + rng.normal(0, 0.1, cfg.hidden)
    lens = [1, 5, 9, 2]
    S = 12
    seqs = [rng.integers(0, cfg.vocab, L + 1) for L in lens]
    k_cache = np.zeros((cfg.n_layers, len(lens), cfg.n_kv_heads, S, cfg.head_dim))
    v_cache = np.zeros_like(k_cache)
    for b, L in enumerate(lens):
        k, v = _prefill_cache(cfg, layers, embed, seqs[b][None, :L])
        k_cache[:, b, :, :L] = k[:, 0]
        v_cache[:, b, :, :L] = v[:, 0]
        k_cache[:, b, :, L:] = 99.0        # slots past the length must not be read
        v_cache[:, b, :, L:] = -99.0
    # slots that fall out of layer 1's window (3) must not be read either
    k_cache[1, 2, :, :9 - 2] = 77.0
    v_cache[1, 2, :, :9 - 2] = -77.0
    ids = np.array([s[-1] for s in seqs])
    logits, k_new, v_new = O.decode_step(cfg, layers, embed, fnorm, ids, lens, k_cache, v_cache)
    for b, L in enumerate(lens):
        full = O.model_forward(cfg, layers, embed, fnorm, seqs[b][None])
        np.testing.assert_allclose(logits[b], full[0, -1], rtol=1e-11, atol=1e-12)
        k, v = _prefill_cache(cfg, layers, embed, seqs[b][None])
        np.testing.assert_allclose(k_new[:, b], k[:, 0, :, L], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(v_new[:, b], v[:, 0, :, L], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- next-token choice
# ("model.py" (SmolLM2-135M) section 7 generate; the abi96062 model.py generate)

def _sm(vals):
    e = [math.exp(v) for v in vals]
    return [x / sum(e) for x in e]


def test_sample_greedy_first_maximum():
    row = np.array([[1.0, 5.0, 5.0, 2.0]])
    for kw in (dict(do_sample=False), dict(temperature=0.0)):
        assert O.sample_next(row, u=[0.99], **kw)[0] == 1


def test_sample_top_p_hand_example():
    # softmax([3,2,1,0]) = (0.6439, 0.2369, 0.0871, 0.0321): top_p 0.7 keeps
    # tokens 0 and 1 (the token that crosses 0.7 stays), top_p 0.5 token 0 only
    row = np.array([[3.0, 2.0, 1.0, 0.0]])
    p = _sm([3.0, 2.0, 1.0, 0.0])
    assert p[0] <= 0.7 < p[0] + p[1]
    p0 = math.exp(3.0) / (math.exp(3.0) + math.exp(2.0))        # renormalised over {0, 1}
    assert O.sample_next(row, top_p=0.7, u=[p0 - 1e-9])[0] == 0
    assert O.sample_next(row, top_p=0.7, u=[p0 + 1e-9])[0] == 1
    assert O.sample_next(row, top_p=0.7, u=[0.999999])[0] == 1
    for u in (0.0, 0.5, 0.999999):
        assert O.sample_next(row, top_p=0.5, u=[u])[0] == 0


def test_sample_top_p_applies_after_top_k():
    # top_k 2 first: softmax over {3, 2} gives token 0 probability 0.7311 > 0.7,
    # so top_p 0.7 then keeps token 0 alone; without top_k it keeps 0 and 1
    row = np.array([[3.0, 2.0, 1.0, 0.0]])
    assert O.sample_next(row, top_k=2, top_p=0.7, u=[0.9])[0] == 0
    assert O.sample_next(row, top_p=0.7, u=[0.9])[0] == 1


def test_sample_top_k_keeps_ties_with_the_kth():
    row = np.array([[4.0, 4.0, 4.0, 1.0]])
    # three equal survivors, probability 1/3 each; token 3 is never drawn
    assert [O.sample_next(row, top_k=2, u=[u])[0] for u in (0.1, 0.5, 0.9, 0.9999)] == [0, 1, 2, 2]
    # top_k 1 keeps the maximum (and values equal to it)
    rng = np.random.default_rng(30)
    rows = rng.normal(0, 2, (20, 50))
    us = rng.random(20)
    np.testing.assert_array_equal(O.sample_next(rows, top_k=1, u=us), np.argmax(rows, axis=1))


def test_sample_top_p_ties_in_index_order():
    row = np.array([[2.0, 2.0, 2.0, 2.0]])
    # cumulative 0.25, 0.5, ...: top_p 0.3 keeps the first two sorted, i.e. indices 0 and 1
    assert O.sample_next(row, top_p=0.3, u=[0.6])[0] == 1
    assert O.sample_next(row, top_p=0.3, u=[0.4])[0] == 0
    # a tiny, zero or negative top_p keeps only the first sorted entry: the lowest index of the maximum
    row2 = np.array([[1.0, 5.0, 5.0, 2.0]])
    for tp in (1e-9, 0.0, -0.5):
        assert O.sample_next(row2, top_p=tp, u=[0.99])[0] == 1


def test_sample_inverse_cdf_frequencies_match_softmax():
    # u on a uniform grid of N points: token i is drawn for the points in
    # [cdf_{i-1}, cdf_i), so its count is N * softmax_i to within one point
    rng = np.random.default_rng(31)
    vals = rng.normal(0, 1.5, 6)
    temp = 0.8
    N = 20000
    us = (np.arange(N) + 0.5) / N
    toks = O.sample_next(np.repeat(vals[None], N, axis=0), temperature=temp, u=us)
    counts = np.bincount(toks, minlength=6)
    expect = np.array(_sm(list(vals / temp))) * N
    assert np.all(np.abs(counts - expect) <= 1.0 + 1e-9)
    # and the draw is monotone in u (vocabulary order)
    assert np.all(np.diff(toks) >= 0)


def test_sample_temperature_is_a_logit_scale():
    # dividing by 0.5 is multiplying by 2 exactly: the same draws as logits * 2 at temperature 1
    rng = np.random.default_rng(32)
    rows = rng.normal(0, 1, (30, 40))
    us = rng.random(30)
    for kw in (dict(), dict(top_k=7), dict(top_p=0.8), dict(top_k=9, top_p=0.6)):
        np.testing.assert_array_equal(O.sample_next(rows, temperature=0.5, u=us, **kw),
                                      O.sample_next(rows * 2.0, temperature=1.0, u=us, **kw))


# ---------------------------------------------------------------- prefill on top of a cache
# ("model.py" (SmolLM2-135M) section 4 with past_key_value and section 7: the
# causal mask offset by the past, RoPE rows sliced at the past length)

def _chunk_cfg(**kw):
    return O.Config(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=12, n_layers=3,
                    vocab=13, max_pos=64, rms_eps=1e-5, rope_theta=1e4, **kw)


def _cache_from(cfg, layers, embed, seqs, S):
    """Caches [L, B, KV, S, hd] filled by full prefills of each sequence;
    slots past each length hold poison that must never be read."""
    k_cache = np.full((cfg.n_layers, len(seqs), cfg.n_kv_heads, S, cfg.head_dim), 99.0)
    v_cache = np.full_like(k_cache, -99.0)
    for b, sq in enumerate(seqs):
        if len(sq):
            k, v = _prefill_cache(cfg, layers, embed, np.asarray(sq)[None])
            k_cache[:, b, :, :len(sq)] = k[:, 0]
            v_cache[:, b, :, :len(sq)] = v[:, 0]
    return k_cache, v_cache


@pytest.mark.parametrize("kinds", [dict(), dict(no_rope_layers=(1, 0, 1), sliding_window=(0, 3, 5))])
def test_chunked_prefill_equals_full_prefill(kinds):
    cfg = _chunk_cfg(**kinds)
    rng = np.random.default_rng(33)
    layers = [as_block(tiny_weights(cfg, rng)) for _ in range(cfg.n_layers)]
    embed = rng.normal(0, 0.5, (cfg.vocab, cfg.hidden))
    fnorm = 1 + rng.normal(0, 0.1, cfg.hidden)
    T, past = 4, [0, 3, 7]
    seqs = [rng.integers(0, cfg.vocab, p + T) for p in past]
    k_cache, v_cache = _cache_from(cfg, layers, embed, [s[:p] for s, p in zip(seqs, past)], 12)
    new_ids = np.stack([s[p:] for s, p in zip(seqs, past)])
    logits, k_new, v_new = O.prefill_with_cache(cfg, layers, embed, fnorm, new_ids, past, k_cache, v_cache)
    for b, p in enumerate(past):
        full = O.model_forward(cfg, layers, embed, fnorm, seqs[b][None])
        np.testing.assert_allclose(logits[b], full[0, p:], rtol=1e-11, atol=1e-12)
        k, v = _prefill_cache(cfg, layers, embed, seqs[b][None])
        np.testing.assert_allclose(k_new[:, b], k[:, 0, :, p:], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(v_new[:, b], v[:, 0, :, p:], rtol=1e-11, atol=1e-12)


def test_three_chained_chunks_equal_one_prefill():
    cfg = _chunk_cfg(sliding_window=(0, 4, 0))
    rng = np.random.default_rng(34)
    layers = [as_block(tiny_weights(cfg, rng)) for _ in range(cfg.n_layers)]
    embed = rng.normal(0, 0.5, (cfg.vocab, cfg.hidden))
    fnorm = 1 + rng.normal(0, 0.1, cfg.hidden)
    ids = rng.integers(0, cfg.vocab, (2, 9))
    S = 9
    k_cache = np.zeros((cfg.n_layers, 2, cfg.n_kv_heads, S, cfg.head_dim))
    v_cache = np.zeros_like(k_cache)
    outs, at = [], 0
    for T in (2, 4, 3):
        lg, kn, vn = O.prefill_with_cache(cfg, layers, embed, fnorm, ids[:, at:at + T], [at, at],
                                          k_cache, v_cache)
        k_cache[:, :, :, at:at + T] = kn                 # the caller appends
        v_cache[:, :, :, at:at + T] = vn
        outs.append(lg)
        at += T
    full = O.model_forward(cfg, layers, embed, fnorm, ids)
    np.testing.assert_allclose(np.concatenate(outs, axis=1), full, rtol=1e-11, atol=1e-12)


def test_prefill_of_one_token_is_the_decode_step():
    cfg = _chunk_cfg(no_rope_layers=(0, 1, 1), sliding_window=(2, 0, 6))
    rng = np.random.default_rng(35)
    layers = [as_block(tiny_weights(cfg, rng)) for _ in range(cfg.n_layers)]
    embed = rng.normal(0, 0.5, (cfg.vocab, cfg.hidden))
    fnorm = 1 + rng.normal(0, 0.1, cfg.hidden)
    lens = np.array([0, 4, 11])
    k_cache = rng.normal(0, 1, (cfg.n_layers, 3, cfg.n_kv_heads, 11, cfg.head_dim))
    v_cache = rng.normal(0, 1, k_cache.shape)
    ids = rng.integers(0, cfg.vocab, 3)
    lg, kn, vn = O.prefill_with_cache(cfg, layers, embed, fnorm, ids[:, None], lens, k_cache, v_cache)
    dl, dk, dv = O.decode_step(cfg, layers, embed, fnorm, ids, lens, k_cache, v_cache)
    np.testing.assert_allclose(lg[:, 0], dl, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(kn[:, :, :, 0], dk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(vn[:, :, :, 0], dv, rtol=1e-12, atol=1e-13)


def test_prefill_on_empty_caches_is_the_model_forward():
    cfg = _chunk_cfg()
    rng = np.random.default_rng(36)
    layers = [as_block(tiny_weights(cfg, rng)) for _ in range(cfg.n_layers)]
    embed = rng.normal(0, 0.5, (cfg.vocab, cfg.hidden))
    fnorm = 1 + rng.normal(0, 0.1, cfg.hidden)
    ids = rng.integers(0, cfg.vocab, (2, 6))
    cache = np.full((cfg.n_layers, 2, cfg.n_kv_heads, 4, cfg.head_dim), 55.0)   # never read
    lg, _, _ = O.prefill_with_cache(cfg, layers, embed, fnorm, ids, [0, 0], cache, cache)
    np.testing.assert_allclose(lg, O.model_forward(cfg, layers, embed, fnorm, ids), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- additive key mask
# ("model.py" (SmolLM2-135M) section 4: attention_mask of 0 / -inf added to the scores)

def test_key_mask_of_left_padding_is_valid_start():
    rng = np.random.default_rng(37)
    B, H, KV, T, hd = 3, 6, 2, 10, 4
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    vs = [0, 4, 10]
    mask = np.arange(T)[None, :] >= np.array(vs)[:, None]
    np.testing.assert_array_equal(O.gqa_attention(q, k, v, key_mask=mask), O.gqa_attention(q, k, v, vs))
    np.testing.assert_array_equal(O.gqa_attention(q, k, v, key_mask=np.ones((B, T), bool)),
                                  O.gqa_attention(q, k, v))


def test_key_mask_vs_torch_sdpa_boolean_mask():
    rng = np.random.default_rng(38)
    B, H, KV, T, hd = 2, 8, 2, 24, 16
    q, k, v = _rand_qkv(B, H, KV, T, hd, rng)
    mask = rng.random((B, T)) < 0.6
    mask[:, 0] = True                                 # every row keeps its first key
    g = H // KV
    kt = torch.tensor(k).repeat_interleave(g, dim=1)
    vt = torch.tensor(v).repeat_interleave(g, dim=1)
    allowed = torch.tril(torch.ones(T, T, dtype=torch.bool))[None, None] & torch.tensor(mask)[:, None, None, :]
    ref = F.scaled_dot_product_attention(torch.tensor(q), kt, vt, attn_mask=allowed).numpy()
    np.testing.assert_allclose(O.gqa_attention(q, k, v, key_mask=mask), ref, rtol=1e-11, atol=1e-12)
    # a row whose visible keys are all masked out gets 0
    m2 = mask.copy()
    m2[0, :3] = False
    o = O.gqa_attention(q, k, v, key_mask=m2)
    np.testing.assert_array_equal(o[0, :, :3], 0.0)


def test_key_mask_block_vs_bruteforce_loops():
    rng = np.random.default_rng(39)
    w = tiny_weights(TINY, rng)
    x = rng.normal(0, 1, (2, 7, TINY.hidden))
    mask = np.array([[1, 0, 1, 1, 0, 1, 1], [0, 0, 1, 1, 1, 0, 1]], dtype=bool)
    out = O.block_forward(TINY, as_block(w), x, key_mask=mask)
    ref = np.array(bf.block(TINY, {k: nested(a) for k, a in w.items()}, nested(x), key_mask=mask.tolist()))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
