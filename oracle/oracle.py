"""fp64 CPU oracle for the pre-norm LLaMA decoder forward (SmolLM2-135M family).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library and imports
nothing from the ``llama_decoder_forward_gb300`` package.

Every function is the plain definition of one step, written in numpy float64
with no intermediate rounding.  Inputs are whatever the caller passes (the
bf16 values the GPU also sees, widened exactly); all arithmetic is fp64.
A library primitive (``numpy.matmul``) serves as the matrix-product step.

Sources (web pages describing the method, cited by title and section):
  [M1] "model.py" - minimal SmolLM2-135M style model (Sualeh77 Space):
       sections 1 Config, 2 RMSNorm, 3 RoPE, 4 Attention, 5 MLP (SwiGLU),
       6 Transformer Block, 7 Top-level SmolLM2-135M, 8 Quick self-test.
  [M3] "SmolLM3" (nnterp encyclopedia): "The block, in order",
       "Every fourth block has no rotary", "On a NoPE block the queries and
       keys are the projections", "Grouped-query attention", "A sliding window
       the 3B checkpoints leave off", "The readout, the embeddings and the
       tokenizer".
  [M4] "model.py" - complete SmolLM2-135M implementation (abi96062):
       module docstring (parameter total), SmolLM2Model.forward.
  [M5] "components.py" (abi96062): RMSNorm, RotaryEmbedding,
       GroupedQueryAttention, SwiGLU_FFN, TransformerBlock.

Readings taken where the pages are silent or disagree (also listed in the
design notes):
  * RoPE angles come from exact integer positions in fp64 (the first model.py
    builds its cos/sin table in the model dtype, which cannot hold positions
    above 256 exactly; components.py builds it in fp32).
  * Query head h reads key/value head h // (H / KV)  (repeat_interleave in
    [M1] section 4 and [M5] GroupedQueryAttention; "h // 4" in [M3]).
  * A key j is masked for query t iff j > t (causal) or j < valid_start[b]
    (left padding).  A query row with every key masked (a padding row) gets
    an attention output of exactly 0.
  * Left padding: position id of token t of sequence b is t - valid_start[b];
    padding rows take position 0 (their values never reach a valid row).
  * NoPE blocks ([M3] "Every fourth block has no rotary"): a per-block flag
    list with the meaning of the SmolLM3 config's no_rope_layers (1 = the
    block rotates q and k, 0 = it does not); absent = every block rotates.
  * Sliding window ([M3] "A sliding window the 3B checkpoints leave off"
    names the setting, not its bounds): a window of w on a block lets query t
    see the w most recent keys, its own included, i.e. keys j with
    t - w < j <= t, on top of the causal and padding masks; 0 = no window.
    In decode the new token at position L sees cached slots j >= L - w + 1
    plus itself.
  * Prefill with a past ([M1] sections 4 and 7 with past_key_values and
    T > 1): the page drops the causal mask whenever a past exists, which
    would let a new token see the ones after it; the reading taken is the
    causal mask offset by the past: new token t of sequence b sits at
    position cache_len[b] + t and sees the cached slots [0, cache_len[b])
    and the new tokens 0 .. t (window limits as above).  Cache lengths are
    per sequence, as in decode.
  * Additive attention mask ([M1] section 4, attention_mask of 0 / -inf over
    the keys): a key j of sequence b is hidden iff the mask is -inf there,
    on top of the causal mask; positions stay 0 .. T-1 (the page derives no
    positions from it); a row with no visible key gets attention output 0.
  * Next-token choice ([M1] section 7 generate; [M4] generate): greedy is the
    first index of the row maximum; the multinomial draw is the inverse CDF
    in vocabulary order of a uniform number u in [0, 1) that the caller
    passes in (the pages call torch.multinomial, whose internal method they
    do not give); the top-p sort puts equal logits in ascending index order
    (the pages' torch.sort leaves their order open).
  * Decode: the cache holds post-RoPE keys (stored "after RoPE, before GQA
    expansion" in [M1] section 4); only the new token's q and k are rotated,
    at position cache_len[b]; with a single new token no causal mask applies
    ([M1] section 4, the ``past_key_value`` branch).

Parity status: every function below is pinned by tests that do not re-type
its formula (closed forms, invariants, brute force, torch library routines,
the parameter total printed in [M4]).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np

F64 = np.float64


@dataclass
class Config:
    """Model dimensions ([M1] section 1 Config; [M3] printout)."""

    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    n_layers: int
    vocab: int
    max_pos: int
    rms_eps: float
    rope_theta: float
    # [M3] "Every fourth block has no rotary": one flag per block, 1 where the
    # block applies the rotary and 0 on a NoPE block; None = rotary everywhere
    no_rope_layers: Optional[Tuple[int, ...]] = None
    # [M3] "A sliding window ...": per block, 0 = full causal attention, w > 0 =
    # query t sees keys t - w < j <= t; None = no window on any block
    sliding_window: Optional[Tuple[int, ...]] = None


def block_kind(cfg: Config, layer: int) -> Tuple[bool, int]:
    """(applies the rotary, window) of block ``layer`` ([M3] "Every fourth
    block has no rotary", "A sliding window the 3B checkpoints leave off")."""
    rope = True if cfg.no_rope_layers is None else bool(cfg.no_rope_layers[layer])
    window = 0 if cfg.sliding_window is None else int(cfg.sliding_window[layer])
    return rope, window


SMOLLM2_135M = Config(hidden=576, n_heads=9, n_kv_heads=3, head_dim=64,
                      intermediate=1536, n_layers=30, vocab=49152, max_pos=8192,
                      rms_eps=1e-5, rope_theta=100000.0)


def param_count(cfg: Config, tied: bool = True) -> int:
    """Number of parameters of the decoder with a tied head.

    [M1] section 1 (no biases anywhere), sections 4-7 (module shapes);
    [M4] module docstring gives the SmolLM2-135M total.
    """
    d, hd, H, KV, I = cfg.hidden, cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.intermediate
    per_block = (d                       # attn_norm weight
                 + H * hd * d            # q_proj
                 + 2 * KV * hd * d       # k_proj, v_proj
                 + d * H * hd            # o_proj
                 + d                     # mlp_norm weight
                 + 3 * d * I)            # gate, up, down
    embed = cfg.vocab * d
    head = 0 if tied else cfg.vocab * d
    return embed + cfg.n_layers * per_block + d + head   # + final norm


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


def rms_norm(x, w, eps: float) -> np.ndarray:
    """y = w * x / sqrt(mean(x^2) + eps) over the last axis; no centering, no bias.

    [M1] section 2 RMSNorm; [M5] RMSNorm (its stated formula).
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return _f64(w) * (x / np.sqrt(ms + eps))


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """inv_freq[i] = theta^(-2i/head_dim), i in [0, head_dim/2).

    [M1] section 3 rope_freqs writes theta^(-i/half); [M5] RotaryEmbedding
    writes theta^(-2i/dim).  The two are the same number.
    """
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * i / head_dim)


def apply_rope(x, pos, theta: float) -> np.ndarray:
    """Non-interleaved ("rotate_half") rotary embedding.

    x: [..., T, hd] and pos: an integer array broadcastable to x.shape[:-1].
    The pair (x_i, x_{i+hd/2}) is rotated by angle pos * inv_freq[i]:
      y_i         = x_i c - x_{i+hd/2} s
      y_{i+hd/2}  = x_i s + x_{i+hd/2} c
    [M1] section 3 apply_rope; [M5] rotate_half / apply_rotary_pos_emb.
    """
    x = _f64(x)
    hd = x.shape[-1]
    half = hd // 2
    ang = _f64(pos)[..., None] * rope_inv_freq(hd, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def silu(z) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z))  ([M1] section 5; [M5] SwiGLU_FFN)."""
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def linear(x, w) -> np.ndarray:
    """nn.Linear without bias: y = x W^T with W stored [out, in] ([M1] section 4)."""
    return np.matmul(_f64(x), _f64(w).T)


def positions(B: int, T: int, valid_start=None) -> np.ndarray:
    """Position ids [B, T]: t - valid_start[b] (0 at the first valid token).

    Default (no padding) is arange(T) ([M4] SmolLM2Model.forward position_ids;
    [M5] RotaryEmbedding).  Padding rows (t < valid_start[b]) get position 0.
    """
    t = np.arange(T)[None, :].repeat(B, axis=0)
    if valid_start is None:
        return t
    vs = np.asarray(valid_start).reshape(B, 1)
    return np.maximum(t - vs, 0)


def gqa_attention(q, k, v, valid_start=None, window: int = 0, key_mask=None) -> np.ndarray:
    """Causal grouped-query softmax attention.

    q: [B, H, T, hd]; k, v: [B, KV, S, hd] with S == T (prefill).
    o[b,h,t] = sum_{j valid, j<=t} softmax_j(q[b,h,t].k[b,h//g,j] / sqrt(hd)) v[b,h//g,j]
    A row with no valid key returns 0.  With window w > 0 a key is also
    masked when j <= t - w.  key_mask [B, S] (optional, bool, True = visible)
    hides the keys where it is False ([M1] section 4 attention_mask).
    [M1] section 4 (scores / sqrt(head_dim), triu(1) causal mask, additive
    padding mask, softmax, probs @ v); [M3] "Grouped-query attention" and
    "A sliding window the 3B checkpoints leave off".
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, hd = q.shape
    KV = k.shape[1]
    g = H // KV
    t_idx = np.arange(T)[:, None]
    j_idx = np.arange(k.shape[2])[None, :]
    out = np.zeros_like(q)
    for b in range(B):
        vs = 0 if valid_start is None else int(valid_start[b])
        masked = (j_idx > t_idx) | (j_idx < vs)
        if window > 0:
            masked = masked | (j_idx <= t_idx - window)
        if key_mask is not None:
            masked = masked | ~np.asarray(key_mask[b], dtype=bool)[None, :]
        for h in range(H):
            kvh = h // g
            s = np.matmul(q[b, h], k[b, kvh].T) / np.sqrt(F64(hd))
            s = np.where(masked, -np.inf, s)
            row_max = np.max(s, axis=-1, keepdims=True)
            live = np.isfinite(row_max[:, 0])
            e = np.zeros_like(s)
            e[live] = np.exp(s[live] - row_max[live])
            den = np.sum(e, axis=-1, keepdims=True)
            p = np.zeros_like(s)
            p[live] = e[live] / den[live]
            out[b, h] = np.matmul(p, v[b, kvh])
    return out


@dataclass
class BlockWeights:
    """One decoder block; every matrix is nn.Linear layout [out, in]."""

    attn_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    mlp_norm: np.ndarray
    wgate: np.ndarray
    wup: np.ndarray
    wdown: np.ndarray


def block_forward(cfg: Config, w: BlockWeights, x, valid_start=None,
                  taps: Optional[Dict[str, np.ndarray]] = None, layer: int = 0,
                  key_mask=None) -> np.ndarray:
    """Pre-norm decoder block on x [B, T, d]; ``layer`` selects the block's
    NoPE flag and window from cfg.

    h   = x + O(attn(RoPE(Q, K), V)) with Q, K, V projections of RMSNorm1(x)
    out = h + Down(SiLU(Gate(RMSNorm2(h))) * Up(RMSNorm2(h)))
    On a NoPE block Q and K enter attention unrotated ([M3] "On a NoPE block
    the queries and keys are the projections").
    [M1] section 6 SmolBlock; [M3] "The block, in order"; [M5] TransformerBlock.
    ``taps`` (optional) receives the named intermediates used by [M3].
    ``key_mask`` [B, T] (optional, True = visible) is the additive 0 / -inf
    attention_mask of [M1] section 4 in boolean form.
    """
    x = _f64(x)
    B, T, d = x.shape
    H, KV, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    pos = positions(B, T, valid_start)

    n = rms_norm(x, w.attn_norm, cfg.rms_eps)
    q = linear(n, w.wq).reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    k = linear(n, w.wk).reshape(B, T, KV, hd).transpose(0, 2, 1, 3)
    v = linear(n, w.wv).reshape(B, T, KV, hd).transpose(0, 2, 1, 3)
    rope, window = block_kind(cfg, layer)
    if rope:
        q = apply_rope(q, pos[:, None, :], cfg.rope_theta)
        k = apply_rope(k, pos[:, None, :], cfg.rope_theta)
    o = gqa_attention(q, k, v, valid_start, window, key_mask)
    o_tok = o.transpose(0, 2, 1, 3).reshape(B, T, H * hd)
    attn_out = linear(o_tok, w.wo)
    h = x + attn_out

    m = rms_norm(h, w.mlp_norm, cfg.rms_eps)
    act = silu(linear(m, w.wgate)) * linear(m, w.wup)
    mlp_out = linear(act, w.wdown)
    out = h + mlp_out

    if taps is not None:
        taps.update(layer_input=x, attention_norm_output=n, attention_queries=q,
                    attention_keys=k, attention_values=v, attention_head_outputs=o_tok,
                    attention_output=attn_out, layer_mid=h, mlp_norm_output=m,
                    mlp_neurons=act, mlp_output=mlp_out, layer_output=out)
    return out


def lm_head(cfg: Config, x, final_norm, embed) -> np.ndarray:
    """logits = RMSNorm_f(x) E^T, the head tied to the embedding table.

    [M1] section 7 (``lm_head.weight = embed_tokens.weight``); [M3] "The readout".
    """
    return linear(rms_norm(x, final_norm, cfg.rms_eps), embed)


def model_forward(cfg: Config, layers: List[BlockWeights], embed, final_norm, ids,
                  valid_start=None, taps: Optional[Dict[str, np.ndarray]] = None,
                  key_mask=None) -> np.ndarray:
    """Embedding -> L blocks -> final norm -> tied head; logits [B, T, V].

    [M1] section 7 SmolLM2.forward (including its max-position assertion);
    [M4] SmolLM2Model.forward.
    """
    ids = np.asarray(ids)
    B, T = ids.shape
    if T > cfg.max_pos:
        raise ValueError("sequence longer than max_position_embeddings")
    x = _f64(embed)[ids]
    for l, w in enumerate(layers):
        x = block_forward(cfg, w, x, valid_start, layer=l, key_mask=key_mask)
    if taps is not None:
        taps["final_norm_output"] = rms_norm(x, final_norm, cfg.rms_eps)
    logits = lm_head(cfg, x, final_norm, embed)
    if taps is not None:
        taps["logits"] = logits
    return logits


def decode_step(cfg: Config, layers: List[BlockWeights], embed, final_norm, ids,
                cache_len, k_cache, v_cache):
    """One KV-cache decode step for B sequences, one new token each.

    ids [B]; cache_len [B]; k_cache, v_cache [L, B, KV, S, hd] holding post-RoPE
    keys and values in slots [0, cache_len[b]).  The new token sits at position
    cache_len[b]; it attends over the cached entries plus its own key/value,
    with no further mask.  Returns (logits [B, V], k_new [L, B, KV, hd],
    v_new [L, B, KV, hd]); k_new is post-RoPE (unrotated on a NoPE block).
    A block with window w attends over the cached slots j >= cache_len[b] - w + 1
    only.
    [M1] section 4 (cache concat, ``past_key_value`` branch) and section 7
    (``generate``: RoPE rows sliced at past_len); [M3] NoPE blocks and windows.
    """
    ids = np.asarray(ids)
    cache_len = np.asarray(cache_len)
    B = ids.shape[0]
    H, KV, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    g = H // KV
    L = len(layers)
    if np.any(cache_len + 1 > cfg.max_pos):
        raise ValueError("cache_len + 1 exceeds max_position_embeddings")
    x = _f64(embed)[ids]                                   # [B, d]
    k_new = np.zeros((L, B, KV, hd))
    v_new = np.zeros((L, B, KV, hd))
    for l, w in enumerate(layers):
        n = rms_norm(x, w.attn_norm, cfg.rms_eps)
        rope, window = block_kind(cfg, l)
        pos = cache_len[:, None]                           # [B, 1] broadcast over heads
        q = linear(n, w.wq).reshape(B, H, hd)
        k = linear(n, w.wk).reshape(B, KV, hd)
        if rope:
            q = apply_rope(q, pos, cfg.rope_theta)
            k = apply_rope(k, pos, cfg.rope_theta)
        v = linear(n, w.wv).reshape(B, KV, hd)
        k_new[l], v_new[l] = k, v
        o = np.zeros((B, H, hd))
        for b in range(B):
            Lb = int(cache_len[b])
            first = max(0, Lb - window + 1) if window > 0 else 0
            for h in range(H):
                kvh = h // g
                keys = np.concatenate([_f64(k_cache[l, b, kvh, first:Lb]), k[b, kvh][None]], axis=0)
                vals = np.concatenate([_f64(v_cache[l, b, kvh, first:Lb]), v[b, kvh][None]], axis=0)
                s = np.matmul(keys, q[b, h]) / np.sqrt(F64(hd))
                e = np.exp(s - np.max(s))
                o[b, h] = np.matmul(e / np.sum(e), vals)
        x = x + linear(o.reshape(B, H * hd), w.wo)
        m = rms_norm(x, w.mlp_norm, cfg.rms_eps)
        x = x + linear(silu(linear(m, w.wgate)) * linear(m, w.wup), w.wdown)
    return lm_head(cfg, x, final_norm, embed), k_new, v_new


def prefill_with_cache(cfg: Config, layers: List[BlockWeights], embed, final_norm, ids,
                       cache_len, k_cache, v_cache):
    """T new tokens per sequence on top of a KV cache (chunked prefill).

    ids [B, T]; cache_len [B]; k_cache, v_cache [L, B, KV, S, hd] holding
    post-RoPE keys and values in slots [0, cache_len[b]).  New token t of
    sequence b sits at position cache_len[b] + t and attends over the cached
    slots (those inside its block's window) and the new tokens 0 .. t.
    Returns (logits [B, T, V], k_new [L, B, KV, T, hd], v_new [L, B, KV, T, hd]),
    k_new post-RoPE (unrotated on a NoPE block): what a caller appends.
    [M1] section 4 (cache concat; the causal mask offset by the past, see the
    readings above) and section 7 (RoPE rows sliced at past_len).
    """
    ids = np.asarray(ids)
    cache_len = np.asarray(cache_len)
    B, T = ids.shape
    H, KV, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    g = H // KV
    L = len(layers)
    if np.any(cache_len + T > cfg.max_pos):
        raise ValueError("cache_len + T exceeds max_position_embeddings")
    x = _f64(embed)[ids]                                   # [B, T, d]
    k_new = np.zeros((L, B, KV, T, hd))
    v_new = np.zeros((L, B, KV, T, hd))
    t_idx = np.arange(T)
    for l, w in enumerate(layers):
        rope, window = block_kind(cfg, l)
        n = rms_norm(x, w.attn_norm, cfg.rms_eps)
        q = linear(n, w.wq).reshape(B, T, H, hd).transpose(0, 2, 1, 3)
        k = linear(n, w.wk).reshape(B, T, KV, hd).transpose(0, 2, 1, 3)
        v = linear(n, w.wv).reshape(B, T, KV, hd).transpose(0, 2, 1, 3)
        if rope:
            pos = (cache_len[:, None] + t_idx[None, :])[:, None, :]   # [B, 1, T]
            q = apply_rope(q, pos, cfg.rope_theta)
            k = apply_rope(k, pos, cfg.rope_theta)
        k_new[l], v_new[l] = k, v
        o = np.zeros((B, H, T, hd))
        for b in range(B):
            Lb = int(cache_len[b])
            keys_all = np.concatenate([_f64(k_cache[l, b, :, :Lb]), k[b]], axis=1)   # [KV, Lb+T, hd]
            vals_all = np.concatenate([_f64(v_cache[l, b, :, :Lb]), v[b]], axis=1)
            j_pos = np.arange(Lb + T)[None, :]             # key positions
            q_pos = (Lb + t_idx)[:, None]                  # query positions
            masked = j_pos > q_pos
            if window > 0:
                masked = masked | (j_pos <= q_pos - window)
            for h in range(H):
                kvh = h // g
                sc = np.matmul(q[b, h], keys_all[kvh].T) / np.sqrt(F64(hd))
                sc = np.where(masked, -np.inf, sc)
                e = np.exp(sc - np.max(sc, axis=-1, keepdims=True))
                o[b, h] = np.matmul(e / np.sum(e, axis=-1, keepdims=True), vals_all[kvh])
        x = x + linear(o.transpose(0, 2, 1, 3).reshape(B, T, H * hd), w.wo)
        m = rms_norm(x, w.mlp_norm, cfg.rms_eps)
        x = x + linear(silu(linear(m, w.wgate)) * linear(m, w.wup), w.wdown)
    return lm_head(cfg, x, final_norm, embed), k_new, v_new


def _softmax_1d(z) -> np.ndarray:
    """softmax over a 1-D array in which -inf entries get probability 0."""
    z = _f64(z)
    m = np.max(z)
    e = np.exp(z - m)
    return e / np.sum(e)


def sample_next(logits, temperature: float = 1.0, top_k: Optional[int] = None,
                top_p: Optional[float] = None, u=None, do_sample: bool = True) -> np.ndarray:
    """Next token of each row of logits [B, V], as the pages' ``generate`` picks it.

    [M1] section 7 generate and [M4] generate, step by step:
      1. greedy when do_sample is false or temperature is 0 (here: <= 0):
         argmax of the row, the first index among equal maxima;
      2. z = logits / temperature;
      3. top_k > 0: entries with z below the k-th largest z (k clipped to V)
         are set to -inf, so values equal to the k-th stay;
      4. top_p < 1: sort z descending (equal values by ascending index), take
         the cumulative softmax probabilities, remove sorted positions whose
         cumulative probability exceeds top_p after shifting that flag one
         place right (the first position is never removed);
      5. probs = softmax(z); the token is the first index i with
         sum_{j <= i} probs[j] > u[b] (inverse CDF in vocabulary order).
    Returns int64 [B].
    """
    logits = _f64(logits)
    B, V = logits.shape
    out = np.zeros(B, dtype=np.int64)
    for b in range(B):
        row = logits[b]
        if not do_sample or temperature <= 0:
            out[b] = int(np.argmax(row))
            continue
        z = row / F64(temperature)
        if top_k is not None and top_k > 0:
            k = min(int(top_k), V)
            kth = np.sort(z)[::-1][k - 1]
            z = np.where(z < kth, -np.inf, z)
        if top_p is not None and top_p < 1.0:
            order = np.argsort(-z, kind="stable")
            cum = np.cumsum(_softmax_1d(z[order]))
            remove = cum > top_p
            remove[1:] = remove[:-1].copy()
            remove[0] = False
            z = z.copy()
            z[order[remove]] = -np.inf
        probs = _softmax_1d(z)
        cdf = np.cumsum(probs)
        i = int(np.searchsorted(cdf, F64(u[b]), side="right"))
        last = int(np.nonzero(probs > 0)[0][-1])
        out[b] = min(i, last)                  # u within rounding of 1: the last token
    return out
