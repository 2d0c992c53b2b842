"""Seeded synthetic workloads for the decoder forward.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA library's tests/bench and the fp64 oracle consume
what it returns, so neither side generates its own inputs.

Recipe (one ``torch.Generator`` seeded once, draws in this fixed order, each
drawn in fp32 and rounded to bf16):
  1. activations x ~ N(0, 1) [B, T, d]  (block workloads)  or token ids
     uniform in [0, V) [B, T] / [B]  (model and decode workloads);
  2. per layer: attn_norm, wq, wk, wv, wo, mlp_norm, wgate, wup, wdown
     (norm weights 1 + N(0, 0.1^2); matrices N(0, w_std^2) in [out, in] layout);
  3. embed [V, d] ~ N(0, w_std^2) and final_norm (model and decode);
  4. per-sequence lengths (left-padded block: valid lengths; decode: cache
     lengths), integers uniform over the inclusive range;
  5. decode only: cached K and V ~ N(0, 1) [L, B, KV, S_max, hd], drawn layer
     by layer (K then V).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                      # "block" | "model" | "decode"
    B: int
    T: int                         # tokens per sequence (decode: 1)
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    n_layers: int
    vocab: int                     # 0 for block workloads
    max_pos: int
    rms_eps: float
    rope_theta: float
    w_std: float
    len_range: Optional[Tuple[int, int]] = None   # inclusive; left-pad lengths or cache lengths
    s_max: int = 0                 # decode cache slots per (layer, seq, kv head)
    no_rope_layers: Optional[Tuple[int, ...]] = None   # per layer: 1 RoPE, 0 NoPE (SmolLM3)
    sliding_window: Optional[Tuple[int, ...]] = None   # per layer: 0 full causal, w > 0 window

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  Dimensions follow the SmolLM2-135M config (model.py,
# section 1), the SmolLM3 printout (nnterp encyclopedia) and the 125M-class
# block (block.py); distributions are the stated synthetic ones.
WORKLOADS: Dict[str, Workload] = {
    "smollm2_block_b1_t128": Workload(
        "smollm2_block_b1_t128", "block", B=1, T=128, hidden=576, n_heads=9, n_kv_heads=3,
        head_dim=64, intermediate=1536, n_layers=1, vocab=0, max_pos=8192,
        rms_eps=1e-5, rope_theta=1e5, w_std=0.0417),
    "smollm2_model_b8_t2048": Workload(
        "smollm2_model_b8_t2048", "model", B=8, T=2048, hidden=576, n_heads=9, n_kv_heads=3,
        head_dim=64, intermediate=1536, n_layers=30, vocab=49152, max_pos=8192,
        rms_eps=1e-5, rope_theta=1e5, w_std=0.0417),
    "smollm3_4blocks_b4_t4096": Workload(
        "smollm3_4blocks_b4_t4096", "block", B=4, T=4096, hidden=2048, n_heads=16, n_kv_heads=4,
        head_dim=128, intermediate=11008, n_layers=4, vocab=0, max_pos=65536,
        rms_eps=1e-6, rope_theta=1e6, w_std=0.02),
    "slm125m_block_leftpad_b16_t1024": Workload(
        "slm125m_block_leftpad_b16_t1024", "block", B=16, T=1024, hidden=768, n_heads=12,
        n_kv_heads=4, head_dim=64, intermediate=2048, n_layers=1, vocab=0, max_pos=8192,
        rms_eps=1e-5, rope_theta=1e4, w_std=768 ** -0.5, len_range=(128, 1024)),
    "smollm2_decode_b64_cache4096": Workload(
        "smollm2_decode_b64_cache4096", "decode", B=64, T=1, hidden=576, n_heads=9, n_kv_heads=3,
        head_dim=64, intermediate=1536, n_layers=30, vocab=49152, max_pos=8192,
        rms_eps=1e-5, rope_theta=1e5, w_std=0.0417, len_range=(1024, 4096), s_max=4096),
}

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown")


@dataclass
class Inputs:
    wl: Workload
    x: Optional[torch.Tensor] = None             # [B, T, d] bf16 (block)
    ids: Optional[torch.Tensor] = None           # int32 [B, T] (model) or [B] (decode)
    layers: List[Dict[str, torch.Tensor]] = field(default_factory=list)
    embed: Optional[torch.Tensor] = None         # [V, d] bf16
    final_norm: Optional[torch.Tensor] = None    # [d] bf16
    lengths: Optional[torch.Tensor] = None       # int32 [B]
    valid_start: Optional[torch.Tensor] = None   # int32 [B] (left-padded block)
    k_cache: Optional[torch.Tensor] = None       # [L, B, KV, S, hd] bf16 (decode)
    v_cache: Optional[torch.Tensor] = None


def _normal(gen, shape, std, mean, device):
    t = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def layer_shapes(wl: Workload) -> Dict[str, Tuple[int, ...]]:
    d, hd = wl.hidden, wl.head_dim
    return {
        "attn_norm": (d,), "wq": (wl.n_heads * hd, d), "wk": (wl.n_kv_heads * hd, d),
        "wv": (wl.n_kv_heads * hd, d), "wo": (d, wl.n_heads * hd), "mlp_norm": (d,),
        "wgate": (wl.intermediate, d), "wup": (wl.intermediate, d), "wdown": (d, wl.intermediate),
    }


def generate(wl: Workload, seed: int = 0, device="cpu") -> Inputs:
    """Draw one workload's inputs from ``seed`` on ``device`` (cpu or cuda)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    inp = Inputs(wl)
    if wl.kind == "block":
        inp.x = _normal(gen, (wl.B, wl.T, wl.hidden), 1.0, 0.0, device)
    elif wl.kind == "model":
        inp.ids = torch.randint(0, wl.vocab, (wl.B, wl.T), generator=gen, device=device).to(torch.int32)
    else:
        inp.ids = torch.randint(0, wl.vocab, (wl.B,), generator=gen, device=device).to(torch.int32)
    shapes = layer_shapes(wl)
    for _ in range(wl.n_layers):
        lw = {}
        for key in LAYER_KEYS:
            if key.endswith("norm"):
                lw[key] = _normal(gen, shapes[key], 0.1, 1.0, device)
            else:
                lw[key] = _normal(gen, shapes[key], wl.w_std, 0.0, device)
        inp.layers.append(lw)
    if wl.kind in ("model", "decode"):
        inp.embed = _normal(gen, (wl.vocab, wl.hidden), wl.w_std, 0.0, device)
        inp.final_norm = _normal(gen, (wl.hidden,), 0.1, 1.0, device)
    if wl.len_range is not None:
        lo, hi = wl.len_range
        inp.lengths = torch.randint(lo, hi + 1, (wl.B,), generator=gen, device=device).to(torch.int32)
        if wl.kind == "block":
            inp.valid_start = (wl.T - inp.lengths).to(torch.int32)
    if wl.kind == "decode":
        shape = (wl.n_layers, wl.B, wl.n_kv_heads, wl.s_max, wl.head_dim)
        inp.k_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        inp.v_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for l in range(wl.n_layers):
            inp.k_cache[l] = _normal(gen, shape[1:], 1.0, 0.0, device)
            inp.v_cache[l] = _normal(gen, shape[1:], 1.0, 0.0, device)
    return inp


def to_numpy_f32(t: torch.Tensor):
    """Exact widening of a bf16 tensor to a float32 numpy array on the host."""
    return t.detach().to("cpu", torch.float32).numpy()
