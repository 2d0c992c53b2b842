"""Helpers shared by the parity tests: oracle inputs from synthetic workloads
and the acceptance metrics (max error relative to the oracle's RMS, cosine)."""
from __future__ import annotations

import numpy as np
import torch

from llama_decoder_forward_gb300 import synth
from oracle import oracle as O

# Acceptance bars: a block's outputs within 2e-2 x RMS(oracle output); the
# full model's logits with cosine >= 0.999 and max |err| <= 5e-2.  An output
# stored in bf16 additionally carries its own rounding, at most half an ulp,
# i.e. 2^-8 of its magnitude; that allowance is added for bf16 outputs.
BLOCK_REL_TOL = 2e-2
BF16_HALF_ULP_REL = 2.0 ** -8
LOGITS_COS_MIN = 0.999
LOGITS_MAX_ABS = 5e-2


def oracle_config(wl: synth.Workload, n_layers=None) -> O.Config:
    return O.Config(hidden=wl.hidden, n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads,
                    head_dim=wl.head_dim, intermediate=wl.intermediate,
                    n_layers=n_layers if n_layers is not None else wl.n_layers,
                    vocab=wl.vocab, max_pos=wl.max_pos, rms_eps=wl.rms_eps, rope_theta=wl.rope_theta,
                    no_rope_layers=wl.no_rope_layers, sliding_window=wl.sliding_window)


def np32(t: torch.Tensor) -> np.ndarray:
    return synth.to_numpy_f32(t)


def oracle_layers(inp: synth.Inputs, n=None):
    layers = inp.layers if n is None else inp.layers[:n]
    return [O.BlockWeights(**{k: np32(v) for k, v in lw.items()}) for lw in layers]


def rel_max_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(got - ref)) / rms)


def rel_max_err_bf16_out(got, ref) -> float:
    """max(|got - ref| - 2^-8 |ref|) / RMS(ref): the error left after allowing
    the rounding of a bf16 output."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(got - ref) - BF16_HALF_ULP_REL * np.abs(ref)) / rms)


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def to_device(inp: synth.Inputs, device="cuda") -> synth.Inputs:
    out = synth.Inputs(inp.wl)
    mv = lambda t: None if t is None else t.to(device)
    out.x, out.ids, out.embed, out.final_norm = mv(inp.x), mv(inp.ids), mv(inp.embed), mv(inp.final_norm)
    out.lengths, out.valid_start = mv(inp.lengths), mv(inp.valid_start)
    out.k_cache, out.v_cache = mv(inp.k_cache), mv(inp.v_cache)
    out.layers = [{k: v.to(device) for k, v in lw.items()} for lw in inp.layers]
    return out
