"""ctypes binding of libsmol (include/smol.h): argument marshalling only.

Every computation runs in the library's CUDA kernels.  Importing this module
loads ``libsmol.so`` from this package directory and raises ImportError if it
has not been built (``python -c "import __graft_entry__ as g; g.build()"``);
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import POINTER, c_float, c_int, c_size_t, c_void_p
from typing import Dict, List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmol.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "smol.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libsmol.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
_lib = ctypes.CDLL(LIB_PATH)

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_TOO_LONG = -1, -2, -3, -4
ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE, ERR_TIMEOUT = -5, -6, -7, -8
ERR_RANGE, ERR_INPUT = -9, -10
OP_BLOCK, OP_MODEL, OP_DECODE = 1, 2, 3
ACT_BF16, ACT_F32 = 0, 1


class Config(ctypes.Structure):
    # no_rope_layers / sliding_window: host int32 arrays of n_layers entries or
    # NULL (assigning a ctypes array to the field keeps it alive with the struct)
    _fields_ = [("hidden", c_int), ("n_heads", c_int), ("n_kv_heads", c_int), ("head_dim", c_int),
                ("intermediate", c_int), ("n_layers", c_int), ("vocab", c_int), ("max_pos", c_int),
                ("rms_eps", c_float), ("rope_theta", c_float),
                ("no_rope_layers", POINTER(ctypes.c_int32)), ("sliding_window", POINTER(ctypes.c_int32))]


class BlockWeights(ctypes.Structure):
    _fields_ = [(k, c_void_p) for k in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate",
                                       "wup", "wdown")]


class ModelWeights(ctypes.Structure):
    _fields_ = [("layers", POINTER(BlockWeights)), ("embed", c_void_p), ("final_norm", c_void_p)]


_CFG = POINTER(Config)
_SIGS = {
    "smol_packed_bytes": (c_size_t, [_CFG, c_int, c_int]),
    "smol_prepare_weights": (c_int, [_CFG, POINTER(ModelWeights), c_int, c_void_p, c_size_t, c_void_p]),
    "smol_workspace_bytes": (c_size_t, [_CFG, c_int, c_int, c_int]),
    "smol_block_forward": (c_int, [_CFG, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "smol_model_forward": (c_int, [_CFG, c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p,
                                   c_void_p, c_size_t, c_void_p]),
    "smol_block_forward_masked": (c_int, [_CFG, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                          c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "smol_model_forward_masked": (c_int, [_CFG, c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p,
                                          c_void_p, c_size_t, c_void_p]),
    "smol_decode_step": (c_int, [_CFG, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "smol_workspace_status": (c_int, [c_void_p, c_void_p]),
    "smol_last_launch_count": (c_int, []),
    "smol_status_string": (ctypes.c_char_p, [c_int]),
    "smol_decode_step_noalloc": (c_int, [_CFG, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                         c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "smol_decode_noalloc_status": (c_int, [c_void_p]),
    "smol_set_wait_limit_ns": (None, [ctypes.c_ulonglong]),
    "smol_decode_next": (c_int, [_CFG, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                 c_void_p, c_void_p, c_void_p, c_float, c_int, c_float, c_int, c_void_p,
                                 c_void_p, c_void_p, c_size_t, c_void_p]),
    "smol_append_kv": (c_int, [_CFG, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                               c_void_p]),
    "smol_prefill_cache_workspace_bytes": (c_size_t, [_CFG, c_int, c_int, c_int]),
    "smol_prefill_with_cache": (c_int, [_CFG, c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                        c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "smol_sample": (c_int, [c_void_p, c_int, c_int, ctypes.c_longlong, c_float, c_int, c_float, c_int,
                            c_void_p, c_void_p, c_void_p]),
    "smol_profile_begin": (c_int, [ctypes.c_uint, c_int]),
    "smol_profile_end": (c_int, [POINTER(c_int), POINTER(c_float), c_int]),
}

# kernel kinds of smol_profile_begin (SMOL_K_*)
KERNEL_KINDS = ("embed", "rowstats", "qkv_gemm_rope", "flash_attention", "o_gemm_residual",
                "gateup_gemm_swiglu", "down_gemm_residual", "lm_head_gemm", "decode_attention", "other",
                "sample")
(K_EMBED, K_ROWSTATS, K_QKV, K_ATTN, K_OPROJ, K_GATEUP, K_DOWN, K_HEAD, K_DEC_ATTN, K_OTHER,
 K_SAMPLE) = range(11)
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def declared_symbols() -> List[str]:
    """Function names declared in include/smol.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(smol_\w+)\s*\(", text, re.M)))


class SmolError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({status_string(code)})")


def status_string(code: int) -> str:
    return _lib.smol_status_string(code).decode()


def _check(code: int, where: str) -> None:
    if code != OK:
        raise SmolError(code, where)


def _i32_array(vals, n_layers: int, name: str):
    if vals is None:
        return None
    vals = [int(v) for v in vals]
    if len(vals) != n_layers:
        raise ValueError(f"{name} needs one entry per layer ({n_layers}), got {len(vals)}")
    return (ctypes.c_int32 * n_layers)(*vals)


def make_config(hidden, n_heads, n_kv_heads, head_dim, intermediate, n_layers, vocab, max_pos,
                rms_eps, rope_theta, no_rope_layers=None, sliding_window=None) -> Config:
    """no_rope_layers: per layer 1 = RoPE, 0 = NoPE block (None: RoPE everywhere);
    sliding_window: per layer 0 = full causal, w > 0 = window of w keys (None: none)."""
    cfg = Config(hidden, n_heads, n_kv_heads, head_dim, intermediate, n_layers, vocab, max_pos,
                 rms_eps, rope_theta)
    nr = _i32_array(no_rope_layers, n_layers, "no_rope_layers")
    sw = _i32_array(sliding_window, n_layers, "sliding_window")
    if nr is not None:
        cfg.no_rope_layers = nr
    if sw is not None:
        cfg.sliding_window = sw
    return cfg


def config_of(wl) -> Config:
    """Config from a synth.Workload (same field names)."""
    return make_config(wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                       wl.n_layers, wl.vocab, wl.max_pos, wl.rms_eps, wl.rope_theta,
                       getattr(wl, "no_rope_layers", None), getattr(wl, "sliding_window", None))


def _p(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    return t


def packed_bytes(cfg: Config, n_layers: int, with_embed: bool) -> int:
    return _lib.smol_packed_bytes(ctypes.byref(cfg), n_layers, int(with_embed))


def workspace_bytes(cfg: Config, op: int, B: int, T: int) -> int:
    return _lib.smol_workspace_bytes(ctypes.byref(cfg), op, B, T)


def alloc_workspace(cfg: Config, op: int, B: int, T: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg, op, B, T)
    if n == 0:
        raise SmolError(ERR_UNSUPPORTED_SHAPE, "smol_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


_LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown")


def prepare_weights(cfg: Config, layers: Sequence[Dict[str, torch.Tensor]], embed=None,
                    final_norm=None, stream=None) -> torch.Tensor:
    """Packs raw bf16 weights (device tensors) into a new device buffer."""
    n_layers = len(layers)
    arr = (BlockWeights * max(n_layers, 1))()
    for i, lw in enumerate(layers):
        arr[i] = BlockWeights(*[c_void_p(_dev(lw[k], torch.bfloat16, k).data_ptr()) for k in _LAYER_KEYS])
    mw = ModelWeights(arr, _p(embed), _p(final_norm))
    if embed is not None:
        _dev(embed, torch.bfloat16, "embed")
        _dev(final_norm, torch.bfloat16, "final_norm")
    n = packed_bytes(cfg, n_layers, embed is not None)
    if n == 0:
        raise SmolError(ERR_UNSUPPORTED_SHAPE, "smol_packed_bytes")
    device = embed.device if embed is not None else layers[0]["wq"].device
    packed = torch.empty(n, dtype=torch.uint8, device=device)
    _check(_lib.smol_prepare_weights(ctypes.byref(cfg), ctypes.byref(mw), n_layers, _p(packed), n,
                                     _stream(stream)), "smol_prepare_weights")
    return packed


def block_forward(cfg: Config, packed: torch.Tensor, layer: int, x: torch.Tensor, out: torch.Tensor,
                  ws: torch.Tensor, valid_start=None, k_out=None, v_out=None, stream=None) -> None:
    B, T, _ = x.shape
    if x.dtype not in (torch.bfloat16, torch.float32) or out.dtype != x.dtype:
        raise ValueError("x and out must both be bf16 or both fp32")
    _dev(x, x.dtype, "x")
    _dev(out, x.dtype, "out")
    act = ACT_F32 if x.dtype == torch.float32 else ACT_BF16
    if valid_start is not None:
        _dev(valid_start, torch.int32, "valid_start")
    _check(_lib.smol_block_forward(ctypes.byref(cfg), _p(packed), layer, _p(x), _p(out), act, B, T,
                                   _p(valid_start), _p(k_out), _p(v_out), _p(ws), ws.numel(),
                                   _stream(stream)), "smol_block_forward")


def block_forward_masked(cfg: Config, packed: torch.Tensor, layer: int, x: torch.Tensor, out: torch.Tensor,
                         ws: torch.Tensor, key_mask: torch.Tensor, k_out=None, v_out=None, stream=None) -> None:
    """block_forward with a key mask (uint8 [B, T], nonzero = visible) in place of left padding."""
    B, T, _ = x.shape
    if x.dtype not in (torch.bfloat16, torch.float32) or out.dtype != x.dtype:
        raise ValueError("x and out must both be bf16 or both fp32")
    _dev(x, x.dtype, "x")
    _dev(out, x.dtype, "out")
    _dev(key_mask, torch.uint8, "key_mask")
    if tuple(key_mask.shape) != (B, T):
        raise ValueError("key_mask must be [B, T]")
    act = ACT_F32 if x.dtype == torch.float32 else ACT_BF16
    _check(_lib.smol_block_forward_masked(ctypes.byref(cfg), _p(packed), layer, _p(x), _p(out), act, B, T,
                                          _p(key_mask), _p(k_out), _p(v_out), _p(ws), ws.numel(),
                                          _stream(stream)), "smol_block_forward_masked")


def model_forward_masked(cfg: Config, packed: torch.Tensor, ids: torch.Tensor, logits: torch.Tensor,
                         ws: torch.Tensor, key_mask: torch.Tensor, stream=None) -> None:
    """model_forward with a key mask (uint8 [B, T], nonzero = visible) in place of left padding."""
    B, T = ids.shape
    _dev(ids, torch.int32, "ids")
    _dev(logits, torch.bfloat16, "logits")
    _dev(key_mask, torch.uint8, "key_mask")
    if tuple(key_mask.shape) != (B, T):
        raise ValueError("key_mask must be [B, T]")
    _check(_lib.smol_model_forward_masked(ctypes.byref(cfg), _p(packed), _p(ids), B, T, _p(key_mask),
                                          _p(logits), _p(ws), ws.numel(), _stream(stream)),
           "smol_model_forward_masked")


def model_forward(cfg: Config, packed: torch.Tensor, ids: torch.Tensor, logits: torch.Tensor,
                  ws: torch.Tensor, valid_start=None, stream=None) -> None:
    B, T = ids.shape
    _dev(ids, torch.int32, "ids")
    _dev(logits, torch.bfloat16, "logits")
    _check(_lib.smol_model_forward(ctypes.byref(cfg), _p(packed), _p(ids), B, T, _p(valid_start),
                                   _p(logits), _p(ws), ws.numel(), _stream(stream)),
           "smol_model_forward")


def prefill_cache_workspace(cfg: Config, B: int, T: int, S_max: int, device="cuda") -> torch.Tensor:
    n = _lib.smol_prefill_cache_workspace_bytes(ctypes.byref(cfg), B, T, S_max)
    if n == 0:
        raise SmolError(ERR_UNSUPPORTED_SHAPE, "smol_prefill_cache_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prefill_with_cache(cfg: Config, packed: torch.Tensor, ids: torch.Tensor, cache_len: torch.Tensor,
                       k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       logits: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """T new tokens per sequence on top of a KV cache (chunked prefill)."""
    B, T = ids.shape
    S_max = k_cache.shape[3]
    _dev(ids, torch.int32, "ids")
    _dev(cache_len, torch.int32, "cache_len")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new),
                    ("logits", logits)):
        _dev(t, torch.bfloat16, name)
    _check(_lib.smol_prefill_with_cache(ctypes.byref(cfg), _p(packed), _p(ids), B, T, _p(cache_len),
                                        _p(k_cache), _p(v_cache), S_max, _p(k_new), _p(v_new), _p(logits),
                                        _p(ws), ws.numel(), _stream(stream)), "smol_prefill_with_cache")


def decode_step(cfg: Config, packed: torch.Tensor, ids: torch.Tensor, cache_len: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                v_new: torch.Tensor, logits: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    B = ids.shape[0]
    S_max = k_cache.shape[3]
    _dev(ids, torch.int32, "ids")
    _dev(cache_len, torch.int32, "cache_len")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new),
                    ("logits", logits)):
        _dev(t, torch.bfloat16, name)
    _check(_lib.smol_decode_step(ctypes.byref(cfg), _p(packed), _p(ids), _p(cache_len), B,
                                 _p(k_cache), _p(v_cache), S_max, _p(k_new), _p(v_new), _p(logits),
                                 _p(ws), ws.numel(), _stream(stream)), "smol_decode_step")


def decode_step_noalloc(cfg: Config, packed: torch.Tensor, ids: torch.Tensor, cache_len: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor,
                        v_new: torch.Tensor, logits: torch.Tensor, stream=None) -> None:
    """decode_step with the library's fixed device scratch instead of a workspace
    (for callers that cannot provide device memory; calls must not overlap)."""
    B = ids.shape[0]
    S_max = k_cache.shape[3]
    _dev(ids, torch.int32, "ids")
    _dev(cache_len, torch.int32, "cache_len")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new),
                    ("logits", logits)):
        _dev(t, torch.bfloat16, name)
    _check(_lib.smol_decode_step_noalloc(ctypes.byref(cfg), _p(packed), _p(ids), _p(cache_len), B,
                                         _p(k_cache), _p(v_cache), S_max, _p(k_new), _p(v_new),
                                         _p(logits), _stream(stream)), "smol_decode_step_noalloc")


def decode_next(cfg: Config, packed: torch.Tensor, ids: torch.Tensor, cache_len: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                next_ids: torch.Tensor, ws: torch.Tensor, logits: Optional[torch.Tensor] = None,
                uniform: Optional[torch.Tensor] = None, temperature: float = 1.0, top_k: int = 0,
                top_p: float = 1.0, do_sample: bool = False, stream=None) -> None:
    """The decode step and the next-token choice (greedy inside the head GEMM's
    epilogue; sampling through the choice kernel over `logits`)."""
    B = ids.shape[0]
    S_max = k_cache.shape[3]
    _dev(ids, torch.int32, "ids")
    _dev(cache_len, torch.int32, "cache_len")
    _dev(next_ids, torch.int32, "next_ids")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new)):
        _dev(t, torch.bfloat16, name)
    if logits is not None:
        _dev(logits, torch.bfloat16, "logits")
    if uniform is not None:
        _dev(uniform, torch.float32, "uniform")
    _check(_lib.smol_decode_next(ctypes.byref(cfg), _p(packed), _p(ids), _p(cache_len), B, _p(k_cache),
                                 _p(v_cache), S_max, _p(k_new), _p(v_new), _p(logits), float(temperature),
                                 int(top_k), float(top_p), int(bool(do_sample)), _p(uniform), _p(next_ids),
                                 _p(ws), ws.numel(), _stream(stream)), "smol_decode_next")


def append_kv(cfg: Config, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, cache_len: torch.Tensor, stream=None) -> None:
    """Appends a decode step's new keys/values at slot cache_len[b] and increments cache_len."""
    B = cache_len.shape[0]
    S_max = k_cache.shape[3]
    for name, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, torch.bfloat16, name)
    _dev(cache_len, torch.int32, "cache_len")
    _check(_lib.smol_append_kv(ctypes.byref(cfg), B, _p(k_new), _p(v_new), _p(k_cache), _p(v_cache), S_max,
                               _p(cache_len), _stream(stream)), "smol_append_kv")


def sample(logits: torch.Tensor, next_ids: torch.Tensor, uniform: Optional[torch.Tensor] = None,
           temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0, do_sample: bool = True,
           stream=None) -> None:
    """Next token of each row of logits [B, V] (bf16, rows may be strided) into
    next_ids [B] (int32); uniform [B] fp32 in [0, 1) unless greedy."""
    if logits.dim() != 2 or logits.dtype != torch.bfloat16 or not logits.is_cuda or logits.stride(1) != 1:
        raise ValueError("logits must be a CUDA bf16 [B, V] tensor with unit column stride")
    B, V = logits.shape
    _dev(next_ids, torch.int32, "next_ids")
    if uniform is not None:
        _dev(uniform, torch.float32, "uniform")
    _check(_lib.smol_sample(_p(logits), B, V, logits.stride(0), float(temperature), int(top_k),
                            float(top_p), int(bool(do_sample)), _p(uniform), _p(next_ids),
                            _stream(stream)), "smol_sample")


def set_wait_limit_ns(ns: int) -> None:
    """Failure-path tests only: bounded-wait limit of the prefill attention
    kernel for later launches (0 restores the default of 1 s)."""
    _lib.smol_set_wait_limit_ns(int(ns))


def decode_noalloc_status(stream=None) -> int:
    """Synchronising read (and reset) of the status word of decode_step_noalloc."""
    return _lib.smol_decode_noalloc_status(_stream(stream))


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronising read (and reset) of the kernels' status word."""
    return _lib.smol_workspace_status(_p(ws), _stream(stream))


def last_launch_count() -> int:
    return _lib.smol_last_launch_count()


def profile_begin(kind_mask: int, capacity: int) -> None:
    """Start per-launch event timing of the kernel kinds in kind_mask."""
    _check(_lib.smol_profile_begin(kind_mask, capacity), "smol_profile_begin")


def profile_end(cap: int = 65536):
    """Stop timing; returns [(kind, milliseconds), ...] in launch order."""
    kinds = (c_int * cap)()
    ms = (c_float * cap)()
    n = _lib.smol_profile_end(kinds, ms, cap)
    if n < 0:
        raise SmolError(n, "smol_profile_end")
    return [(kinds[i], ms[i]) for i in range(n)]


raw = _lib   # the C entry points themselves, for callers that marshal by hand
