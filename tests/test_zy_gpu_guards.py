"""Every output buffer of the C ABI sits between guard regions holding a
sentinel; after each call the guards must be untouched (no kernel writes
outside the rows and columns it owns) and the outputs finite.  Shapes are
ragged so that partial tiles and per-lane tails are exercised."""
import math

import numpy as np
import pytest
import torch

from llama_decoder_forward_gb300 import synth
from parity_util import to_device

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
GUARD = 256          # elements on each side (512+ bytes: outputs stay 16-byte aligned)


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from llama_decoder_forward_gb300 import smol
    return smol


def guarded(shape, dtype, sentinel):
    """(buffer, view): a contiguous view of `shape` inside a buffer whose first
    and last GUARD elements hold `sentinel`."""
    n = math.prod(shape)
    buf = torch.full((GUARD + n + GUARD,), sentinel, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def assert_guards(buf, name):
    torch.cuda.synchronize()
    s = buf[0].item()
    head, tail = buf[:GUARD], buf[-GUARD:]
    assert bool((head == s).all()) and bool((tail == s).all()), f"{name}: a guard region was overwritten"


def assert_finite(t, name):
    assert bool(torch.isfinite(t.float()).all()), f"{name}: non-finite values"


def test_block_outputs_stay_in_bounds(S):
    wl = W["smollm2_block_b1_t128"].scaled(B=2, T=67)
    inp = to_device(synth.generate(wl, seed=80))
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, wl.B, wl.T)
    kv_shape = (wl.B, wl.n_kv_heads, wl.T, wl.head_dim)
    for dtype in (torch.bfloat16, torch.float32):
        ob, out = guarded((wl.B, wl.T, wl.hidden), dtype, -12352.0)
        kb, k_out = guarded(kv_shape, torch.bfloat16, -12352.0)
        vb, v_out = guarded(kv_shape, torch.bfloat16, -12352.0)
        S.block_forward(cfg, packed, 0, inp.x.to(dtype).contiguous(), out, ws, k_out=k_out, v_out=v_out)
        assert S.workspace_status(ws) == S.OK
        for b, name in ((ob, "out"), (kb, "k_out"), (vb, "v_out")):
            assert_guards(b, name)
        assert_finite(out, "out")


def test_model_logits_stay_in_bounds(S):
    wl = W["smollm2_model_b8_t2048"].scaled(B=3, T=37, n_layers=2, vocab=1024)
    inp = to_device(synth.generate(wl, seed=81))
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers, inp.embed, inp.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, wl.B, wl.T)
    lb, logits = guarded((wl.B, wl.T, wl.vocab), torch.bfloat16, -12352.0)
    S.model_forward(cfg, packed, inp.ids, logits, ws)
    assert S.workspace_status(ws) == S.OK
    assert_guards(lb, "logits")
    assert_finite(logits, "logits")


@pytest.mark.parametrize("B", [5, 80])
def test_decode_outputs_stay_in_bounds(S, B):
    # B = 5: narrow-unit projections; B = 80: the tile GEMM
    wl = W["smollm2_decode_b64_cache4096"].scaled(B=B, n_layers=2, s_max=96, vocab=1024)
    inp = synth.generate(wl, seed=82 + B)
    inp.lengths = torch.tensor(np.random.default_rng(B).integers(0, 97, size=B), dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_DECODE, B, 1)
    kv_shape = (wl.n_layers, B, wl.n_kv_heads, wl.head_dim)
    kb, k_new = guarded(kv_shape, torch.bfloat16, -12352.0)
    vb, v_new = guarded(kv_shape, torch.bfloat16, -12352.0)
    lb, logits = guarded((B, wl.vocab), torch.bfloat16, -12352.0)
    S.decode_step(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    for b, name in ((kb, "k_new"), (vb, "v_new"), (lb, "logits")):
        assert_guards(b, name)
    assert_finite(logits, "logits")


def test_sample_writes_one_token_per_row(S):
    B, V = 7, 3000
    g = torch.Generator().manual_seed(83)
    logits = (torch.randn(B, V, generator=g) * 2).to(torch.bfloat16).cuda()
    u = torch.rand(B, generator=g).cuda()
    nb, nxt = guarded((B,), torch.int32, -777)
    for kw in (dict(do_sample=False), dict(temperature=0.8, top_k=40, top_p=0.9)):
        S.sample(logits, nxt, u, **kw)
        assert_guards(nb, "next")
        got = nxt.cpu().numpy()
        assert np.all((got >= 0) & (got < V))
