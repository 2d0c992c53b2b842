"""The status word's failure paths on the GPU: values beyond the f16 range of
the residual stream, clamped input values, and a bounded wait that gives up.
Each case checks that the code is reported (instead of a silent wrong result)
and that a normal call right after it succeeds and matches the oracle."""
import numpy as np
import pytest
import torch

from llama_decoder_forward_gb300 import synth
from oracle import oracle as O
from parity_util import (BLOCK_REL_TOL, LOGITS_COS_MIN, LOGITS_MAX_ABS, cosine, max_abs, np32,
                         oracle_config, oracle_layers, rel_max_err, to_device)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from llama_decoder_forward_gb300 import smol
    return smol


def _block(S, T=160, B=2, seed=30):
    wl = W["smollm2_block_b1_t128"].scaled(B=B, T=T)
    inp = synth.generate(wl, seed=seed)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, B, T)
    return wl, inp, dev, cfg, packed, ws


def _normal_block_call(S, wl, inp, dev, cfg, packed, ws):
    x = dev.x.float().contiguous()
    out = torch.empty_like(x)
    S.block_forward(cfg, packed, 0, x, out, ws)
    assert S.workspace_status(ws) == S.OK
    ref = O.block_forward(oracle_config(wl), oracle_layers(inp)[0], np32(inp.x))
    assert rel_max_err(out.cpu().numpy(), ref) <= BLOCK_REL_TOL


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_input_beyond_f16_range(S, dtype):
    # the residual stream and the projections' operands are f16: an input
    # row with values past 65504 is reported, not turned silently into inf
    wl, inp, dev, cfg, packed, ws = _block(S)
    x = dev.x.to(dtype).clone()
    x[1, 7, 3] = 1.0e5
    out = torch.empty_like(x)
    S.block_forward(cfg, packed, 0, x, out, ws)
    assert S.workspace_status(ws) == S.ERR_RANGE
    _normal_block_call(S, wl, inp, dev, cfg, packed, ws)


def test_block_residual_overflow(S):
    # inputs inside the range, but an O projection scaled so that the residual
    # h = x + o Wo^T (f16 inside the block) leaves it: the residual epilogue
    # reports it (the packed weights themselves, ~4e3, are still f16 values)
    wl, inp, dev, cfg, packed, ws = _block(S)
    layers = [dict(lw) for lw in dev.layers]
    layers[0]["wo"] = (layers[0]["wo"].float() * 1.0e5).to(torch.bfloat16)
    big = S.prepare_weights(cfg, layers)
    x = dev.x.float().contiguous()
    out = torch.empty_like(x)
    S.block_forward(cfg, big, 0, x, out, ws)
    assert S.workspace_status(ws) == S.ERR_RANGE
    _normal_block_call(S, wl, inp, dev, cfg, packed, ws)


def test_block_left_padding_start_out_of_range(S):
    wl, inp, dev, cfg, packed, ws = _block(S)
    out = torch.empty_like(dev.x)
    vs = torch.tensor([0, wl.T + 5], dtype=torch.int32, device="cuda")
    S.block_forward(cfg, packed, 0, dev.x, out, ws, valid_start=vs)
    assert S.workspace_status(ws) == S.ERR_INPUT
    _normal_block_call(S, wl, inp, dev, cfg, packed, ws)


def test_model_token_id_out_of_range(S):
    wl = W["smollm2_model_b8_t2048"].scaled(B=2, T=40, n_layers=1, vocab=512)
    inp = synth.generate(wl, seed=31)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, wl.B, wl.T)
    logits = torch.empty(wl.B, wl.T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    bad = dev.ids.clone()
    bad[1, 3] = wl.vocab
    S.model_forward(cfg, packed, bad, logits, ws)
    assert S.workspace_status(ws) == S.ERR_INPUT
    bad[1, 3] = -1
    S.model_forward(cfg, packed, bad, logits, ws)
    assert S.workspace_status(ws) == S.ERR_INPUT
    S.model_forward(cfg, packed, dev.ids, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref = O.model_forward(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                          inp.ids.numpy().astype(np.int64))
    got = np32(logits)
    assert cosine(got, ref) >= LOGITS_COS_MIN and max_abs(got, ref) <= LOGITS_MAX_ABS


def test_decode_cache_length_out_of_range(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(B=3, n_layers=1, s_max=96, vocab=512)
    inp = synth.generate(wl, seed=32)
    inp.lengths = torch.tensor([5, 96, 40], dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_DECODE, wl.B, 1)
    k_new = torch.empty(1, 3, wl.n_kv_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(3, wl.vocab, dtype=torch.bfloat16, device="cuda")
    for bad in ([5, 97, 40], [-3, 10, 40]):
        S.decode_step(cfg, packed, dev.ids, torch.tensor(bad, dtype=torch.int32, device="cuda"),
                      dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
        assert S.workspace_status(ws) == S.ERR_INPUT, bad
    S.decode_step(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref, _, _ = O.decode_step(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                              inp.ids.numpy().astype(np.int64), inp.lengths.numpy(), np32(inp.k_cache),
                              np32(inp.v_cache))
    got = np32(logits)
    assert cosine(got, ref) >= LOGITS_COS_MIN and max_abs(got, ref) <= LOGITS_MAX_ABS


def test_prefill_with_cache_length_out_of_range(S):
    # a cache length beyond what the call can hold (S_max, and max_pos - T for
    # the new tokens' positions) or below 0 is clamped on the device and reported
    wl = W["smollm2_decode_b64_cache4096"].scaled(B=2, n_layers=1, s_max=96, vocab=512)
    inp = synth.generate(wl, seed=33)
    T = 12
    g = torch.Generator().manual_seed(34)
    ids = torch.randint(0, wl.vocab, (wl.B, T), generator=g).to(torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.prefill_cache_workspace(cfg, wl.B, T, wl.s_max)
    k_new = torch.empty(1, wl.B, wl.n_kv_heads, T, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(wl.B, T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    for bad in ([97, 10], [-1, 10]):
        S.prefill_with_cache(cfg, packed, ids.cuda(), torch.tensor(bad, dtype=torch.int32, device="cuda"),
                             dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
        assert S.workspace_status(ws) == S.ERR_INPUT, bad
    lens = [96, 10]
    S.prefill_with_cache(cfg, packed, ids.cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda"),
                         dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref, _, _ = O.prefill_with_cache(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                                     ids.numpy().astype(np.int64), np.asarray(lens), np32(inp.k_cache),
                                     np32(inp.v_cache))
    got = np32(logits)
    assert cosine(got, ref) >= LOGITS_COS_MIN and max_abs(got, ref) <= LOGITS_MAX_ABS


def test_attention_wait_gives_up(S):
    # a wait limit far below the attention kernel's own latencies: a wait gives
    # up, the kernel drains what it issued and reports a timeout; the device
    # stays usable and the next call (default limit) is correct
    wl, inp, dev, cfg, packed, ws = _block(S, T=300)
    x = dev.x.float().contiguous()
    out = torch.empty_like(x)
    try:
        S.set_wait_limit_ns(1)
        S.block_forward(cfg, packed, 0, x, out, ws)
        torch.cuda.synchronize()
        assert S.workspace_status(ws) == S.ERR_TIMEOUT
    finally:
        S.set_wait_limit_ns(0)
    _normal_block_call(S, wl, inp, dev, cfg, packed, ws)


def test_model_attention_wait_gives_up(S):
    # the model forward hands row blocks from the attention to the O projection
    # and from each down projection to the next QKV projection through
    # completion flags: an attention whose waits give up still raises its
    # flags, the step ends (no kernel waits out its limit on a flag), the
    # status word reports the timeout, and the next call is correct
    wl = W["smollm2_model_b8_t2048"].scaled(B=2, T=256, n_layers=2, vocab=512)
    inp = synth.generate(wl, seed=35)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, wl.B, wl.T)
    logits = torch.empty(wl.B, wl.T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    try:
        S.set_wait_limit_ns(1)
        S.model_forward(cfg, packed, dev.ids, logits, ws)
        torch.cuda.synchronize()
        assert S.workspace_status(ws) == S.ERR_TIMEOUT
    finally:
        S.set_wait_limit_ns(0)
    S.model_forward(cfg, packed, dev.ids, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref = O.model_forward(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                          inp.ids.numpy().astype(np.int64))
    got = np32(logits)
    assert cosine(got, ref) >= LOGITS_COS_MIN and max_abs(got, ref) <= LOGITS_MAX_ABS
