"""Parity at the workloads' full sizes, in the launch configuration bench.py
times, on sampled outputs the fp64 oracle can compute.

Causality makes a prefix exact: the outputs of tokens [0, P) of a sequence
depend only on those tokens, so the oracle runs on a prefix of a sampled
sequence (or on a whole sampled sequence) while the GPU runs the full batch.
Every GPU output is also scanned for non-finite values.
"""
import numpy as np
import pytest
import torch

from llama_decoder_forward_gb300 import synth
from oracle import oracle as O
from parity_util import (BLOCK_REL_TOL, LOGITS_COS_MIN, LOGITS_MAX_ABS, cosine, max_abs, np32,
                         oracle_config, oracle_layers, rel_max_err, rel_max_err_bf16_out)


def check_cache_entries(got_k, got_v, ref_k, ref_v, what):
    """New cache entries of a whole-model pass [L, ...]: layer 0's come from a
    block whose input is the oracle's own (the embedding), held to the block
    bar; every layer's are intermediate outputs deep in the model, held to the
    model bar (cosine >= 0.999 and max |err| <= 5e-2 x RMS of the entries)."""
    for got, ref, name in ((got_k, ref_k, "k"), (got_v, ref_v, "v")):
        e0 = rel_max_err_bf16_out(got[0], ref[0])
        cos = cosine(got, ref)
        rel = max_abs(got, ref) / float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
        print(f"{what} {name}: layer 0 {e0:.3e}, all layers cos {cos:.7f} max/rms {rel:.3e}")
        assert e0 <= BLOCK_REL_TOL, (what, name, e0)
        assert cos >= LOGITS_COS_MIN and rel <= LOGITS_MAX_ABS, (what, name, cos, rel)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from llama_decoder_forward_gb300 import smol
    return smol


def test_full_model_smollm2_b8_t2048(S):
    wl = W["smollm2_model_b8_t2048"]
    inp = synth.generate(wl, seed=0, device="cuda")
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers, inp.embed, inp.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, wl.B, wl.T)
    logits = torch.empty(wl.B, wl.T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.model_forward(cfg, packed, inp.ids, logits, ws)
    assert S.workspace_status(ws) == S.OK
    assert bool(torch.isfinite(logits).all())
    oc, ol = oracle_config(wl), oracle_layers(inp)
    E, fn = np32(inp.embed), np32(inp.final_norm)
    ids = inp.ids.cpu().numpy().astype(np.int64)
    # sequence 0 whole (rows up to 2047), sequence 5 over a 256-token prefix
    for b, P in ((0, wl.T), (5, 256)):
        ref = O.model_forward(oc, ol, E, fn, ids[b:b + 1, :P])[0]
        got = np32(logits[b, :P])
        cos, mabs = cosine(got, ref), max_abs(got, ref)
        print(f"seq {b} prefix {P}: cos {cos:.7f} max abs {mabs:.3e}")
        assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (b, cos, mabs)


def test_full_smollm3_4blocks_b4_t4096(S):
    wl = W["smollm3_4blocks_b4_t4096"]
    inp = synth.generate(wl, seed=0, device="cuda")
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, wl.B, wl.T)
    x = inp.x.float().contiguous()
    outs = []
    for l in range(wl.n_layers):                   # fp32 residual stream between blocks
        y = torch.empty_like(x)
        S.block_forward(cfg, packed, l, x, y, ws)
        outs.append(y)
        x = y
    assert S.workspace_status(ws) == S.OK
    assert all(bool(torch.isfinite(o).all()) for o in outs)
    P = 384                                        # sequence 2, prefix of 384 tokens
    oc, ol = oracle_config(wl, 1), oracle_layers(inp)
    xr = np32(inp.x[2:3, :P]).astype(np.float64)
    for l in range(wl.n_layers):
        xr = O.block_forward(oc, ol[l], xr)
        err = rel_max_err(outs[l][2, :P].cpu().numpy(), xr[0])
        print(f"block {l}: rel max err {err:.3e}")
        assert err <= BLOCK_REL_TOL, (l, err)


def test_full_leftpad_125m_b16_t1024(S):
    wl = W["slm125m_block_leftpad_b16_t1024"]
    inp = synth.generate(wl, seed=0, device="cuda")
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, wl.B, wl.T)
    x = inp.x.float().contiguous()
    out = torch.empty_like(x)
    k_out = torch.empty(wl.B, wl.n_kv_heads, wl.T, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    v_out = torch.empty_like(k_out)
    S.block_forward(cfg, packed, 0, x, out, ws, valid_start=inp.valid_start, k_out=k_out, v_out=v_out)
    assert S.workspace_status(ws) == S.OK
    assert bool(torch.isfinite(out).all())
    vs = inp.valid_start.cpu().numpy()
    oc, ow = oracle_config(wl, 1), oracle_layers(inp)[0]
    # the shortest and the longest sequence, whole
    for b in (int(np.argmax(vs)), int(np.argmin(vs))):
        taps = {}
        ref = O.block_forward(oc, ow, np32(inp.x[b:b + 1]), [vs[b]], taps=taps)[0]
        got = out[b].cpu().numpy()
        err = rel_max_err(got[vs[b]:], ref[vs[b]:])
        ek = rel_max_err_bf16_out(np32(k_out[b])[:, vs[b]:], taps["attention_keys"][0][:, vs[b]:])
        print(f"seq {b} (valid from {vs[b]}): out {err:.3e} k {ek:.3e}")
        assert err <= BLOCK_REL_TOL and ek <= BLOCK_REL_TOL, (b, err, ek)


def test_full_decode_smollm2_b64_cache4096(S):
    wl = W["smollm2_decode_b64_cache4096"]
    inp = synth.generate(wl, seed=0, device="cuda")
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers, inp.embed, inp.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_DECODE, wl.B, 1)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    k_new = torch.empty(L, B, KV, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(B, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.decode_step(cfg, packed, inp.ids, inp.lengths, inp.k_cache, inp.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    assert bool(torch.isfinite(logits).all())
    lens = inp.lengths.cpu().numpy()
    oc, ol = oracle_config(wl), oracle_layers(inp)
    E, fn = np32(inp.embed), np32(inp.final_norm)
    ids = inp.ids.cpu().numpy().astype(np.int64)
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 17})
    kc = np32(inp.k_cache[:, picks])
    vc = np32(inp.v_cache[:, picks])
    ref, kr, vr = O.decode_step(oc, ol, E, fn, ids[picks], lens[picks], kc, vc)
    got = np32(logits[picks])
    cos, mabs = cosine(got, ref), max_abs(got, ref)
    print(f"decode seqs {picks} (lengths {lens[picks].tolist()}): cos {cos:.7f} max abs {mabs:.3e}")
    assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (cos, mabs)
    check_cache_entries(np32(k_new[:, picks]), np32(v_new[:, picks]), kr, vr, "decode")


def test_full_prefill_with_cache_smollm2_b64_cache4096(S):
    # a 64-token chunk on top of the decode workload's caches (B = 64, 30
    # layers, lengths uniform in [1024, 4096] in 4096-slot caches)
    wl = W["smollm2_decode_b64_cache4096"]
    inp = synth.generate(wl, seed=1, device="cuda")
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, inp.layers, inp.embed, inp.final_norm)
    L, B, KV, hd, T = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim, 64
    g = torch.Generator(device="cuda").manual_seed(2)
    ids = torch.randint(0, wl.vocab, (B, T), generator=g, device="cuda", dtype=torch.int32)
    ws = S.prefill_cache_workspace(cfg, B, T, wl.s_max)
    k_new = torch.empty(L, B, KV, T, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(B, T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.prefill_with_cache(cfg, packed, ids, inp.lengths, inp.k_cache, inp.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    assert bool(torch.isfinite(logits).all())
    lens = inp.lengths.cpu().numpy()
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 40})
    ref, kr, vr = O.prefill_with_cache(oracle_config(wl), oracle_layers(inp), np32(inp.embed),
                                       np32(inp.final_norm), ids[picks].cpu().numpy().astype(np.int64),
                                       lens[picks], np32(inp.k_cache[:, picks]), np32(inp.v_cache[:, picks]))
    got = np32(logits[picks])
    cos, mabs = cosine(got, ref), max_abs(got, ref)
    print(f"prefill on cache seqs {picks} (lengths {lens[picks].tolist()}): cos {cos:.7f} max abs {mabs:.3e}")
    assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (cos, mabs)
    check_cache_entries(np32(k_new[:, picks]), np32(v_new[:, picks]), kr, vr, "prefill on cache")
