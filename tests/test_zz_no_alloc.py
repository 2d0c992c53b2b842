"""smol_decode_step_noalloc through the C ABI (collected last).

Some callers cannot give the library device memory when they decode (a
serving loop that allows no allocation after start-up, or code that must not
call cudaMalloc because it can synchronise the device).  For them the decode
step has a variant whose scratch is a fixed array inside the library.  This
test runs it twice in a row and checks each result against the oracle and
against the workspace-taking entry point on the same inputs, and reads the
variant's own status word after each call.
"""
import ctypes

import numpy as np
import pytest
import torch

from llama_decoder_forward_gb300 import synth
from oracle import oracle as O
from parity_util import (BLOCK_REL_TOL, LOGITS_COS_MIN, LOGITS_MAX_ABS, cosine, max_abs, np32,
                         oracle_config, oracle_layers, rel_max_err, rel_max_err_bf16_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from llama_decoder_forward_gb300 import smol
    return smol


def test_noalloc_decode_matches_oracle_and_workspace_decode(S):
    wl = synth.WORKLOADS["smollm2_decode_b64_cache4096"].scaled(B=6, n_layers=2, s_max=700)
    inp = synth.generate(wl, seed=21)
    lengths = [700, 0, 1, 512, 513, 250]
    inp.lengths = torch.tensor(lengths, dtype=torch.int32)
    dev = lambda t: t.to("cuda")
    cfg = S.config_of(wl)
    layers = [{k: dev(v) for k, v in lw.items()} for lw in inp.layers]
    packed = S.prepare_weights(cfg, layers, dev(inp.embed), dev(inp.final_norm))
    ids, lens, kc, vc = dev(inp.ids), dev(inp.lengths), dev(inp.k_cache), dev(inp.v_cache)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim

    def outputs():
        k_new = torch.full((L, B, KV, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        v_new = torch.full_like(k_new, float("nan"))
        logits = torch.full((B, wl.vocab), float("nan"), dtype=torch.bfloat16, device="cuda")
        return k_new, v_new, logits

    ref_logits, ref_k, ref_v = O.decode_step(oracle_config(wl), oracle_layers(inp), np32(inp.embed),
                                             np32(inp.final_norm), inp.ids.numpy().astype(np.int64),
                                             np.asarray(lengths), np32(inp.k_cache), np32(inp.v_cache))
    ws_k, ws_v, ws_logits = outputs()
    ws = S.alloc_workspace(cfg, S.OP_DECODE, B, 1)
    S.decode_step(cfg, packed, ids, lens, kc, vc, ws_k, ws_v, ws_logits, ws)
    assert S.workspace_status(ws) == S.OK
    with_ws = [np32(t) for t in (ws_logits, ws_k, ws_v)]
    for call in range(2):
        k_new, v_new, logits = outputs()
        S.decode_step_noalloc(cfg, packed, ids, lens, kc, vc, k_new, v_new, logits)
        assert S.decode_noalloc_status() == S.OK, call
        got = [np32(t) for t in (logits, k_new, v_new)]
        assert all(np.all(np.isfinite(g)) for g in got), f"call {call}: non-finite output"
        # against the oracle, at the decode step's acceptance bars
        assert cosine(got[0], ref_logits) >= LOGITS_COS_MIN, call
        assert max_abs(got[0], ref_logits) <= LOGITS_MAX_ABS, call
        assert rel_max_err_bf16_out(got[1], ref_k) <= BLOCK_REL_TOL, call
        assert rel_max_err_bf16_out(got[2], ref_v) <= BLOCK_REL_TOL, call
        # against the entry point that takes a workspace, within the same bars
        assert cosine(got[0], with_ws[0]) >= LOGITS_COS_MIN, call
        assert max_abs(got[0], with_ws[0]) <= LOGITS_MAX_ABS, call
        assert rel_max_err(got[1], with_ws[1]) <= BLOCK_REL_TOL, call
        assert rel_max_err(got[2], with_ws[2]) <= BLOCK_REL_TOL, call


def test_noalloc_rejects_batches_beyond_its_scratch(S):
    wl = synth.WORKLOADS["smollm2_decode_b64_cache4096"]
    cfg = S.config_of(wl)
    big_b = 1
    while S.workspace_bytes(cfg, S.OP_DECODE, big_b, 1) <= (8 << 20):
        big_b *= 2
    f = ctypes.c_void_p(0x10000)
    rc = S.raw.smol_decode_step_noalloc(ctypes.byref(cfg), f, f, f, big_b, f, f, 4096, f, f, f, None)
    assert rc == S.ERR_WORKSPACE
    assert S.decode_noalloc_status() == S.OK
