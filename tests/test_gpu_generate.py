"""The next-token choice inside the decode step and a generate loop over it
("model.py" (SmolLM2-135M) section 7 generate, "model.py" (abi96062)
generate): decode step -> choice -> append the new keys and values -> feed the
chosen ids back.  The GPU loop is compared token for token with the oracle's
own loop (oracle.decode_step, oracle.sample_next, its own appends).

Both sides decide on bf16 logits (the model dtype of the pages): the oracle's
fp64 logits are rounded to bf16 before its choice.  The two sides' logits
differ by up to the logits bar (5e-2), so a step whose choice changes under
that much (a near tie for greedy, a uniform draw near a boundary of the
cumulative distribution when sampling) accepts any of the choices and ends the
comparison of that sequence (the two loops may legitimately part there)."""
import numpy as np
import pytest
import torch

from llama_decoder_forward_gb300 import synth
from oracle import oracle as O
from parity_util import LOGITS_MAX_ABS, np32, oracle_config, oracle_layers, to_device

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from llama_decoder_forward_gb300 import smol
    return smol


def _bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def _decode_case(S, seed, B=5, s_max=300, vocab=2048, lengths=None):
    wl = W["smollm2_decode_b64_cache4096"].scaled(B=B, n_layers=2, s_max=s_max, vocab=vocab,
                                                  len_range=(0, s_max))
    inp = synth.generate(wl, seed=seed)
    if lengths is not None:
        inp.lengths = torch.tensor(lengths, dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_DECODE, B, 1)
    return wl, inp, dev, cfg, packed, ws


def test_greedy_choice_in_the_head_epilogue(S):
    wl, inp, dev, cfg, packed, ws = _decode_case(S, 80)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    k_new = torch.empty(L, B, KV, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(B, wl.vocab, dtype=torch.bfloat16, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.decode_next(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, nxt, ws,
                  logits=logits)
    assert S.workspace_status(ws) == S.OK
    # the same bf16 logits through the separate choice kernel: the same tokens
    ref = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.sample(logits, ref, do_sample=False)
    assert torch.equal(nxt, ref)
    # without writing the logits at all
    nxt2 = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.decode_next(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, nxt2, ws)
    assert S.workspace_status(ws) == S.OK
    assert torch.equal(nxt, nxt2)
    # against the oracle's choice on its own logits (rounded to bf16)
    lg, _, _ = O.decode_step(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                             inp.ids.numpy().astype(np.int64), inp.lengths.numpy(), np32(inp.k_cache),
                             np32(inp.v_cache))
    lb = _bf16(lg)
    want = O.sample_next(lb, do_sample=False)
    got = nxt.cpu().numpy()
    for b in range(B):
        srt = np.sort(lb[b])[::-1]
        if srt[0] - srt[1] > 2 * LOGITS_MAX_ABS:
            assert got[b] == want[b], (b, got[b], want[b])
        else:
            assert lb[b, got[b]] >= srt[0] - 2 * LOGITS_MAX_ABS


def test_sampled_choice_after_the_step(S):
    wl, inp, dev, cfg, packed, ws = _decode_case(S, 81)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    k_new = torch.empty(L, B, KV, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(B, wl.vocab, dtype=torch.bfloat16, device="cuda")
    u = torch.tensor([0.05, 0.3, 0.5, 0.77, 0.99], dtype=torch.float32, device="cuda")
    kw = dict(temperature=0.8, top_k=40, top_p=0.9)
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.decode_next(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, nxt, ws,
                  logits=logits, uniform=u, do_sample=True, **kw)
    assert S.workspace_status(ws) == S.OK
    ref = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.sample(logits, ref, u, **kw)
    assert torch.equal(nxt, ref)


def test_append_kv(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(B=4, n_layers=3, s_max=20, vocab=256)
    cfg = S.config_of(wl)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn(L, B, KV, 20, hd, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(L, B, KV, 20, hd, generator=g, device="cuda").to(torch.bfloat16)
    kn = torch.randn(L, B, KV, hd, generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn(L, B, KV, hd, generator=g, device="cuda").to(torch.bfloat16)
    lens = torch.tensor([0, 7, 19, 20], dtype=torch.int32, device="cuda")   # the last cache is full
    kc0, vc0 = kc.clone(), vc.clone()
    S.append_kv(cfg, kn, vn, kc, vc, lens)
    assert lens.cpu().tolist() == [1, 8, 20, 20]
    for b, pos in enumerate([0, 7, 19]):
        assert torch.equal(kc[:, b, :, pos], kn[:, b])
        assert torch.equal(vc[:, b, :, pos], vn[:, b])
        kc0[:, b, :, pos] = kn[:, b]
        vc0[:, b, :, pos] = vn[:, b]
    assert torch.equal(kc, kc0) and torch.equal(vc, vc0)   # nothing else written, the full row untouched


@pytest.mark.parametrize("do_sample", [False, True])
def test_generate_loop_against_the_oracle(S, do_sample):
    lengths = [0, 7, 20]
    wl, inp, dev, cfg, packed, ws = _decode_case(S, 82 + do_sample, B=3, s_max=48, vocab=512, lengths=lengths)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    steps = 8
    kw = dict(temperature=0.8, top_k=20, top_p=0.9) if do_sample else {}
    us = torch.rand(steps, B, generator=torch.Generator().manual_seed(84))
    # GPU loop: the chosen ids are fed back through the same buffer; the
    # logits are kept for the comparison below (the greedy choice is still
    # taken in the head's epilogue)
    ids = dev.ids.clone()
    lens = dev.lengths.clone()
    kc, vc = dev.k_cache.clone(), dev.v_cache.clone()
    k_new = torch.empty(L, B, KV, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(B, wl.vocab, dtype=torch.bfloat16, device="cuda")
    got, got_logits = [], []
    for s in range(steps):
        S.decode_next(cfg, packed, ids, lens, kc, vc, k_new, v_new, ids, ws, logits=logits,
                      uniform=us[s].cuda() if do_sample else None, do_sample=do_sample, **kw)
        S.append_kv(cfg, k_new, v_new, kc, vc, lens)
        got.append(ids.cpu().numpy().copy())
        got_logits.append(np32(logits).astype(np.float64))
    assert S.workspace_status(ws) == S.OK
    assert lens.cpu().tolist() == [n + steps for n in lengths]
    # the oracle's own loop
    oc, ol = oracle_config(wl), oracle_layers(inp)
    E, fn = np32(inp.embed), np32(inp.final_norm)
    okc = np32(inp.k_cache).astype(np.float64)
    ovc = np32(inp.v_cache).astype(np.float64)
    o_ids = inp.ids.numpy().astype(np.int64)
    o_lens = np.asarray(lengths)
    live = np.ones(B, dtype=bool)
    agreed = 0
    okw = {k: (float(np.float32(v)) if isinstance(v, float) else v) for k, v in kw.items()}
    for s in range(steps):
        lg, kn, vn = O.decode_step(oc, ol, E, fn, o_ids, o_lens, okc, ovc)
        lb = _bf16(lg)
        u = us[s].numpy().astype(np.float64)
        choice = O.sample_next(lb, u=u, do_sample=do_sample, **okw)
        for b in range(B):
            if not live[b]:
                continue
            gl = got_logits[s][b]
            # the step itself meets the decode bar along the loop
            assert np.max(np.abs(gl - lg[b])) <= LOGITS_MAX_ABS, (s, b)
            g, o = int(got[s][b]), int(choice[b])
            if g == o:
                agreed += 1
                continue
            # a different token must be explained by the two sides' logits
            if do_sample:
                # the choice rule on the GPU's own row gives the GPU's token
                assert int(O.sample_next(gl[None], u=u[b:b + 1], do_sample=True, **okw)[0]) == g, (s, b)
            else:
                # a near tie: the oracle's margin is within the measured errors
                assert lb[b, o] - lb[b, g] <= abs(gl[o] - lb[b, o]) + abs(gl[g] - lb[b, g]) + 1e-6, (s, b)
            live[b] = False                       # the loops part from here on
        for b in range(B):
            okc[:, b, :, o_lens[b]] = kn[:, b]
            ovc[:, b, :, o_lens[b]] = vn[:, b]
        o_lens = o_lens + 1
        o_ids = choice
    print(f"generate loop (sample={do_sample}): {agreed} tokens equal to the oracle's, "
          f"{int(live.sum())} of {B} sequences equal to the end")
    assert agreed >= steps                        # at least one sequence's worth of equal tokens
