"""GPU-vs-oracle parity through the C ABI, at sizes the fp64 oracle finishes in
seconds that still span several tiles and a ragged tail."""
import numpy as np
import pytest
import torch

from llama_decoder_forward_gb300 import synth
from oracle import oracle as O
from parity_util import (BLOCK_REL_TOL, LOGITS_COS_MIN, LOGITS_MAX_ABS, cosine, max_abs, np32,
                         oracle_config, oracle_layers, rel_max_err, rel_max_err_bf16_out, to_device)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from llama_decoder_forward_gb300 import smol
    return smol


def run_block_case(S, wl, seed=0, check_kv=True, act=torch.float32, x_scale=1.0, layer=0):
    """Block `layer` of the workload through the C ABI vs the oracle.  act is
    the residual-stream type of x/out (fp32: the stated bar; bf16: the bar plus
    the output's own rounding).  k/v are bf16 cache entries, checked like bf16
    outputs."""
    inp = synth.generate(wl, seed=seed)
    if x_scale != 1.0:
        inp.x = (inp.x.float() * x_scale).to(torch.bfloat16)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, wl.B, wl.T)
    x = dev.x.to(act).contiguous()
    out = torch.empty_like(x)
    k_out = torch.empty(wl.B, wl.n_kv_heads, wl.T, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    v_out = torch.empty_like(k_out)
    S.block_forward(cfg, packed, layer, x, out, ws, valid_start=dev.valid_start, k_out=k_out, v_out=v_out)
    assert S.workspace_status(ws) == S.OK
    torch.cuda.synchronize()
    taps = {}
    vs = None if inp.valid_start is None else inp.valid_start.numpy()
    ref = O.block_forward(oracle_config(wl), oracle_layers(inp)[layer], np32(inp.x), vs, taps=taps,
                          layer=layer)
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    rows = np.ones((wl.B, wl.T), dtype=bool)
    if vs is not None:
        for b in range(wl.B):
            rows[b, :vs[b]] = False
    metric = rel_max_err if act == torch.float32 else rel_max_err_bf16_out
    err = metric(got[rows], ref[rows])
    ek = ev = 0.0
    if check_kv:
        kmask = np.broadcast_to(rows[:, None, :, None], taps["attention_keys"].shape)
        ek = rel_max_err_bf16_out(np32(k_out)[kmask], taps["attention_keys"][kmask])
        ev = rel_max_err_bf16_out(np32(v_out)[kmask], taps["attention_values"][kmask])
    msg = f"rel max err ({act}): out {err:.3e}, k {ek:.3e}, v {ev:.3e}"
    print(msg)
    assert err <= BLOCK_REL_TOL and ek <= BLOCK_REL_TOL and ev <= BLOCK_REL_TOL, msg
    return err


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_block_smollm2_b1_t128(S, act):
    run_block_case(S, W["smollm2_block_b1_t128"], act=act)


def test_block_small_residual_input(S):
    # input at the embedding's scale (std 0.0417): the block output is then
    # almost entirely attention + MLP, the hardest case for the relative bar
    run_block_case(S, W["smollm2_block_b1_t128"].scaled(B=2, T=96), x_scale=0.0417)


@pytest.mark.parametrize("B,T", [(2, 200), (1, 1), (3, 67), (1, 385), (1, 2), (2, 3), (1, 65), (2, 127),
                                 (1, 129)])
def test_block_smollm2_ragged(S, B, T):
    run_block_case(S, W["smollm2_block_b1_t128"].scaled(B=B, T=T), seed=B * 1000 + T)


@pytest.mark.parametrize("H,KV", [(4, 4), (4, 2), (4, 1), (6, 1), (5, 1), (7, 1), (8, 1)])
def test_block_group_sizes(S, H, KV):
    # query heads per kv head 1, 2, 4, 6, 5, 7 and 8: one CTA per group of 1 or
    # 2 heads (one softmax warpgroup, or two taking the slots in turn) and groups
    # split over several CTAs (two or three heads each, or one for 5 and 7)
    wl = W["smollm2_block_b1_t128"].scaled(B=2, T=300, hidden=64 * H, n_heads=H, n_kv_heads=KV,
                                           intermediate=512)
    run_block_case(S, wl, seed=40 + H * 10 + KV)


def test_block_smollm3_shape(S):
    run_block_case(S, W["smollm3_4blocks_b4_t4096"].scaled(B=1, T=160, n_layers=1))


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_block_left_padded(S, act):
    wl = W["slm125m_block_leftpad_b16_t1024"].scaled(B=4, T=192, len_range=(1, 192))
    run_block_case(S, wl, seed=3, act=act)


def test_block_left_padded_all_padding_row(S):
    # one sequence is entirely padding (valid_start == T): its rows must stay finite
    wl = W["slm125m_block_leftpad_b16_t1024"].scaled(B=2, T=64, len_range=(1, 64))
    inp = synth.generate(wl, seed=5)
    inp.valid_start = torch.tensor([64, 10], dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, 2, 64)
    out = torch.empty_like(dev.x)
    S.block_forward(cfg, packed, 0, dev.x, out, ws, valid_start=dev.valid_start)
    torch.cuda.synchronize()
    got = np32(out)
    assert np.all(np.isfinite(got))
    ref = O.block_forward(oracle_config(wl, 1), oracle_layers(inp, 1)[0], np32(inp.x), [64, 10])
    assert rel_max_err_bf16_out(got[1, 10:], ref[1, 10:]) <= BLOCK_REL_TOL


def test_block_in_place(S):
    wl = W["smollm2_block_b1_t128"].scaled(B=2, T=130)
    inp = synth.generate(wl, seed=9)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, wl.B, wl.T)
    x = dev.x.clone()
    S.block_forward(cfg, packed, 0, x, x, ws)
    torch.cuda.synchronize()
    ref = O.block_forward(oracle_config(wl, 1), oracle_layers(inp, 1)[0], np32(inp.x))
    assert rel_max_err_bf16_out(np32(x), ref) <= BLOCK_REL_TOL
    # fp32 residual stream in place
    x32 = dev.x.float().contiguous()
    S.block_forward(cfg, packed, 0, x32, x32, ws)
    torch.cuda.synchronize()
    assert rel_max_err(x32.cpu().numpy(), ref) <= BLOCK_REL_TOL


def run_model_case(S, wl, seed=0, valid_start=None):
    inp = synth.generate(wl, seed=seed)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, wl.B, wl.T)
    logits = torch.empty(wl.B, wl.T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.model_forward(cfg, packed, dev.ids, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref = O.model_forward(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                          inp.ids.numpy().astype(np.int64))
    got = np32(logits)
    assert np.all(np.isfinite(got))
    cos, mabs = cosine(got, ref), max_abs(got, ref)
    print(f"model: cos {cos:.7f} max abs {mabs:.3e}")
    assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (cos, mabs)
    return cos, mabs


def test_model_two_layers(S):
    run_model_case(S, W["smollm2_model_b8_t2048"].scaled(B=2, T=96, n_layers=2))


def test_model_ragged_small_vocab(S):
    run_model_case(S, W["smollm2_model_b8_t2048"].scaled(B=3, T=37, n_layers=3, vocab=1024), seed=4)


def test_model_left_padded(S):
    # left padding in the model forward (the attention's completion flags on:
    # T is a multiple of 128); rows before each sequence's start are not compared
    wl = W["smollm2_model_b8_t2048"].scaled(B=3, T=256, n_layers=2, vocab=512)
    inp = synth.generate(wl, seed=6)
    vs = torch.tensor([0, 37, 200], dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, wl.B, wl.T)
    logits = torch.empty(wl.B, wl.T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.model_forward(cfg, packed, dev.ids, logits, ws, valid_start=vs.cuda())
    assert S.workspace_status(ws) == S.OK
    ref = O.model_forward(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                          inp.ids.numpy().astype(np.int64), valid_start=vs.numpy())
    got = np32(logits)
    for b in range(wl.B):
        g, r = got[b, int(vs[b]):], ref[b, int(vs[b]):]
        cos, mabs = cosine(g, r), max_abs(g, r)
        assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (b, cos, mabs)


@pytest.mark.parametrize("B,T", [(1, 1100), (1, 1152), (3, 384)])
def test_model_row_block_flags(S, B, T):
    # the model forward hands row blocks over through completion flags: CTA
    # pairs over an odd number of 128-row blocks (the last pair's second block
    # lies past M), with the attention's flags (T a multiple of 128) and
    # without them
    run_model_case(S, W["smollm2_model_b8_t2048"].scaled(B=B, T=T, n_layers=2, vocab=512), seed=5)


def test_model_at_max_positions(S):
    # the longest sequence a configuration takes: T = max_pos, so the last row
    # rotates at position max_pos - 1, the table's last entry
    run_model_case(S, W["smollm2_model_b8_t2048"].scaled(B=1, T=1024, n_layers=2, vocab=512, max_pos=1024),
                   seed=8)


def run_decode_case(S, wl, lengths, seed=0):
    wl = wl.scaled(B=len(lengths))
    inp = synth.generate(wl, seed=seed)
    inp.lengths = torch.tensor(lengths, dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_DECODE, wl.B, 1)
    L, Bn, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    k_new = torch.empty(L, Bn, KV, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(Bn, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.decode_step(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref, kr, vr = O.decode_step(oracle_config(wl), oracle_layers(inp), np32(inp.embed),
                                np32(inp.final_norm), inp.ids.numpy().astype(np.int64),
                                np.asarray(lengths), np32(inp.k_cache), np32(inp.v_cache))
    got = np32(logits)
    cos, mabs = cosine(got, ref), max_abs(got, ref)
    ek, ev = rel_max_err_bf16_out(np32(k_new), kr), rel_max_err_bf16_out(np32(v_new), vr)
    print(f"decode: cos {cos:.6f} max abs {mabs:.3e} k {ek:.3e} v {ev:.3e}")
    assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (cos, mabs)
    assert ek <= BLOCK_REL_TOL and ev <= BLOCK_REL_TOL, (ek, ev)
    return cos, mabs


def test_decode_small(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=700)
    run_decode_case(S, wl, [0, 1, 511, 512, 513, 700, 37])


def test_decode_one_chunk_many_layers(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=4, s_max=64, vocab=512)
    run_decode_case(S, wl, [64, 3, 17], seed=2)


def test_decode_batch_beyond_narrow_units(S):
    # B > 64: the projections run on the tile GEMM instead of the narrow-unit kernel
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=320, vocab=1024)
    lengths = [int(v) for v in np.random.default_rng(5).integers(0, 321, size=80)]
    run_decode_case(S, wl, lengths, seed=6)


def test_decode_head_dim_128(S):
    # SmolLM3-shaped layer (hd 128): CUDA-core decode attention, tile-GEMM projections
    wl = W["smollm2_decode_b64_cache4096"].scaled(
        hidden=2048, n_heads=16, n_kv_heads=4, head_dim=128, intermediate=11008, n_layers=1,
        vocab=512, s_max=300, rms_eps=1e-6, rope_theta=1e6, w_std=0.02)
    run_decode_case(S, wl, [0, 129, 300], seed=7)


def test_decode_single_sequence_long_cache(S):
    # one sequence, 16 chunks per kv head: the persistent attention spreads the
    # 48 chunks over as many CTAs, so each (sequence, kv head) is merged from
    # up to 16 partials; most CTAs get no work at all
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=1, s_max=4096, vocab=512)
    run_decode_case(S, wl, [4095], seed=8)


@pytest.mark.parametrize("H,KV", [(4, 4), (4, 2), (8, 2), (6, 1), (8, 1)])
def test_decode_group_sizes(S, H, KV):
    # query heads per kv head 1, 2, 4, 6 and 8 in the persistent decode
    # attention (groups above 4 take its eight-row fragment layout)
    wl = W["smollm2_decode_b64_cache4096"].scaled(hidden=64 * H, n_heads=H, n_kv_heads=KV, intermediate=512,
                                                  n_layers=2, s_max=600, vocab=512)
    run_decode_case(S, wl, [0, 1, 255, 256, 257, 600, 413], seed=50 + H * 10 + KV)


def test_decode_empty_caches(S):
    # no cached keys: attention over the new token alone
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=64, vocab=512)
    run_decode_case(S, wl, [0, 0, 1], seed=9)


# ---------------------------------------------------------------- SmolLM3 per-block variants
# NoPE blocks and sliding windows ("SmolLM3" page: "Every fourth block has no
# rotary", "A sliding window the 3B checkpoints leave off")

@pytest.mark.parametrize("rope,window", [(0, 0), (1, 100), (0, 128), (1, 1), (1, 257), (0, 385)])
def test_block_nope_window_tc_attention(S, rope, window):
    # head dim 64, groups of 3: the tcgen05 attention; windows below, at and
    # across the 128-key tiles, and one as long as the sequence
    wl = W["smollm2_block_b1_t128"].scaled(B=2, T=385, n_layers=2, no_rope_layers=(1, rope),
                                           sliding_window=(0, window))
    run_block_case(S, wl, seed=40 + window, layer=1)


def test_block_window_left_padded(S):
    wl = W["slm125m_block_leftpad_b16_t1024"].scaled(B=4, T=300, len_range=(1, 300), n_layers=1,
                                                     sliding_window=(70,))
    run_block_case(S, wl, seed=41, act=torch.bfloat16)


def test_block_smollm3_nope_window_head_dim_128(S):
    # head dim 128: the tcgen05 attention with one query head per CTA
    wl = W["smollm3_4blocks_b4_t4096"].scaled(B=2, T=150, n_layers=2, no_rope_layers=(1, 0),
                                              sliding_window=(0, 37))
    run_block_case(S, wl, seed=42, layer=1)


def test_model_nope_and_window_layers(S):
    # the two-block layout of the SmolLM3 page's small checkpoint: block 1 is a
    # NoPE block with a window
    wl = W["smollm2_model_b8_t2048"].scaled(B=2, T=200, n_layers=2, vocab=1024,
                                            no_rope_layers=(1, 0), sliding_window=(0, 128))
    run_model_case(S, wl, seed=43)


def test_decode_nope_and_window_layers(S):
    # persistent decode attention: lengths below, at and above the windows, and
    # windows that start inside a 256-key chunk
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=3, s_max=700, vocab=512,
                                                  no_rope_layers=(1, 0, 1),
                                                  sliding_window=(0, 128, 300))
    run_decode_case(S, wl, [0, 1, 127, 128, 129, 299, 300, 301, 700, 555], seed=44)


def test_decode_window_head_dim_128(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(
        hidden=2048, n_heads=16, n_kv_heads=4, head_dim=128, intermediate=11008, n_layers=2,
        vocab=512, s_max=300, rms_eps=1e-6, rope_theta=1e6, w_std=0.02,
        no_rope_layers=(0, 1), sliding_window=(128, 0))
    run_decode_case(S, wl, [0, 129, 300, 64], seed=45)


def test_decode_batch_beyond_persistent_limit(S):
    # more than 2048 sequences: the per-chunk tensor-core decode attention
    # (one CTA per (chunk, kv head, sequence)), with and without a window
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=96, vocab=512,
                                                  sliding_window=(0, 60))
    lengths = [int(v) for v in np.random.default_rng(46).integers(0, 97, size=2100)]
    run_decode_case(S, wl, lengths, seed=46)


# ---------------------------------------------------------------- next-token choice
# ("model.py" (SmolLM2-135M) section 7 generate; the abi96062 model.py generate)

def _oracle_choices(rows, u, **kw):
    """The oracle's tokens, and the tokens it gives when u or top_p move by 1e-6
    (a fp32 kernel may land either way that close to a boundary)."""
    base = O.sample_next(rows, u=u, **kw)
    alts = [base]
    for du in (-1e-6, 1e-6):
        alts.append(O.sample_next(rows, u=np.clip(u + du, 0.0, 1.0 - 1e-12), **kw))
    tp = kw.get("top_p")
    if tp is not None and tp < 1.0:
        for dp in (-1e-6, 1e-6):
            alts.append(O.sample_next(rows, u=u, **{**kw, "top_p": tp + dp}))
    return base, np.stack(alts)


def _check_sample(S, logits_bf16, u, **kw):
    B = logits_bf16.shape[0]
    dev = logits_bf16.cuda()
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.sample(dev, nxt, u.cuda(), **kw)
    torch.cuda.synchronize()
    got = nxt.cpu().numpy().astype(np.int64)
    rows = logits_bf16.float().numpy().astype(np.float64)
    okw = {k: v for k, v in kw.items() if k in ("temperature", "top_k", "top_p", "do_sample")}
    for k in ("temperature", "top_p"):            # the kernel takes them as fp32
        if k in okw:
            okw[k] = float(np.float32(okw[k]))
    base, alts = _oracle_choices(rows, u.numpy().astype(np.float64), **okw)
    decisive = np.all(alts == base[None], axis=0)
    assert np.all(got[decisive] == base[decisive]), (kw, np.nonzero(got[decisive] != base[decisive]))
    assert np.all(np.any(alts == got[None], axis=0)), kw
    return int(decisive.sum())


@pytest.mark.parametrize("kw", [
    dict(do_sample=False), dict(temperature=0.0), dict(temperature=1.0),
    dict(temperature=0.7, top_k=50), dict(temperature=1.0, top_p=0.9),
    dict(temperature=0.8, top_k=40, top_p=0.5), dict(temperature=1.3, top_k=1),
    dict(temperature=1.0, top_p=1e-6), dict(temperature=0.6, top_k=49152, top_p=0.95),
    dict(temperature=1.0, top_p=0.0), dict(temperature=0.9, top_k=30, top_p=-0.5)])
@pytest.mark.parametrize("dist", ["normal", "ties"])
def test_sample_matches_oracle(S, kw, dist):
    B, V = 32, 49152
    g = torch.Generator().manual_seed(50 + (dist == "ties"))
    x = torch.randn(B, V, generator=g)
    # "ties": whole-number logits, thousands of equal values per row
    logits = ((x * 3.0) if dist == "normal" else torch.round(x * 2.0)).to(torch.bfloat16)
    u = torch.rand(B, generator=g)
    n = _check_sample(S, logits, u, **kw)
    assert n >= B // 2                            # most draws are nowhere near a boundary


def test_sample_smollm3_vocab_strided_rows(S):
    # the SmolLM3 vocabulary (128256) and rows with a pitch beyond V
    B, V, ld = 4, 128256, 128256 + 64
    g = torch.Generator().manual_seed(52)
    buf = (torch.randn(B, ld, generator=g) * 2.0).to(torch.bfloat16)
    u = torch.rand(B, generator=g)
    logits = buf.cuda()[:, :V]
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    S.sample(logits, nxt, u.cuda(), temperature=0.9, top_k=100, top_p=0.8)
    torch.cuda.synchronize()
    rows = buf[:, :V].float().numpy().astype(np.float64)
    base, alts = _oracle_choices(rows, u.numpy().astype(np.float64), temperature=float(np.float32(0.9)),
                                 top_k=100, top_p=float(np.float32(0.8)))
    got = nxt.cpu().numpy()
    assert np.all(np.any(alts == got[None], axis=0))


def test_sample_degenerate_rows(S):
    # one-token vocabulary; all-equal rows (greedy takes index 0, the draw is uniform)
    one = torch.tensor([[1.5], [-2.0]], dtype=torch.bfloat16)
    for kw in (dict(do_sample=False), dict(temperature=1.0, top_p=0.5, top_k=3)):
        assert _check_sample(S, one, torch.tensor([0.3, 0.99]), **kw) == 2
    flat = torch.zeros(3, 1000, dtype=torch.bfloat16)
    _check_sample(S, flat, torch.tensor([0.0, 0.5004, 0.99999]), temperature=1.0)
    _check_sample(S, flat, torch.tensor([0.0, 0.5, 0.99999]), do_sample=False)
    _check_sample(S, flat, torch.tensor([0.1, 0.6, 0.99999]), temperature=1.0, top_p=0.3)


def test_sample_after_decode_step(S):
    # the decode step's logits feed the choice directly (no host round trip)
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=128, vocab=4096, B=5)
    inp = synth.generate(wl, seed=53)
    inp.lengths = torch.tensor([0, 5, 64, 100, 128], dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_DECODE, wl.B, 1)
    k_new = torch.empty(2, 5, 3, 64, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(5, 4096, dtype=torch.bfloat16, device="cuda")
    S.decode_step(cfg, packed, dev.ids, dev.lengths, dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
    u = torch.tensor([0.1, 0.3, 0.5, 0.7, 0.9])
    _check_sample(S, logits.cpu(), u, temperature=0.8, top_k=20, top_p=0.9)


# ---------------------------------------------------------------- additive key mask
# ("model.py" (SmolLM2-135M) section 4: attention_mask of 0 / -inf over the keys)

def _key_mask(B, T, seed, keep=0.6):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand(B, T, generator=g) < keep).to(torch.uint8)
    m[:, 1::97] = 0                                   # hidden keys at tile-crossing strides
    return m


@pytest.mark.parametrize("wl_name,B,T,layer_kw", [
    ("smollm2_block_b1_t128", 2, 300, dict()),                                   # tcgen05, G = 3
    ("smollm2_block_b1_t128", 1, 257, dict(sliding_window=(90,))),               # mask + window
    ("smollm3_4blocks_b4_t4096", 2, 130, dict()),                                # tcgen05, hd 128
])
def test_block_key_mask(S, wl_name, B, T, layer_kw):
    wl = W[wl_name].scaled(B=B, T=T, n_layers=1, **layer_kw)
    inp = synth.generate(wl, seed=60 + T)
    mask = _key_mask(B, T, 61 + T)
    mask[0, :5] = 0                                   # the first rows of sequence 0 see no key
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers)
    ws = S.alloc_workspace(cfg, S.OP_BLOCK, B, T)
    x = dev.x.float().contiguous()
    out = torch.empty_like(x)
    S.block_forward_masked(cfg, packed, 0, x, out, ws, mask.cuda())
    assert S.workspace_status(ws) == S.OK
    torch.cuda.synchronize()
    ref = O.block_forward(oracle_config(wl), oracle_layers(inp)[0], np32(inp.x), key_mask=mask.numpy().astype(bool))
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    err = rel_max_err(got, ref)
    print(f"key mask block: rel max err {err:.3e}")
    assert err <= BLOCK_REL_TOL


@pytest.mark.parametrize("B,T,kind,shape", [(2, 150, "random", "smollm2"), (2, 384, "random", "smollm2"),
                                           (2, 384, "prefix", "smollm2"), (1, 256, "random", "smollm3")])
def test_model_key_mask(S, B, T, kind, shape):
    # T = 384: whole 128-row blocks, so the O projection waits on the attention's
    # row-block flags instead of its completion.  "prefix": a padding-shaped mask
    # (each sequence hides a leading run of keys), so whole key tiles hide
    # nothing and take the attention's unmasked branch.  "smollm3": head_dim 128,
    # groups of 4, with the flags
    if shape == "smollm2":
        wl = W["smollm2_model_b8_t2048"].scaled(B=B, T=T, n_layers=2, vocab=1024)
    else:
        wl = W["smollm3_4blocks_b4_t4096"].scaled(kind="model", B=B, T=T, n_layers=2, vocab=1024)
    inp = synth.generate(wl, seed=62)
    if kind == "random":
        mask = _key_mask(B, T, 63)
        mask[:, 0] = 1
    else:
        mask = torch.ones(B, T, dtype=torch.uint8)
        mask[0, :5] = 0                               # rows 0..4 of sequence 0 see no key
        mask[1, :200] = 0
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.alloc_workspace(cfg, S.OP_MODEL, B, T)
    logits = torch.empty(B, T, 1024, dtype=torch.bfloat16, device="cuda")
    S.model_forward_masked(cfg, packed, dev.ids, logits, ws, mask.cuda())
    assert S.workspace_status(ws) == S.OK
    ref = O.model_forward(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                          inp.ids.numpy().astype(np.int64), key_mask=mask.numpy().astype(bool))
    got = np32(logits)
    cos, mabs = cosine(got, ref), max_abs(got, ref)
    print(f"key mask model: cos {cos:.7f} max abs {mabs:.3e}")
    assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (cos, mabs)


# ---------------------------------------------------------------- prefill on top of a cache
# ("model.py" (SmolLM2-135M) section 4 with past_key_value, section 7 with past_key_values)

def run_prefill_cache_case(S, wl, lengths, T, seed=0):
    wl = wl.scaled(B=len(lengths))
    inp = synth.generate(wl, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    ids = torch.randint(0, wl.vocab, (wl.B, T), generator=g).to(torch.int32)
    lens = torch.tensor(lengths, dtype=torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    ws = S.prefill_cache_workspace(cfg, wl.B, T, wl.s_max)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    k_new = torch.empty(L, B, KV, T, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits = torch.empty(B, T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.prefill_with_cache(cfg, packed, ids.cuda(), lens.cuda(), dev.k_cache, dev.v_cache, k_new, v_new, logits, ws)
    assert S.workspace_status(ws) == S.OK
    ref, kr, vr = O.prefill_with_cache(oracle_config(wl), oracle_layers(inp), np32(inp.embed), np32(inp.final_norm),
                                       ids.numpy().astype(np.int64), np.asarray(lengths), np32(inp.k_cache),
                                       np32(inp.v_cache))
    got = np32(logits)
    cos, mabs = cosine(got, ref), max_abs(got, ref)
    ek, ev = rel_max_err_bf16_out(np32(k_new), kr), rel_max_err_bf16_out(np32(v_new), vr)
    print(f"prefill with cache: cos {cos:.6f} max abs {mabs:.3e} k {ek:.3e} v {ev:.3e}")
    assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (cos, mabs)
    assert ek <= BLOCK_REL_TOL and ev <= BLOCK_REL_TOL, (ek, ev)


def test_prefill_with_cache_ragged(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=300, vocab=512)
    run_prefill_cache_case(S, wl, [0, 1, 130, 300], T=37, seed=70)


def test_prefill_with_cache_equal_lengths(S):
    # the attention takes the sequences longest cache first; equal lengths keep
    # their index order, and the order must still cover every sequence once
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=300, vocab=512)
    run_prefill_cache_case(S, wl, [130, 7, 130, 130, 0, 7, 300, 0], T=20, seed=72)


def test_prefill_with_cache_long_chunk_nope_window(S):
    wl = W["smollm2_decode_b64_cache4096"].scaled(n_layers=2, s_max=200, vocab=512, no_rope_layers=(1, 0),
                                                  sliding_window=(0, 150))
    run_prefill_cache_case(S, wl, [5, 200], T=260, seed=71)


def test_prefill_with_cache_head_dim_128(S):
    # SmolLM3-shaped layer (hd 128, groups of 4)
    wl = W["smollm2_decode_b64_cache4096"].scaled(
        hidden=2048, n_heads=16, n_kv_heads=4, head_dim=128, intermediate=11008, n_layers=1,
        vocab=512, s_max=300, rms_eps=1e-6, rope_theta=1e6, w_std=0.02)
    run_prefill_cache_case(S, wl, [0, 129, 300], T=45, seed=74)


def test_prefill_append_decode_chain(S):
    # prefill a chunk on top of the caches, append its keys and values, then
    # decode the next token: the GPU chain against the oracle's own chain
    wl = W["smollm2_decode_b64_cache4096"].scaled(B=3, n_layers=2, s_max=300, vocab=512,
                                                  sliding_window=(0, 40))
    inp = synth.generate(wl, seed=72)
    lengths = [0, 37, 250]
    T = 20
    g = torch.Generator().manual_seed(73)
    ids = torch.randint(0, wl.vocab, (wl.B, T), generator=g).to(torch.int32)
    nxt = torch.randint(0, wl.vocab, (wl.B,), generator=g).to(torch.int32)
    dev = to_device(inp)
    cfg = S.config_of(wl)
    packed = S.prepare_weights(cfg, dev.layers, dev.embed, dev.final_norm)
    L, B, KV, hd = wl.n_layers, wl.B, wl.n_kv_heads, wl.head_dim
    lens = torch.tensor(lengths, dtype=torch.int32)
    # GPU: prefill, append, decode
    ws = S.prefill_cache_workspace(cfg, B, T, wl.s_max)
    k_new = torch.empty(L, B, KV, T, hd, dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    logits_p = torch.empty(B, T, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.prefill_with_cache(cfg, packed, ids.cuda(), lens.cuda(), dev.k_cache, dev.v_cache, k_new, v_new,
                         logits_p, ws)
    assert S.workspace_status(ws) == S.OK
    kc, vc = dev.k_cache.clone(), dev.v_cache.clone()
    for b, Lb in enumerate(lengths):
        kc[:, b, :, Lb:Lb + T] = k_new[:, b]
        vc[:, b, :, Lb:Lb + T] = v_new[:, b]
    wsd = S.alloc_workspace(cfg, S.OP_DECODE, B, 1)
    k1 = torch.empty(L, B, KV, hd, dtype=torch.bfloat16, device="cuda")
    v1 = torch.empty_like(k1)
    logits_d = torch.empty(B, wl.vocab, dtype=torch.bfloat16, device="cuda")
    S.decode_step(cfg, packed, nxt.cuda(), (lens + T).cuda(), kc, vc, k1, v1, logits_d, wsd)
    assert S.workspace_status(wsd) == S.OK
    # oracle: the same chain on its own values
    oc, ol = oracle_config(wl), oracle_layers(inp)
    E, fn = np32(inp.embed), np32(inp.final_norm)
    ref_p, kr, vr = O.prefill_with_cache(oc, ol, E, fn, ids.numpy().astype(np.int64), np.asarray(lengths),
                                         np32(inp.k_cache), np32(inp.v_cache))
    okc = np32(inp.k_cache).astype(np.float64)
    ovc = np32(inp.v_cache).astype(np.float64)
    for b, Lb in enumerate(lengths):
        okc[:, b, :, Lb:Lb + T] = kr[:, b]
        ovc[:, b, :, Lb:Lb + T] = vr[:, b]
    ref_d, _, _ = O.decode_step(oc, ol, E, fn, nxt.numpy().astype(np.int64), np.asarray(lengths) + T, okc, ovc)
    for got, ref, what in ((np32(logits_p), ref_p, "prefill"), (np32(logits_d), ref_d, "decode")):
        cos, mabs = cosine(got, ref), max_abs(got, ref)
        print(f"chain {what}: cos {cos:.7f} max abs {mabs:.3e}")
        assert cos >= LOGITS_COS_MIN and mabs <= LOGITS_MAX_ABS, (what, cos, mabs)
