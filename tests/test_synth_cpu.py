"""The seeded synthetic inputs follow the stated recipe: one generator per
workload, draws in a fixed order, bf16-rounded normal weights of the stated
standard deviations, norm weights 1 + N(0, 0.1^2), token ids in [0, V), and
integer lengths uniform over an inclusive range.  CPU only."""
import numpy as np
import torch

from llama_decoder_forward_gb300 import synth


def _small(name, **kw):
    return synth.WORKLOADS[name].scaled(**kw)


def test_same_seed_same_inputs_other_seed_other_inputs():
    wl = _small("smollm2_decode_b64_cache4096", B=4, n_layers=2, s_max=64, vocab=512)
    a, b, c = synth.generate(wl, seed=3), synth.generate(wl, seed=3), synth.generate(wl, seed=4)
    assert torch.equal(a.ids, b.ids) and torch.equal(a.k_cache, b.k_cache) and torch.equal(a.lengths, b.lengths)
    for k in synth.LAYER_KEYS:
        assert torch.equal(a.layers[1][k], b.layers[1][k])
    assert not torch.equal(a.k_cache, c.k_cache)


def test_weight_and_activation_distributions():
    wl = _small("smollm2_block_b1_t128", B=4, T=256)
    inp = synth.generate(wl, seed=0)
    assert inp.x.dtype == torch.bfloat16 and tuple(inp.x.shape) == (4, 256, wl.hidden)
    x = inp.x.float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    lw = inp.layers[0]
    for k, shape in synth.layer_shapes(wl).items():
        t = lw[k]
        assert t.dtype == torch.bfloat16 and tuple(t.shape) == shape
        f = t.float()
        if k.endswith("norm"):
            assert abs(f.mean().item() - 1.0) < 0.02 and abs(f.std().item() - 0.1) < 0.01
        else:
            assert abs(f.mean().item()) < 0.002 and abs(f.std().item() / wl.w_std - 1.0) < 0.02
    # every value is exactly a bf16 number
    assert torch.equal(x.to(torch.bfloat16).float(), x)


def test_ids_and_inclusive_length_ranges():
    wl = _small("smollm2_decode_b64_cache4096", B=4000, n_layers=1, s_max=8, vocab=640, len_range=(3, 7))
    inp = synth.generate(wl, seed=1)
    ids = inp.ids.numpy()
    assert ids.min() >= 0 and ids.max() < 640 and inp.ids.dtype == torch.int32
    lens = inp.lengths.numpy()
    assert set(np.unique(lens)) == {3, 4, 5, 6, 7}        # both ends drawn
    k = inp.k_cache.float()
    assert abs(k.mean().item()) < 0.02 and abs(k.std().item() - 1.0) < 0.02


def test_left_padding_from_lengths():
    wl = _small("slm125m_block_leftpad_b16_t1024", B=64, T=40, len_range=(1, 40))
    inp = synth.generate(wl, seed=2)
    assert torch.equal(inp.valid_start, (40 - inp.lengths).to(torch.int32))
    assert inp.valid_start.min().item() >= 0 and inp.valid_start.max().item() <= 39


def test_stated_workload_shapes():
    W = synth.WORKLOADS
    assert (W["smollm2_model_b8_t2048"].B, W["smollm2_model_b8_t2048"].T) == (8, 2048)
    dec = W["smollm2_decode_b64_cache4096"]
    assert (dec.B, dec.s_max, dec.len_range, dec.n_layers) == (64, 4096, (1024, 4096), 30)
    s3 = W["smollm3_4blocks_b4_t4096"]
    assert (s3.hidden, s3.n_heads, s3.n_kv_heads, s3.head_dim, s3.intermediate, s3.rope_theta) == \
        (2048, 16, 4, 128, 11008, 1e6)
    lp = W["slm125m_block_leftpad_b16_t1024"]
    assert (lp.B, lp.T, lp.len_range, lp.hidden) == (16, 1024, (128, 1024), 768)
