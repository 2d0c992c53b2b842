"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/smol.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import re

import pytest

from llama_decoder_forward_gb300 import build as B


@pytest.fixture(scope="module")
def smol():
    B.build()
    from llama_decoder_forward_gb300 import smol as S
    return S


def test_exports_every_declared_symbol(smol):
    names = smol.declared_symbols()
    assert len(names) >= 9
    for n in ("smol_block_forward", "smol_model_forward", "smol_decode_step", "smol_prepare_weights",
              "smol_workspace_bytes", "smol_packed_bytes", "smol_status_string"):
        assert n in names
    lib = ctypes.CDLL(smol.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_no_unexpected_exports(smol):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", smol.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {n for n in exported if n.startswith("smol_")}
    assert ours == set(smol.declared_symbols())


def _prototypes(text):
    """name -> list of parameter declarations of every smol_* prototype in the header."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    out = {}
    for m in re.finditer(r"(smol_\w+)\s*\(([^;{]*?)\)\s*;", text):
        args = " ".join(m.group(2).split())
        out[m.group(1)] = [] if args in ("", "void") else [a.strip() for a in args.split(",")]
    return out


def test_binding_matches_header_prototypes(smol):
    # every function the binding declares has the header's arity, and pointer
    # parameters are marshalled as pointers, integers as integers, floats as floats
    protos = _prototypes(open(smol.HEADER_PATH).read())
    ints = (ctypes.c_int, ctypes.c_uint, ctypes.c_size_t, ctypes.c_longlong)
    for name, (_, argtypes) in smol._SIGS.items():
        assert name in protos, name
        decl = protos[name]
        assert len(decl) == len(argtypes), (name, decl, argtypes)
        for d, t in zip(decl, argtypes):
            if "*" in d:
                assert t is ctypes.c_void_p or hasattr(t, "contents") or t is ctypes.c_char_p, (name, d, t)
            elif d.startswith("float"):
                assert t is ctypes.c_float, (name, d, t)
            else:
                assert t in ints, (name, d, t)
    assert set(protos) == set(smol._SIGS)


def _cfg(smol, **kw):
    base = dict(hidden=576, n_heads=9, n_kv_heads=3, head_dim=64, intermediate=1536, n_layers=30,
                vocab=49152, max_pos=8192, rms_eps=1e-5, rope_theta=1e5)
    base.update(kw)
    return smol.make_config(**base)


def test_size_queries(smol):
    cfg = _cfg(smol)
    d, hd, H, KV, I, V = 576, 64, 9, 3, 1536, 49152
    layer = (H + 2 * KV) * hd * d * 2 + d * H * hd * 2 + 2 * I * d * 2 + d * I * 2
    rope = (64 + 8192 // 64) * (hd // 2) * 8     # two-level (cos, sin) table
    total = smol.packed_bytes(cfg, 30, True)
    assert total >= rope + 30 * layer + 2 * V * d * 2
    assert total < rope + 30 * layer + 2 * V * d * 2 + 64 * 1024
    assert smol.packed_bytes(cfg, 1, False) < smol.packed_bytes(cfg, 2, False)
    assert smol.packed_bytes(cfg, 31, False) == 0
    ws = smol.workspace_bytes(cfg, smol.OP_MODEL, 8, 2048)
    M = 8 * 2048
    assert ws >= M * (2 * d + 2 * H * hd + 2 * KV * hd + I) * 2 + 2 * M * 4
    assert smol.workspace_bytes(cfg, smol.OP_DECODE, 64, 1) > 0
    # the decode batch of 64 fits the no-alloc variant's fixed 8 MiB scratch
    assert smol.workspace_bytes(cfg, smol.OP_DECODE, 64, 1) <= 8 << 20
    assert smol.workspace_bytes(cfg, 99, 8, 2048) == 0
    assert smol.workspace_bytes(_cfg(smol, head_dim=96, hidden=864), smol.OP_BLOCK, 1, 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96, hidden=864), -2),     # unsupported head_dim
    (dict(n_kv_heads=4), -2),                # H % KV != 0
    (dict(hidden=512), -2),                  # d != H * hd
    (dict(n_kv_heads=1, n_heads=9), 0),      # group 9 > 8 is rejected below separately
    (dict(intermediate=1500), -2),           # not a multiple of 64
    (dict(rms_eps=-1.0), -1),
    (dict(n_layers=0), -1),
])
def test_config_validation(smol, kw, code):
    cfg = _cfg(smol, **kw)
    fake = ctypes.c_void_p(0x10000)
    rc = smol.raw.smol_block_forward(ctypes.byref(cfg), fake, 0, fake, fake, 0, 1, 8, None, None, None,
                                     fake, 1 << 40, None)
    if code == 0:
        assert rc == -2   # group of 9 query heads per kv head exceeds 8
    else:
        assert rc == code


def test_per_block_variant_arrays(smol):
    # SmolLM3 NoPE flags must be 0 or 1 and windows non-negative; the arrays
    # have one entry per layer (the binding checks the length)
    n = 30
    ok = _cfg(smol, no_rope_layers=[1, 1, 1, 0] * 7 + [1, 1], sliding_window=[0, 128] * 15)
    assert smol.packed_bytes(ok, n, True) == smol.packed_bytes(_cfg(smol), n, True)
    assert smol.workspace_bytes(ok, smol.OP_DECODE, 64, 1) == smol.workspace_bytes(_cfg(smol), smol.OP_DECODE, 64, 1)
    assert smol.packed_bytes(_cfg(smol, no_rope_layers=[1] * 29 + [2]), n, True) == 0
    assert smol.packed_bytes(_cfg(smol, sliding_window=[0] * 29 + [-1]), n, True) == 0
    with pytest.raises(ValueError):
        _cfg(smol, sliding_window=[0] * 29)
    f = ctypes.c_void_p(0x10000)
    bad = _cfg(smol, sliding_window=[-5] + [0] * 29)
    assert smol.raw.smol_block_forward(ctypes.byref(bad), f, 0, f, f, 0, 1, 8, None, None, None, f,
                                       1 << 40, None) == -1


def test_masked_forward_needs_a_mask(smol):
    cfg = _cfg(smol)
    f = ctypes.c_void_p(0x10000)
    big = 1 << 40
    assert smol.raw.smol_block_forward_masked(ctypes.byref(cfg), f, 0, f, f, 0, 1, 8, None, None, None, f,
                                              big, None) == -1
    assert smol.raw.smol_model_forward_masked(ctypes.byref(cfg), f, f, 1, 8, None, f, f, big, None) == -1
    assert smol.raw.smol_block_forward_masked(ctypes.byref(cfg), f, 0, f, f, 0, 1, 8193, f, None, None, f,
                                              big, None) == -4


def test_prefill_with_cache_argument_errors(smol):
    cfg = _cfg(smol)
    f = ctypes.c_void_p(0x10000)
    big = 1 << 40
    pwc = smol.raw.smol_prefill_with_cache
    assert pwc(ctypes.byref(cfg), f, f, 2, 8, None, f, f, 64, f, f, f, f, big, None) == -1     # cache_len
    assert pwc(ctypes.byref(cfg), f, f, 2, 8, f, f, f, 0, f, f, f, f, big, None) == -1        # S_max
    assert pwc(ctypes.byref(cfg), f, f, 2, 8192, f, f, f, 64, f, f, f, f, big, None) == -4    # T >= max_pos
    assert pwc(ctypes.byref(cfg), f, f, 2, 8, f, f, f, 64, f, f, f, f, 16, None) == -5        # workspace
    hd96 = _cfg(smol, hidden=864, head_dim=96)
    assert pwc(ctypes.byref(hd96), f, f, 2, 8, f, f, f, 64, f, f, f, f, big, None) == -2    # head_dim
    assert smol.raw.smol_prefill_cache_workspace_bytes(ctypes.byref(cfg), 2, 8, 64) > \
        smol.workspace_bytes(cfg, smol.OP_MODEL, 2, 8)
    assert smol.last_launch_count() == 0


def test_sample_argument_errors(smol):
    f = ctypes.c_void_p(0x10000)
    smp = smol.raw.smol_sample
    nan = float("nan")
    assert smp(None, 4, 100, 100, 1.0, 0, 1.0, 1, f, f, None) == -1          # logits
    assert smp(f, 4, 100, 100, 1.0, 0, 1.0, 1, None, f, None) == -1          # uniform when sampling
    assert smp(f, 4, 100, 100, 1.0, 0, 1.0, 1, f, None, None) == -1          # next
    assert smp(f, 0, 100, 100, 1.0, 0, 1.0, 1, f, f, None) == -1             # B
    assert smp(f, 4, 0, 100, 1.0, 0, 1.0, 1, f, f, None) == -1               # V
    assert smp(f, 4, 100, 99, 1.0, 0, 1.0, 1, f, f, None) == -1              # ld < V
    assert smp(f, 4, 100, 100, nan, 0, 1.0, 1, f, f, None) == -1             # temperature
    assert smp(f, 4, 100, 100, 1.0, 0, nan, 1, f, f, None) == -1             # top_p
    assert smp(ctypes.c_void_p(0x10001), 4, 100, 100, 1.0, 0, 1.0, 1, f, f, None) == -3
    assert smp(f, 4, 100, 100, 1.0, 0, 1.0, 1, f, ctypes.c_void_p(0x10002), None) == -3
    assert smol.last_launch_count() == 0


def test_argument_errors_return_before_any_launch(smol):
    cfg = _cfg(smol)
    f = ctypes.c_void_p(0x10000)
    big = 1 << 40
    blk = smol.raw.smol_block_forward
    assert blk(ctypes.byref(cfg), None, 0, f, f, 0, 1, 8, None, None, None, f, big, None) == -1
    assert blk(ctypes.byref(cfg), f, 30, f, f, 0, 1, 8, None, None, None, f, big, None) == -1   # layer
    assert blk(ctypes.byref(cfg), f, 0, f, f, 0, 0, 8, None, None, None, f, big, None) == -1    # B
    assert blk(ctypes.byref(cfg), f, 0, f, f, 0, 1, 8193, None, None, None, f, big, None) == -4  # too long
    assert blk(ctypes.byref(cfg), f, 0, ctypes.c_void_p(0x10008), f, 0, 1, 8, None, None, None, f, big,
               None) == -3                                                                   # misaligned
    assert blk(ctypes.byref(cfg), f, 0, f, f, 0, 1, 8, None, None, None, f, 16, None) == -5      # workspace
    mdl = smol.raw.smol_model_forward
    assert mdl(ctypes.byref(cfg), f, f, 1, 8193, None, f, f, big, None) == -4
    assert mdl(ctypes.byref(cfg), f, ctypes.c_void_p(0x10002), 1, 8, None, f, f, big, None) == -3
    assert mdl(ctypes.byref(_cfg(smol, vocab=0)), f, f, 1, 8, None, f, f, big, None) == -1
    dec = smol.raw.smol_decode_step
    assert dec(ctypes.byref(cfg), f, f, f, 64, f, f, 0, f, f, f, f, big, None) == -1          # S_max
    assert dec(ctypes.byref(cfg), f, f, f, 64, f, f, 4096, f, f, f, f, 16, None) == -5
    assert smol.last_launch_count() == 0


def test_status_strings(smol):
    for code in range(-8, 1):
        assert smol.status_string(code)
    assert "unknown" in smol.status_string(-99)


def test_decode_next_and_append_argument_errors(smol):
    cfg = _cfg(smol)
    f = ctypes.c_void_p(0x10000)
    big = 1 << 40
    nxt = smol.raw.smol_decode_next
    nan = float("nan")
    # no `next`
    assert nxt(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, f, 1.0, 0, 1.0, 0, None, None, f, big, None) == -1
    # NaN temperature / top_p
    assert nxt(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, f, nan, 0, 1.0, 1, f, f, f, big, None) == -1
    assert nxt(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, f, 1.0, 0, nan, 1, f, f, f, big, None) == -1
    # sampling needs logits and uniform
    assert nxt(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, None, 1.0, 0, 1.0, 1, f, f, f, big, None) == -1
    assert nxt(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, f, 1.0, 0, 1.0, 1, None, f, f, big, None) == -1
    # greedy without logits is accepted up to the workspace check
    assert nxt(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, None, 1.0, 0, 1.0, 0, None, f, f, 16, None) == -5
    # smol_decode_step still needs its logits
    assert smol.raw.smol_decode_step(ctypes.byref(cfg), f, f, f, 4, f, f, 64, f, f, None, f, big, None) == -1
    app = smol.raw.smol_append_kv
    assert app(ctypes.byref(cfg), 4, None, f, f, f, 64, f, None) == -1
    assert app(ctypes.byref(cfg), 0, f, f, f, f, 64, f, None) == -1
    assert app(ctypes.byref(cfg), 4, f, f, f, f, 64, ctypes.c_void_p(0x10002), None) == -3
    assert smol.last_launch_count() == 0
