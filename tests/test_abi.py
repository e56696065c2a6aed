"""The C ABI library: it loads, exports every declared entry point, and rejects
bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "pnb.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pnb_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    import transformer_decode_step_gb300 as pnb
    lib = ctypes.CDLL(pnb.LIB)
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pnb.EXPORTED)


def _cfg(**kw):
    import transformer_decode_step_gb300 as pnb
    base = dict(n_vocab=1024, n_embd=256, n_head=8, n_kv_head=4, n_layer=2, n_ff=688, n_ctx=128,
                rope_theta=1e4, rms_norm_eps=1e-5, sliding_window=0, expert_count=0,
                expert_used=0, dtype=0)
    base.update(kw)
    return pnb.pnb_config(**base)


def _weights(ptr=4096, n_layer=2, n_sets=1, router=False):
    import transformer_decode_step_gb300 as pnb
    arr = lambda n: (ctypes.c_void_p * n)(*([ptr] * n))
    keep = [arr(n_layer), arr(n_layer), arr(n_layer), arr(n_layer), arr(n_layer * n_sets),
            arr(n_layer * n_sets), arr(n_layer)]
    w = pnb.pnb_weights()
    w.tok_embd = w.out_norm = w.output = ptr
    c = lambda a: ctypes.cast(a, ctypes.c_void_p)
    w.attn_norm, w.wqkv, w.wo, w.ffn_norm = c(keep[0]), c(keep[1]), c(keep[2]), c(keep[3])
    w.w_gate_up, w.w_down = c(keep[4]), c(keep[5])
    w.w_router = c(keep[6]) if router else None
    return w, keep


def _create(cfg, w):
    import transformer_decode_step_gb300 as pnb
    h = ctypes.c_void_p()
    return pnb.pnb_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))


@pytest.mark.parametrize("bad", [
    dict(n_embd=250),                  # not a multiple of n_head
    dict(n_kv_head=3),                 # n_head % n_kv_head != 0
    dict(n_head=4, n_kv_head=4, n_embd=260),
    dict(n_ff=690),                    # not a multiple of 8
    dict(n_vocab=0), dict(n_layer=0), dict(n_ctx=0),
    dict(sliding_window=-1), dict(rope_theta=0.0), dict(rms_norm_eps=-1.0),
    dict(dtype=7), dict(rope_neox=2),
    dict(expert_count=8, expert_used=0), dict(expert_count=8, expert_used=9),
    dict(expert_count=65, expert_used=2), dict(expert_count=16, expert_used=9),
])
def test_invalid_configs_are_rejected_on_the_host(bad):
    import transformer_decode_step_gb300 as pnb
    w, keep = _weights(router=True, n_sets=max(1, bad.get("expert_count", 1)))
    assert _create(_cfg(**bad), w) == -1   # PNB_E_INVAL


def test_unsupported_head_dim():
    w, keep = _weights()
    assert _create(_cfg(n_embd=384, n_head=4, n_kv_head=4), w) == -5   # hd = 96


def test_null_and_misaligned_pointers():
    w, keep = _weights()
    w.output = None
    assert _create(_cfg(), w) == -2
    w, keep = _weights(ptr=4104)           # 8-byte aligned only
    assert _create(_cfg(), w) == -3
    w, keep = _weights()
    keep[1][1] = None                      # a NULL per-layer pointer
    assert _create(_cfg(), w) == -2
    w, keep = _weights()                   # MoE without router pointers
    assert _create(_cfg(expert_count=4, expert_used=2), w) == -2
    w, keep = _weights()                   # a bias array with a NULL layer entry
    bias = (ctypes.c_void_p * 2)(4096, None)
    w.bqkv = ctypes.cast(bias, ctypes.c_void_p)
    assert _create(_cfg(), w) == -2
    bias = (ctypes.c_void_p * 2)(4096, 4100)   # and one not 16-byte aligned
    w.bqkv = ctypes.cast(bias, ctypes.c_void_p)
    assert _create(_cfg(), w) == -3


def test_null_handles():
    import transformer_decode_step_gb300 as pnb
    assert pnb.pnb_forward(None, None, 0, None, None, None) == -2
    # sampler, draw counter and the begin / poll seam
    p = pnb.sampling_params(0.8, 1.1, 40, 0.95, 7)
    assert pnb.pnb_sample(None, None, None, ctypes.byref(p), None, 0, None, None) == -2
    assert pnb.pnb_sample_batch(None, None, 1, None, None, None, None, None, None) == -2
    assert pnb.pnb_state_set_draw(None, 3, None) == -2
    assert pnb.pnb_forward_begin(None, None, 0, None, None) == -2
    assert pnb.pnb_sample_begin(None, None, None, ctypes.byref(p), None, 0, None) == -2
    assert pnb.pnb_forward_poll(None, None, None) == -2
    assert pnb.pnb_state_stream(None, None) == -2
    assert pnb.pnb_prefill(None, None, None, 4, None, None, None) == -2
    assert pnb.pnb_strerror(-12).startswith(b"a begun step")
    assert p.temperature == pytest.approx(0.8) and p.top_k == 40 and p.seed == 7
    assert pnb.pnb_state_new(None, None, 0, None) == -2
    assert pnb.pnb_state_kv_bytes(None) == 0
    assert pnb.pnb_strerror(-4) == b"position reached n_ctx"
