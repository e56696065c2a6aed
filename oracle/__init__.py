"""CPU oracle of the transformer decode step - TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never loads it and
never falls back to it.  The forward itself is plain C (``oracle.c``):
fp32 vectors between operations, fp64 accumulation inside each reduction,
OpenMP over output rows and attention heads.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, special cases that reduce to library routines,
and a whole step composed of library routines).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

import synth
from synth.workloads import KV_SIGMA, WEIGHT_SIGMA, Shape, weight_specs

_DIR = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_DIR, "liboracle.so")
_ROOT = os.path.dirname(_DIR)


def build_commands():
    return [["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-fno-fast-math",
             "-ffp-contract=off", "-I", _ROOT, "-o", LIB, os.path.join(_DIR, "oracle.c"), "-lm"]]


class OrcConfig(ctypes.Structure):
    _fields_ = [("n_vocab", ctypes.c_int32), ("n_embd", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_kv_head", ctypes.c_int32),
                ("n_layer", ctypes.c_int32), ("n_ff", ctypes.c_int32), ("n_ctx", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rms_norm_eps", ctypes.c_double),
                ("sliding_window", ctypes.c_int32), ("expert_count", ctypes.c_int32),
                ("expert_used", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("qkv_bias", ctypes.c_int32), ("rope_neox", ctypes.c_int32)]


class OrcTensor(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("data", ctypes.c_void_p), ("key", ctypes.c_uint64),
                ("sigma", ctypes.c_float), ("value", ctypes.c_float)]


EXPLICIT, SYNTH, CONST = 0, 1, 2
# per-layer slots (oracle.c); experts follow as (gate, up, down) triples
L_ATTN_NORM, L_WQ, L_WK, L_WV, L_WO, L_FFN_NORM, L_WROUTER, L_EXPERT0 = range(8)

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        p, i64, i32, f, d = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                             ctypes.c_double)
        L.orc_round_bf16.restype = f
        L.orc_round_bf16.argtypes = [f]
        L.orc_matvec.argtypes = [p, i64, i64, i32, p, p]
        L.orc_rmsnorm.argtypes = [p, p, i64, d, p]
        L.orc_rope.argtypes = [p, i32, i64, d]
        L.orc_rope_neox.argtypes = [p, i32, i64, d]
        L.orc_attention.argtypes = [p, p, p, i32, i32, i32, i64, i32, p]
        L.orc_silu.restype = d
        L.orc_silu.argtypes = [d]
        L.orc_ffn.argtypes = [p, p, p, i64, i64, i32, p, p]
        L.orc_topk_softmax.argtypes = [p, i32, i32, p, p]
        L.orc_argmax.restype = ctypes.c_int32
        L.orc_argmax.argtypes = [p, i64]
        L.orc_model_new.restype = p
        L.orc_model_new.argtypes = [p, p, p]
        L.orc_model_free.argtypes = [p]
        L.orc_state_new.restype = p
        L.orc_state_new.argtypes = [p]
        L.orc_state_free.argtypes = [p]
        L.orc_state_reset.argtypes = [p]
        L.orc_state_pos.restype = i64
        L.orc_state_pos.argtypes = [p]
        L.orc_state_set_pos.argtypes = [p, i64]
        L.orc_state_route_margin.restype = d
        L.orc_state_route_margin.argtypes = [p]
        L.orc_state_kv.restype = p
        L.orc_state_kv.argtypes = [p, i32, i32]
        L.orc_state_prefill_synth.restype = i32
        L.orc_state_prefill_synth.argtypes = [p, ctypes.c_uint64, ctypes.c_uint32, i64, i64, f]
        L.orc_forward.restype = i32
        L.orc_forward.argtypes = [p, p, ctypes.c_int32, p, p]
        L.orc_embed.restype = i32
        L.orc_embed.argtypes = [p, ctypes.c_int32, p]
        L.orc_layer.restype = i32
        L.orc_layer.argtypes = [p, p, i32, p]
        L.orc_head.argtypes = [p, p, p, p]
        L.orc_sample.restype = ctypes.c_int32
        L.orc_sample.argtypes = [p, i64, f, f, p, i64, i64, f, d, p, p, p]
        L.orc_sample_uniform.restype = d
        L.orc_sample_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.orc_set_threads.argtypes = [i32]
        L.orc_max_threads.restype = i32
        _lib = L
    return _lib


def set_threads(n: int):
    lib().orc_set_threads(n)


def max_threads() -> int:
    return int(lib().orc_max_threads())


# -------------------------------------------------------------- building blocks

def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def round_bf16(x: float) -> float:
    return float(lib().orc_round_bf16(x))


def _explicit(a: np.ndarray) -> OrcTensor:
    return OrcTensor(mode=EXPLICIT, data=a.ctypes.data)


def matvec(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    w, x = _f32(w), _f32(x)
    y = np.empty(w.shape[0], dtype=np.float32)
    t = _explicit(w)
    lib().orc_matvec(ctypes.byref(t), w.shape[0], w.shape[1], 0, x.ctypes.data, y.ctypes.data)
    return y


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x, w = _f32(x), _f32(w)
    out = np.empty_like(x)
    lib().orc_rmsnorm(x.ctypes.data, w.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = _f32(v).copy()
    lib().orc_rope(v.ctypes.data, v.size, pos, theta)
    return v


def rope_neox(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = _f32(v).copy()
    lib().orc_rope_neox(v.ctypes.data, v.size, pos, theta)
    return v


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_head: int, n_kv: int, p: int,
              window: int = 0) -> np.ndarray:
    """q [n_head*hd]; K, V [n_pos][n_kv][hd] with positions 0..p valid."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    hd = q.size // n_head
    o = np.empty(n_head * hd, dtype=np.float32)
    lib().orc_attention(q.ctypes.data, K.ctypes.data, V.ctypes.data, n_head, n_kv, hd, p, window,
                        o.ctypes.data)
    return o


def silu(z: float) -> float:
    return float(lib().orc_silu(z))


def ffn(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, xn: np.ndarray) -> np.ndarray:
    wg, wu, wd, xn = _f32(wg), _f32(wu), _f32(wd), _f32(xn)
    out = np.empty(wd.shape[0], dtype=np.float32)
    tg, tu, td = _explicit(wg), _explicit(wu), _explicit(wd)
    lib().orc_ffn(ctypes.byref(tg), ctypes.byref(tu), ctypes.byref(td), wd.shape[0], wg.shape[0],
                  0, xn.ctypes.data, out.ctypes.data)
    return out


def topk_softmax(r: np.ndarray, k: int):
    r = _f32(r)
    idx = np.empty(k, dtype=np.int32)
    g = np.empty(k, dtype=np.float64)
    lib().orc_topk_softmax(r.ctypes.data, r.size, k, idx.ctypes.data, g.ctypes.data)
    return idx, g


def argmax(x: np.ndarray) -> int:
    x = _f32(x)
    return int(lib().orc_argmax(x.ctypes.data, x.size))


def sample(logits, temperature: float, repeat_penalty: float = 1.0, recent=(), top_k: int = 0,
           top_p: float = 1.0, u: float = 0.0):
    """(token, kept token ids in draw order, their cumulative probabilities)."""
    x = _f32(logits)
    rec = np.asarray(recent, dtype=np.int32)
    V = x.size
    idx = np.empty(V, dtype=np.int32)
    cum = np.empty(V, dtype=np.float64)
    n = ctypes.c_int64(0)
    tok = lib().orc_sample(x.ctypes.data, V, temperature, repeat_penalty,
                           rec.ctypes.data if rec.size else None, rec.size, top_k, top_p, u,
                           idx.ctypes.data, cum.ctypes.data, ctypes.byref(n))
    return int(tok), idx[:n.value].copy(), cum[:n.value].copy()


def sample_uniform(seed: int, draw: int) -> float:
    return float(lib().orc_sample_uniform(seed, draw))


# ----------------------------------------------------------------- whole model

def _config(shape: Shape) -> OrcConfig:
    return OrcConfig(shape.n_vocab, shape.n_embd, shape.n_head, shape.n_kv_head, shape.n_layer,
                     shape.n_ff, shape.n_ctx, shape.rope_theta, shape.rms_norm_eps,
                     shape.sliding_window, shape.expert_count, shape.expert_used, shape.dtype,
                     int(shape.qkv_bias), int(shape.rope_neox))


class Model:
    """Oracle model.  Weights are generated from ``seed`` (synth recipe) unless
    ``arrays`` supplies explicit values: {name: array} for globals ("tok_embd",
    "out_norm", "output") and {(name, layer, expert): array} for layer tensors.
    Explicit values must already be storage values (bf16-representable for bf16)."""

    def __init__(self, shape: Shape, seed: Optional[int] = None,
                 arrays: Optional[Dict] = None):
        self.shape = shape
        self._keep = []  # explicit arrays must outlive the C model
        nsets = max(1, shape.expert_count)
        slots = 7 + 3 * nsets + 3   # ..., experts, then the q / k / v biases
        glob = (OrcTensor * 3)()
        layers = (OrcTensor * (shape.n_layer * slots))()
        for spec in weight_specs(shape):
            if spec.name in ("tok_embd", "out_norm", "output"):
                akey = spec.name
                tgt = glob[{"tok_embd": 0, "out_norm": 1, "output": 2}[spec.name]]
            else:
                akey = (spec.name, spec.layer, spec.sub)
                base = spec.layer * slots
                slot = {"attn_norm": L_ATTN_NORM, "wq": L_WQ, "wk": L_WK, "wv": L_WV,
                        "wo": L_WO, "ffn_norm": L_FFN_NORM, "wrouter": L_WROUTER,
                        "wgate": L_EXPERT0 + 3 * spec.sub, "wup": L_EXPERT0 + 3 * spec.sub + 1,
                        "wdown": L_EXPERT0 + 3 * spec.sub + 2,
                        "bq": L_EXPERT0 + 3 * nsets, "bk": L_EXPERT0 + 3 * nsets + 1,
                        "bv": L_EXPERT0 + 3 * nsets + 2}[spec.name]
                tgt = layers[base + slot]
            if arrays is not None and akey in arrays:
                a = _f32(arrays[akey]).reshape(spec.rows, spec.cols)
                self._keep.append(a)
                tgt.mode, tgt.data = EXPLICIT, a.ctypes.data
            elif spec.const is not None:
                tgt.mode, tgt.value = CONST, spec.const
            else:
                if seed is None:
                    raise ValueError(f"no values for {akey} and no seed")
                tgt.mode, tgt.key, tgt.sigma = SYNTH, spec.key(seed), spec.sigma
        cfg = _config(shape)
        self._h = lib().orc_model_new(ctypes.byref(cfg), glob, layers)
        if not self._h:
            raise ValueError("oracle rejected the config")

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_model_free(self._h)
            self._h = None

    def new_state(self) -> "State":
        return State(self)


class State:
    def __init__(self, model: Model):
        self.model = model
        self._h = lib().orc_state_new(model._h)
        if not self._h:
            raise MemoryError("oracle state allocation failed")

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_state_free(self._h)
            self._h = None

    @property
    def pos(self) -> int:
        return int(lib().orc_state_pos(self._h))

    @pos.setter
    def pos(self, p: int):
        lib().orc_state_set_pos(self._h, p)

    def reset(self):
        lib().orc_state_reset(self._h)

    @property
    def route_margin(self) -> float:
        """After a forward of a MoE model: over its layers, the smallest gap between
        the k-th chosen router logit and the best unchosen one, relative to the
        layer's largest |logit| (a routing near-tie when small); inf for dense."""
        return float(lib().orc_state_route_margin(self._h))

    def kv(self, layer: int, kind: int) -> np.ndarray:
        """Writable view [n_ctx][n_kv_head][head_dim] of one layer's K (0) or V (1)."""
        s = self.model.shape
        ptr = lib().orc_state_kv(self._h, layer, kind)
        n = s.n_ctx * s.n_kv_head * s.head_dim
        arr = np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ctypes.c_float)), shape=(n,))
        return arr.reshape(s.n_ctx, s.n_kv_head, s.head_dim)

    def prefill_synth(self, seed: int, sub: int, j_lo: int, P: int, sigma: float = KV_SIGMA):
        rc = lib().orc_state_prefill_synth(self._h, seed, sub, j_lo, P, sigma)
        if rc != 0:
            raise ValueError("bad pre-fill range")

    def forward(self, token: int, want_logits: bool = True):
        """One decode step; returns (logits or None, argmax)."""
        V = self.model.shape.n_vocab
        logits = np.empty(V, dtype=np.float32) if want_logits else None
        am = ctypes.c_int32(-1)
        rc = lib().orc_forward(self.model._h, self._h, token,
                               logits.ctypes.data if logits is not None else None,
                               ctypes.byref(am))
        if rc == -1:
            raise ValueError(f"token {token} out of range")
        if rc == -2:
            raise ValueError("KV cache full")
        return logits, int(am.value)

    # The step in parts (same arithmetic as forward): embed, each layer, head.
    def embed(self, token: int) -> np.ndarray:
        x = np.empty(self.model.shape.n_embd, dtype=np.float32)
        if lib().orc_embed(self.model._h, token, x.ctypes.data) != 0:
            raise ValueError(f"token {token} out of range")
        return x

    def layer(self, l: int, x: np.ndarray) -> np.ndarray:
        """Layer l for the token at the current pos (pos is not advanced); x in place."""
        if lib().orc_layer(self.model._h, self._h, l, x.ctypes.data) != 0:
            raise ValueError("KV cache full")
        return x

    def head(self, x: np.ndarray, want_logits: bool = True):
        V = self.model.shape.n_vocab
        logits = np.empty(V, dtype=np.float32) if want_logits else None
        am = ctypes.c_int32(-1)
        lib().orc_head(self.model._h, x.ctypes.data,
                       logits.ctypes.data if logits is not None else None, ctypes.byref(am))
        return logits, int(am.value)
