"""GB300 (sm_103a) transformer decode step: Python binding of libpnb.so.

The binding only marshals arguments to the C ABI declared in include/pnb.h;
every step of the decode path runs in the library's CUDA kernels.  PyTorch is
used by callers for device memory and streams only.  Importing this package
fails loudly when the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from ._build import LIB

if not os.path.exists(LIB):
    raise ImportError(f"{LIB} is missing: build it with __graft_entry__.build() "
                      "(the decode step has no non-CUDA implementation)")

_lib = ctypes.CDLL(LIB)

PNB_F32, PNB_BF16, PNB_Q8_0, PNB_Q4_0 = 0, 1, 2, 3
PNB_TOKEN_PREV = -1
PNB_DEV_ERR_TOKEN, PNB_DEV_ERR_TIMEOUT = 1, 2
(PNB_KERNEL_QKV, PNB_KERNEL_ATTN, PNB_KERNEL_OPROJ, PNB_KERNEL_ROUTER, PNB_KERNEL_GATE_UP,
 PNB_KERNEL_DOWN, PNB_KERNEL_LM_HEAD) = range(7)
ERRORS = {0: "PNB_OK", -1: "PNB_E_INVAL", -2: "PNB_E_NULL", -3: "PNB_E_ALIGN",
          -4: "PNB_E_CTX_FULL", -5: "PNB_E_UNSUPPORTED", -6: "PNB_E_CUDA", -7: "PNB_E_TOKEN",
          -8: "PNB_E_DEVICE", -9: "PNB_E_NOMEM", -10: "PNB_E_WRONG_DEVICE", -11: "PNB_E_TOO_LARGE",
          -12: "PNB_E_BUSY"}


class pnb_config(ctypes.Structure):
    _fields_ = [("n_vocab", ctypes.c_int32), ("n_embd", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_kv_head", ctypes.c_int32),
                ("n_layer", ctypes.c_int32), ("n_ff", ctypes.c_int32), ("n_ctx", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rms_norm_eps", ctypes.c_double),
                ("sliding_window", ctypes.c_int32), ("expert_count", ctypes.c_int32),
                ("expert_used", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("rope_neox", ctypes.c_int32)]


class pnb_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("tok_embd", "out_norm", "output", "attn_norm", "wqkv", "wo", "ffn_norm",
                 "w_router", "w_gate_up", "w_down", "bqkv")]


class pnb_sampling_params(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("repeat_penalty", ctypes.c_float),
                ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float), ("seed", ctypes.c_uint64)]


def sampling_params(temperature: float = 0.0, repeat_penalty: float = 1.0, top_k: int = 0,
                    top_p: float = 1.0, seed: int = 0) -> pnb_sampling_params:
    return pnb_sampling_params(temperature, repeat_penalty, top_k, top_p, seed)


class pnb_activations(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "q", "attn", "h")]


_p, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_SIGS = {
    "pnb_model_create": (_i32, [_p, _p, _p]),
    "pnb_model_free": (None, [_p]),
    "pnb_state_kv_bytes": (_sz, [_p]),
    "pnb_state_new": (_i32, [_p, _p, _sz, _p]),
    "pnb_state_free": (None, [_p]),
    "pnb_state_reset": (_i32, [_p, _p]),
    "pnb_state_set_pos": (_i32, [_p, _i32, _p]),
    "pnb_state_get_pos": (_i32, [_p, _p]),
    "pnb_state_check": (_i32, [_p, _p]),
    "pnb_forward": (_i32, [_p, _p, _i32, _p, _p, _p]),
    "pnb_forward_batch": (_i32, [_p, _p, _i32, _p, _p, _p, _p]),
    "pnb_prefill": (_i32, [_p, _p, _p, _i32, _p, _p, _p]),
    "pnb_sample": (_i32, [_p, _p, _p, _p, _p, _i32, _p, _p]),
    "pnb_sample_batch": (_i32, [_p, _p, _i32, _p, _p, _p, _p, _p, _p]),
    "pnb_state_set_draw": (_i32, [_p, ctypes.c_uint32, _p]),
    "pnb_forward_begin": (_i32, [_p, _p, _i32, _p, _p]),
    "pnb_sample_begin": (_i32, [_p, _p, _p, _p, _p, _i32, _p]),
    "pnb_forward_poll": (_i32, [_p, _p, _p]),
    "pnb_state_stream": (_i32, [_p, _p]),
    "pnb_model_set_graphs": (_i32, [_p, _i32]),
    "pnb_model_set_deterministic_batch": (_i32, [_p, _i32]),
    "pnb_model_set_tensor_attention": (_i32, [_p, _i32]),
    "pnb_model_is_tensor_attention": (_i32, [_p]),
    "pnb_step_kernel_count": (_i32, [_p, _i32]),
    "pnb_state_activations": (_i32, [_p, _p]),
    "pnb_step_kernel": (_i32, [_p, _p, _i32, _i32, _p]),
    "pnb_state_set_trace": (_i32, [_p, _p, _sz]),
    "pnb_attention_decode_static": (_i32, [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                           _p, _p, _p]),
    "pnb_state_wait_probe": (_i32, [_p, ctypes.c_uint64, _p]),
    "pnb_strerror": (ctypes.c_char_p, [_i32]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn

EXPORTED = tuple(_SIGS)


def attention_decode_static(q, k, v, dtype: int, n_head: int, n_kv_head: int, head_dim: int,
                            cap: int, window: int, pos: int, out, err=None, stream=None):
    """One layer's decode attention with no device allocation
    (pnb_attention_decode_static): the library's static scratch array is used.
    ``err`` (optional device int32) receives the call's device error bits."""
    check(pnb_attention_decode_static(_ptr(q), _ptr(k), _ptr(v), dtype, n_head, n_kv_head,
                                      head_dim, cap, window, pos, _ptr(out), _ptr(err),
                                      _stream(stream)),
          "pnb_attention_decode_static")


class PnbError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({pnb_strerror(code).decode()})")
        self.code = code


def check(code: int, what: str):
    if code != 0:
        raise PnbError(code, what)


def _ptr(t) -> Optional[int]:
    """Device pointer of a torch tensor (or an int), None for None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Model:
    """A pnb_model over caller-owned device weights.

    cfg: pnb_config.  Pointers (ints): tok_embd, out_norm, output; per-layer
    lists attn_norm, wqkv, wo, ffn_norm, w_router (MoE) and w_gate_up, w_down
    with n_layer * max(1, expert_count) entries (layout: include/pnb.h)."""

    def __init__(self, cfg: pnb_config, *, tok_embd, out_norm, output, attn_norm, wqkv, wo,
                 ffn_norm, w_gate_up, w_down, w_router=None, bqkv=None, keepalive=None):
        self.cfg = cfg
        self._keep = [keepalive]
        arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs) if xs else None
        self._arrays = [arr(attn_norm), arr(wqkv), arr(wo), arr(ffn_norm), arr(w_router),
                        arr(w_gate_up), arr(w_down), arr(bqkv)]
        w = pnb_weights()
        w.tok_embd, w.out_norm, w.output = tok_embd, out_norm, output
        (an, qkv, o, fn, rt, gu, dn, bq) = self._arrays
        cast = lambda a: ctypes.cast(a, ctypes.c_void_p) if a is not None else None
        w.attn_norm, w.wqkv, w.wo, w.ffn_norm = cast(an), cast(qkv), cast(o), cast(fn)
        w.w_router, w.w_gate_up, w.w_down, w.bqkv = cast(rt), cast(gu), cast(dn), cast(bq)
        h = ctypes.c_void_p()
        check(pnb_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)),
              "pnb_model_create")
        self._h = h.value

    def __del__(self):
        if getattr(self, "_h", None):
            pnb_model_free(self._h)
            self._h = None

    @property
    def handle(self) -> int:
        return self._h

    def kv_bytes(self) -> int:
        return int(pnb_state_kv_bytes(self._h))

    def set_graphs(self, enable: bool):
        check(pnb_model_set_graphs(self._h, 1 if enable else 0), "pnb_model_set_graphs")

    def set_deterministic_batch(self, enable: bool):
        check(pnb_model_set_deterministic_batch(self._h, 1 if enable else 0),
              "pnb_model_set_deterministic_batch")

    def set_tensor_attention(self, enable: bool):
        check(pnb_model_set_tensor_attention(self._h, 1 if enable else 0),
              "pnb_model_set_tensor_attention")

    @property
    def tensor_attention(self) -> bool:
        return bool(pnb_model_is_tensor_attention(self._h))

    def step_kernel_count(self, batch: int = 0) -> int:
        return int(pnb_step_kernel_count(self._h, batch))

    def new_state(self, kv=None) -> "State":
        """A state over `kv` (a device tensor of at least kv_bytes()), allocated if None."""
        if kv is None:
            import torch
            kv = torch.zeros(self.kv_bytes(), dtype=torch.uint8, device="cuda")
        return State(self, kv)

    def forward_batch(self, states: Sequence["State"], tokens=None, logits=None, argmax=None,
                      stream=None):
        arr = (ctypes.c_void_p * len(states))(*[s.handle for s in states])
        check(pnb_forward_batch(self._h, arr, len(states), _ptr(tokens), _stream(stream),
                                _ptr(logits), _ptr(argmax)), "pnb_forward_batch")


    def sample_batch(self, states: Sequence["State"], logits, params, recent=None, tokens=None,
                     stream=None):
        """pnb_sample_batch: params a list of pnb_sampling_params (one per state),
        recent a list of device int32 tensors (or None) - the penalty windows."""
        n = len(states)
        arr = (ctypes.c_void_p * n)(*[s.handle for s in states])
        ps = (pnb_sampling_params * n)(*params)
        rec = nrec = None
        if recent is not None:
            rec = (ctypes.c_void_p * n)(*[_ptr(r) if r is not None and r.numel() else None
                                          for r in recent])
            nrec = (ctypes.c_int32 * n)(*[int(r.numel()) if r is not None else 0 for r in recent])
        check(pnb_sample_batch(self._h, arr, n, _ptr(logits), ps, rec, nrec, _stream(stream),
                               _ptr(tokens)), "pnb_sample_batch")


class State:
    def __init__(self, model: Model, kv):
        self.model = model
        self.kv = kv
        h = ctypes.c_void_p()
        check(pnb_state_new(model.handle, _ptr(kv), kv.numel() * kv.element_size(),
                            ctypes.byref(h)), "pnb_state_new")
        self._h = h.value

    def __del__(self):
        if getattr(self, "_h", None):
            pnb_state_free(self._h)
            self._h = None

    @property
    def handle(self) -> int:
        return self._h

    def forward(self, token: int, logits=None, argmax=None, stream=None):
        check(pnb_forward(self.model.handle, self._h, token, _stream(stream), _ptr(logits),
                          _ptr(argmax)), "pnb_forward")

    def prefill(self, tokens, logits=None, argmax=None, stream=None):
        """Feed the prompt `tokens` (device int32 tensor [T]); logits [T][n_vocab]
        and argmax [T] optional device tensors."""
        check(pnb_prefill(self.model.handle, self._h, _ptr(tokens), int(tokens.numel()),
                          _stream(stream), _ptr(logits), _ptr(argmax)), "pnb_prefill")

    def sample(self, logits, params: pnb_sampling_params, recent=None, token=None, stream=None):
        """Draw the next token from `logits` (changed in place); `recent` a device
        int32 tensor of the penalty window; `token` an optional device int32 [1]."""
        n = int(recent.numel()) if recent is not None else 0
        check(pnb_sample(self.model.handle, self._h, _ptr(logits), ctypes.byref(params),
                         _ptr(recent) if n else None, n, _stream(stream), _ptr(token)),
              "pnb_sample")

    def set_draw(self, draw: int, stream=None):
        check(pnb_state_set_draw(self._h, draw, _stream(stream)), "pnb_state_set_draw")

    # begin / poll: the step (and a sampling) on the state's own stream
    def forward_begin(self, token: int, logits=None, argmax=None):
        self._begun_logits = logits
        check(pnb_forward_begin(self.model.handle, self._h, token, _ptr(logits), _ptr(argmax)),
              "pnb_forward_begin")

    def sample_begin(self, logits, params: pnb_sampling_params, recent=None, token=None):
        n = int(recent.numel()) if recent is not None else 0
        check(pnb_sample_begin(self.model.handle, self._h, _ptr(logits), ctypes.byref(params),
                               _ptr(recent) if n else None, n, _ptr(token)), "pnb_sample_begin")

    def poll(self) -> bool:
        """True when the begun work is done (raises PnbError on its errors)."""
        out = ctypes.c_void_p()
        rc = pnb_forward_poll(self.model.handle, self._h, ctypes.byref(out))
        if rc == 1:
            return False
        check(rc, "pnb_forward_poll")
        return True

    def stream(self) -> int:
        """The state's own CUDA stream (as an int handle)."""
        out = ctypes.c_void_p()
        check(pnb_state_stream(self._h, ctypes.byref(out)), "pnb_state_stream")
        return out.value or 0

    def reset(self, stream=None):
        check(pnb_state_reset(self._h, _stream(stream)), "pnb_state_reset")

    def set_pos(self, pos: int, stream=None):
        check(pnb_state_set_pos(self._h, pos, _stream(stream)), "pnb_state_set_pos")

    @property
    def pos(self) -> int:
        p = ctypes.c_int32()
        check(pnb_state_get_pos(self._h, ctypes.byref(p)), "pnb_state_get_pos")
        return p.value

    def device_error(self) -> int:
        e = ctypes.c_int32()
        rc = pnb_state_check(self._h, ctypes.byref(e))
        if rc not in (0, -8):
            check(rc, "pnb_state_check")
        return e.value

    def wait_probe(self, limit_ns: int, stream=None):
        """Make one bounded device wait run out after limit_ns (pnb_state_wait_probe)."""
        check(pnb_state_wait_probe(self._h, limit_ns, _stream(stream)), "pnb_state_wait_probe")

    def run_kernel(self, kind: int, layer: int, stream=None):
        """One kernel of the step in isolation (pnb_step_kernel)."""
        check(pnb_step_kernel(self.model.handle, self._h, kind, layer, _stream(stream)),
              "pnb_step_kernel")

    def set_trace(self, buf):
        """Per-CTA timestamps of the step's kernels into `buf` (device int64 tensor) or off."""
        nbytes = buf.numel() * buf.element_size() if buf is not None else 0
        check(pnb_state_set_trace(self._h, _ptr(buf), nbytes), "pnb_state_set_trace")

    def activations(self) -> dict:
        a = pnb_activations()
        check(pnb_state_activations(self._h, ctypes.byref(a)), "pnb_state_activations")
        return {"x": a.x, "q": a.q, "attn": a.attn, "h": a.h}


from .synthetic import SynthModel  # noqa: E402  (generated-weight models for tests / bench)
