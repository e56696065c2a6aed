"""Models with generated weights in the library's device layout.

The seeded generator (``synth``) writes every weight and pre-filled cache
entry straight into device memory; the values equal the host generator's, so
the CPU oracle sees the same model.  Layout per include/pnb.h: Wq, Wk, Wv
rows stacked into one [(n_head + 2 n_kv_head) hd][n_embd] matrix; gate and
up rows interleaved (row 2i = gate row i, row 2i+1 = up row i); Q8 rows hold
their int8 values, then one fp16 scale per 32.
"""
from __future__ import annotations

import ctypes

import synth
from synth.workloads import BIAS_SIGMA, KV_SIGMA, WEIGHT_SIGMA, Shape, kv_prefill_range


class _Arena:
    """One flat device buffer carved into 256-byte aligned tensors."""

    def __init__(self):
        self.items = []
        self.size = 0

    def add(self, nbytes: int) -> int:
        off = self.size
        self.size += (nbytes + 255) // 256 * 256
        return off


class SynthModel:
    def __init__(self, shape: Shape, seed: int, device=None, stream=None):
        import torch

        from . import Model, pnb_config

        self.shape, self.seed = shape, seed
        dev = torch.device(device or "cuda")
        s = shape
        mb = s.matrix_bytes
        E, H, Hkv, hd, F, V, L = (s.n_embd, s.n_head, s.n_kv_head, s.head_dim, s.n_ff, s.n_vocab,
                                  s.n_layer)
        nsets = max(1, s.expert_count)
        ar = _Arena()
        o_emb, o_onorm, o_out = ar.add(mb(V, E)), ar.add(E * 4), ar.add(mb(V, E))
        lay = []
        for l in range(L):
            d = {"attn_norm": ar.add(E * 4), "wqkv": ar.add(mb((H + 2 * Hkv) * hd, E)),
                 "wo": ar.add(mb(E, H * hd)), "ffn_norm": ar.add(E * 4)}
            if s.qkv_bias:
                d["bqkv"] = ar.add((H + 2 * Hkv) * hd * 4)
            if s.expert_count > 0:
                d["w_router"] = ar.add(mb(s.expert_count, E))
            d["w_gate_up"] = [ar.add(mb(2 * F, E)) for _ in range(nsets)]
            d["w_down"] = [ar.add(mb(E, F)) for _ in range(nsets)]
            lay.append(d)
        self.buf = torch.empty(ar.size, dtype=torch.uint8, device=dev)
        base = self.buf.data_ptr()
        st = (stream or torch.cuda.current_stream(dev)).cuda_stream
        dt = s.dtype
        key = lambda kind, layer=0, sub=0: synth.key(seed, kind, layer, sub)

        synth.dev_fill_matrix(base + o_emb, dt, 0, 1, V, E, key(synth.TOK_EMBD), WEIGHT_SIGMA, st)
        synth.dev_fill_const(base + o_onorm, synth.F32, E, 1.0, st)
        synth.dev_fill_matrix(base + o_out, dt, 0, 1, V, E, key(synth.OUTPUT), WEIGHT_SIGMA, st)
        for l, d in enumerate(lay):
            synth.dev_fill_const(base + d["attn_norm"], synth.F32, E, 1.0, st)
            synth.dev_fill_const(base + d["ffn_norm"], synth.F32, E, 1.0, st)
            q = base + d["wqkv"]
            synth.dev_fill_matrix(q, dt, 0, 1, H * hd, E, key(synth.WQ, l), WEIGHT_SIGMA, st)
            synth.dev_fill_matrix(q, dt, H * hd, 1, Hkv * hd, E, key(synth.WK, l), WEIGHT_SIGMA, st)
            synth.dev_fill_matrix(q, dt, (H + Hkv) * hd, 1, Hkv * hd, E, key(synth.WV, l),
                                  WEIGHT_SIGMA, st)
            if s.qkv_bias:
                b = base + d["bqkv"]
                for j, (kind, n) in enumerate(((synth.BQ, H * hd), (synth.BK, Hkv * hd),
                                               (synth.BV, Hkv * hd))):
                    off = (0, H * hd, (H + Hkv) * hd)[j] * 4
                    synth.dev_fill_matrix(b + off, synth.F32, 0, 1, 1, n, key(kind, l), BIAS_SIGMA,
                                          st)
            if s.rope_neox:
                self._interleave_halves(d, H, Hkv, hd, mb(1, E), s.qkv_bias)
            synth.dev_fill_matrix(base + d["wo"], dt, 0, 1, E, H * hd, key(synth.WO, l),
                                  WEIGHT_SIGMA, st)
            if s.expert_count > 0:
                synth.dev_fill_matrix(base + d["w_router"], dt, 0, 1, s.expert_count, E,
                                      key(synth.WROUTER, l), WEIGHT_SIGMA, st)
            for e in range(nsets):
                gu = base + d["w_gate_up"][e]
                synth.dev_fill_matrix(gu, dt, 0, 2, F, E, key(synth.WGATE, l, e), WEIGHT_SIGMA, st)
                synth.dev_fill_matrix(gu, dt, 1, 2, F, E, key(synth.WUP, l, e), WEIGHT_SIGMA, st)
                synth.dev_fill_matrix(base + d["w_down"][e], dt, 0, 1, E, F, key(synth.WDOWN, l, e),
                                      WEIGHT_SIGMA, st)

        cfg = pnb_config(V, E, H, Hkv, L, F, s.n_ctx, s.rope_theta, s.rms_norm_eps,
                         s.sliding_window, s.expert_count, s.expert_used, dt, int(s.rope_neox))
        self.model = Model(
            cfg, tok_embd=base + o_emb, out_norm=base + o_onorm, output=base + o_out,
            attn_norm=[base + d["attn_norm"] for d in lay], wqkv=[base + d["wqkv"] for d in lay],
            wo=[base + d["wo"] for d in lay], ffn_norm=[base + d["ffn_norm"] for d in lay],
            w_router=[base + d["w_router"] for d in lay] if s.expert_count > 0 else None,
            w_gate_up=[base + off for d in lay for off in d["w_gate_up"]],
            w_down=[base + off for d in lay for off in d["w_down"]],
            bqkv=[base + d["bqkv"] for d in lay] if s.qkv_bias else None, keepalive=self.buf)
        self.weight_bytes = ar.size

    def _interleave_halves(self, d, H, Hkv, hd, row_bytes, bias):
        """NeoX models: each head's Wq / Wk rows (and q / k bias entries) in the
        order 0, hd/2, 1, hd/2 + 1, ... - the library's layout for them."""
        import torch

        perm = torch.empty(hd, dtype=torch.long)
        perm[0::2] = torch.arange(hd // 2)
        perm[1::2] = torch.arange(hd // 2) + hd // 2
        perm = perm.to(self.buf.device)
        torch.cuda.synchronize(self.buf.device)   # the fills ran on the generator's stream
        heads = H + Hkv                       # Wq then Wk, one block of hd rows per head
        w = self.buf[d["wqkv"]:d["wqkv"] + heads * hd * row_bytes].view(heads, hd, row_bytes)
        w.copy_(w[:, perm, :].clone())
        if bias:
            b = self.buf[d["bqkv"]:d["bqkv"] + heads * hd * 4].view(torch.float32).view(heads, hd)
            b.copy_(b[:, perm].clone())

    def new_state(self, start_pos: int = 0, slot: int = 0, stream=None):
        """A zeroed state; with start_pos > 0 the cache positions below it (the last
        kv_cap of them) hold generated contents and pos = start_pos."""
        import torch

        state = self.model.new_state()
        if start_pos > 0:
            self.prefill(state, start_pos, slot, stream)
        return state

    def prefill(self, state, start_pos: int, slot: int = 0, stream=None):
        """Generated cache contents for positions below start_pos.  They are in
        the library's layout; for NeoX models that is the interleaved key order,
        which is not the order an oracle cache of the same values uses."""
        import torch

        s = self.shape
        st = (stream or torch.cuda.current_stream()).cuda_stream
        cap, hd, Hkv, es = s.kv_cap, s.head_dim, s.n_kv_head, s.elem_bytes
        lo, hi = kv_prefill_range(s, start_pos)
        block = Hkv * cap * hd * es
        base = state.kv.data_ptr()
        for l in range(s.n_layer):
            for kind, kk in ((0, synth.KCACHE), (1, synth.VCACHE)):
                synth.dev_fill_kv(base + (2 * l + kind) * block, s.kv_dtype, Hkv, cap, hd, lo, hi,
                                  synth.key(self.seed, kk, l, slot), KV_SIGMA, st)
        state.set_pos(start_pos, stream)

    def __getattr__(self, name):
        if name == "model":
            raise AttributeError(name)
        return getattr(self.model, name)
