"""The allocation-free attention entry point against the library's own attention.

pnb_attention_decode_static is for callers that may not allocate device
memory (allocation forbidden after start-up, a foreign memory pool that owns
all device memory, or a plugin that only gets input and output buffers): its
scratch is a static device array inside the library.  This test feeds it the
same queries and KV cache as the state-based attention kernel (which uses the
scratch its state allocated) and checks both outputs agree, on two calls in a
row, within the bf16 tolerance the parity tests use.  It is collected last
and also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import synth.workloads as wl
from synth import BF16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

SHAPE = wl.Shape(n_vocab=1000, n_embd=1024, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                 n_ctx=96, rope_theta=1e4, rms_norm_eps=1e-5, sliding_window=48, dtype=BF16)
TOL = 2e-2   # bf16 tolerance of the parity tests, relative to max |value|


def _device_view(ptr: int, n: int):
    """A torch view of n fp32 values at a device pointer owned by the library."""
    class _Holder:
        __cuda_array_interface__ = {"shape": (n,), "typestr": "<f4", "data": (ptr, False),
                                    "version": 3}
    return torch.as_tensor(_Holder(), device="cuda")


def test_static_scratch_attention_matches_state_attention():
    s = SHAPE
    sm = pnb.SynthModel(s, 21, device="cuda")
    sm.model.set_persistent(False)
    st = sm.new_state(start_pos=70)          # ring of 48 slots, already wrapped
    layer = s.n_layer - 1
    cap, hd = s.kv_cap, s.head_dim
    block = s.n_kv_head * cap * hd * s.elem_bytes
    kp = st.kv.data_ptr() + 2 * layer * block
    vp = kp + block
    act = st.activations()
    n = s.n_head * hd
    out = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    for call, pos in enumerate((70, 71)):
        st.set_pos(pos)
        st.run_kernel(pnb.PNB_KERNEL_QKV, layer)    # queries and this position's K / V
        st.run_kernel(pnb.PNB_KERNEL_ATTN, layer)   # existing entry point, state scratch
        ref = _device_view(act["attn"], n).clone()
        pnb.attention_decode_static(act["q"], kp, vp, BF16, s.n_head, s.n_kv_head, hd, cap,
                                    s.sliding_window, pos, out)
        torch.cuda.synchronize()
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        scale = float(np.max(np.abs(want)))
        assert scale > 0 and np.all(np.isfinite(got))
        err = float(np.max(np.abs(got - want)))
        assert err <= TOL * scale, f"call {call}: max|d|={err:.3e} vs {TOL}*{scale:.3e}"
        out.fill_(float("nan"))                  # the next call must write every element
    assert st.device_error() == 0


def test_static_scratch_rejects_oversized_and_unsupported_requests():
    buf = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    # 2 MiB cannot hold the partials of even one split for 8192 heads of 128
    with pytest.raises(pnb.PnbError) as e:
        pnb.attention_decode_static(p, p, p, BF16, 8192, 8192, 128, 64, 0, 3, p)
    assert e.value.code == -11
    with pytest.raises(pnb.PnbError) as e:
        pnb.attention_decode_static(p, p, p, BF16, 8, 2, 96, 64, 0, 3, p)
    assert e.value.code == -5
