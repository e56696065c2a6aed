"""The allocation-free attention entry point, against the oracle and the library.

pnb_attention_decode_static is for callers that may not allocate device
memory: code where allocation is forbidden once it has started, a framework
whose own pool owns all device memory, or a plugin that is only handed input
and output buffers.  Its scratch is a static device array inside the library.

On each shape, two calls in a row (positions p and p + 1, the cache appended
between them by the library's own QKV kernel) are checked:

* against the oracle's attention on the same rotated queries and cache
  contents (read back from the device);
* against the state-based attention kernel, which uses the scratch its state
  allocated (1e-5 of max |value|: the same arithmetic, possibly another split
  of the positions);
* its error output reads 0, and device free memory is the same before and
  after the second call.

The file is collected last, and also passes on its own in a fresh process.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth.workloads as wl
from synth import BF16, F32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

BASE = wl.Shape(n_vocab=1000, n_embd=1024, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                n_ctx=96, rope_theta=1e4, rms_norm_eps=1e-5, sliding_window=48, dtype=BF16)
CASES = {
    # bf16, head_dim 128, GQA 4, a 48-slot window ring that has wrapped
    "bf16_hd128_ring": (BASE, 70),
    # fp32, head_dim 32, GQA 2, no window, position below the capacity
    "f32_hd32": (dataclasses.replace(BASE, n_embd=256, n_head=8, n_kv_head=4, sliding_window=0,
                                     dtype=F32), 40),
    # bf16, head_dim 64, MHA, no window
    "bf16_hd64_mha": (dataclasses.replace(BASE, n_embd=512, n_head=8, n_kv_head=8,
                                          sliding_window=0, n_ctx=200), 150),
}
TOL_SAME_KERNEL = 1e-5   # relative to max |value|
TOL_ORACLE = 1e-4        # fp32 kernel arithmetic against the oracle's fp64 sums


def _device_view(ptr: int, n: int):
    """A torch view of n fp32 values at a device pointer owned by the library."""
    class _Holder:
        __cuda_array_interface__ = {"shape": (n,), "typestr": "<f4", "data": (ptr, False),
                                    "version": 3}
    return torch.as_tensor(_Holder(), device="cuda")


def _oracle_attention(s, q, kblk, vblk, pos):
    """The oracle's attention over the cache block's slots, laid out linearly."""
    cap, window = s.kv_cap, s.sliding_window
    K = np.zeros((pos + 1, s.n_kv_head, s.head_dim), dtype=np.float32)
    V = np.zeros_like(K)
    lo = max(0, pos - window + 1) if window > 0 else 0
    for j in range(lo, pos + 1):
        K[j] = kblk[:, j % cap, :]
        V[j] = vblk[:, j % cap, :]
    return oracle.attention(q, K, V, s.n_head, s.n_kv_head, pos, window)


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_attention_matches_oracle_and_state_attention(name):
    s, p0 = CASES[name]
    sm = pnb.SynthModel(s, 21, device="cuda")
    sm.model.set_tensor_attention(False)      # the state path runs the same CUDA-core kernel
    st = sm.new_state(start_pos=p0)
    layer = s.n_layer - 1
    cap, hd = s.kv_cap, s.head_dim
    block = s.n_kv_head * cap * hd * s.elem_bytes
    kp = st.kv.data_ptr() + 2 * layer * block
    vp = kp + block
    act = st.activations()
    n = s.n_head * hd
    out = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    et = torch.bfloat16 if s.dtype == BF16 else torch.float32
    for call, pos in enumerate((p0, p0 + 1)):
        st.set_pos(pos)
        st.run_kernel(pnb.PNB_KERNEL_QKV, layer)    # queries and this position's K / V
        st.run_kernel(pnb.PNB_KERNEL_ATTN, layer)   # existing entry point, state scratch
        ref = _device_view(act["attn"], n).clone()
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        pnb.attention_decode_static(act["q"], kp, vp, s.dtype,
                                    s.n_head, s.n_kv_head, hd, cap, s.sliding_window, pos, out,
                                    err=err)
        torch.cuda.synchronize()
        if call == 1:   # after the first call's one-time set-up: nothing is allocated
            assert torch.cuda.mem_get_info()[0] == free0
        assert int(err.item()) == 0
        got, same = out.cpu().numpy(), ref.cpu().numpy()
        scale = float(np.max(np.abs(same)))
        assert scale > 0 and np.all(np.isfinite(got))
        d = float(np.max(np.abs(got - same)))
        assert d <= TOL_SAME_KERNEL * scale, f"call {call}: vs state kernel {d:.3e} / {scale:.3e}"
        q = _device_view(act["q"], n).cpu().numpy()
        kv = torch.as_tensor(st.kv).view(torch.uint8)
        kblk = kv[2 * layer * block:(2 * layer + 1) * block].view(et).float().cpu().numpy()
        vblk = kv[(2 * layer + 1) * block:(2 * layer + 2) * block].view(et).float().cpu().numpy()
        want = _oracle_attention(s, q, kblk.reshape(s.n_kv_head, cap, hd),
                                 vblk.reshape(s.n_kv_head, cap, hd), pos)
        d = float(np.max(np.abs(got - want)))
        assert d <= TOL_ORACLE * float(np.max(np.abs(want))), f"call {call}: vs oracle {d:.3e}"
        out.fill_(float("nan"))                  # the next call must write every element
        err.fill_(-1)
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
    with pytest.raises(pnb.PnbError) as e:   # the error word must be int32-aligned
        pnb.attention_decode_static(p, p, p, BF16, 8, 2, 128, 64, 0, 3, p, err=p + 2)
    assert e.value.code == -3
