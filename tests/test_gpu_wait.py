"""A bounded device wait that runs out, and the state afterwards.

Every spin-wait in the library's kernels is bounded: when one gives up, the
kernel sets PNB_DEV_ERR_TIMEOUT in the state's error word, lets its own copies
land and returns.  pnb_state_wait_probe makes one such wait run out on
purpose (an mbarrier that nothing arrives on, after a real bulk copy), with a
short limit, so the path is exercised without faulting or hanging anything.
The test checks that the error reaches the host through pnb_state_check and
through the begin / poll seam, that a reset clears it, and that the state then
decodes exactly as the oracle does.
"""
import numpy as np
import pytest

import oracle
import synth.workloads as wl
from synth import BF16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transformer_decode_step_gb300 as pnb  # noqa: E402

DEV = torch.device("cuda:0")
SHAPE = wl.Shape(n_vocab=1000, n_embd=512, n_head=8, n_kv_head=2, n_layer=2, n_ff=1024,
                 n_ctx=64, rope_theta=1e4, rms_norm_eps=1e-5, dtype=BF16)
SEED = 41
TOL = 2e-2


def test_bounded_wait_runs_out_and_the_state_recovers():
    sm = pnb.SynthModel(SHAPE, SEED, device=DEV)
    st = sm.new_state()
    assert st.device_error() == 0
    st.wait_probe(200_000)                      # 0.2 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert st.device_error() == pnb.PNB_DEV_ERR_TIMEOUT
    st.reset()
    assert st.device_error() == 0

    # through the begin / poll seam: the probe on the state's own stream, then a step
    st.wait_probe(200_000, stream=st.stream())
    lg = torch.empty(SHAPE.n_vocab, dtype=torch.float32, device=DEV)
    st.forward_begin(3, logits=lg)
    with pytest.raises(pnb.PnbError) as e:
        while not st.poll():
            pass
    assert e.value.code == -8                   # PNB_E_DEVICE
    st.reset()

    # the context and the state are usable: a short decode equals the oracle's
    tokens = [3, 141, 592, 653, 589]
    got, gam = [], []
    for t in tokens:
        st.forward(t, logits=lg)
        got.append(lg.cpu().numpy().copy())
        gam.append(int(np.argmax(got[-1])))
    assert st.device_error() == 0
    om = oracle.Model(SHAPE, seed=SEED)
    os_ = om.new_state()
    for i, t in enumerate(tokens):
        ref, ram = os_.forward(t)
        scale = float(np.max(np.abs(ref)))
        assert float(np.max(np.abs(got[i] - ref))) <= TOL * scale, f"step {i}"
        if gam[i] != ram:
            top = np.sort(ref)[-2:]
            assert float(top[1] - top[0]) <= TOL * scale, f"step {i}: argmax {gam[i]} != {ram}"


def test_wait_probe_rejects_limits_above_one_second():
    sm = pnb.SynthModel(SHAPE, SEED, device=DEV)
    st = sm.new_state()
    with pytest.raises(pnb.PnbError) as e:
        st.wait_probe(2_000_000_000)
    assert e.value.code == -1
