"""Pins of the seeded input generator (host side; the device side is compared in GPU tests)."""
import os

import numpy as np
import pytest
import torch

import synth
import synth.workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_ints(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(l) for l in f if l.strip() and not l.startswith("#")]


def test_splitmix64_published_sequence():
    # word n of a stream is the (n+1)-th SplitMix64 output of a state seeded with the key
    got = [int(v) for v in synth.words(1234567, 0, 5)]
    assert got == _golden_ints("splitmix64_seed1234567.txt")


def test_irwin_hall_range_and_moments():
    k = synth.key(7, synth.WQ, 3, 0)
    n = synth.ih12(k, 0, 400_000).astype(np.int64)
    assert n.min() >= -393210 and n.max() <= 393210
    z = n / 65536.0
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    # Irwin-Hall(12) kurtosis is 3 - 1.2/12 = 2.9
    kurt = np.mean(z ** 4) / np.mean(z ** 2) ** 2
    assert abs(kurt - 2.9) < 0.05


@pytest.mark.parametrize("sigma", [0.02, 1.0])
def test_values_are_scaled_irwin_hall(sigma):
    k = synth.key(2, synth.WO, 0, 0)
    n = synth.ih12(k, 1000, 5000)
    v = synth.values(k, 1000, 5000, sigma, synth.F32)
    # exact: (float(n) * 2^-16) * sigma, one fp32 rounding
    expect = ((n.astype(np.float32) * np.float32(1 / 65536)) * np.float32(sigma)).astype(np.float32)
    assert np.array_equal(v, expect)
    assert abs(v.std() / sigma - 1.0) < 0.05


def test_bf16_rounding_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200_000).astype(np.float32) * np.float32(0.02)
    # add exact halfway cases: low 16 bits = 0x8000
    bits = x.view(np.uint32)
    half = (bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = np.concatenate([x, half.view(np.float32)])
    ours = np.array([synth.f32_to_bf16_bits(float(v)) for v in x[:2000]] , dtype=np.uint16)
    ref = torch.from_numpy(x[:2000]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    ours_h = np.array([synth.f32_to_bf16_bits(float(v)) for v in x[-2000:]], dtype=np.uint16)
    ref_h = torch.from_numpy(x[-2000:]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours_h, ref_h)


def test_bf16_values_are_rounded_f32_values():
    k = synth.key(3, synth.WGATE, 5, 1)
    f = synth.values(k, 0, 10_000, 0.02, synth.F32)
    b = synth.values(k, 0, 10_000, 0.02, synth.BF16)
    ref = torch.from_numpy(f).to(torch.bfloat16).float().numpy()
    assert np.array_equal(b, ref)
    bits = synth.bf16_bits(k, 0, 10_000, 0.02)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), b)


def test_keys_separate_tensors_and_are_deterministic():
    a = synth.values(synth.key(1, synth.WQ, 0, 0), 0, 64, 1.0, synth.F32)
    assert np.array_equal(a, synth.values(synth.key(1, synth.WQ, 0, 0), 0, 64, 1.0, synth.F32))
    for other in (synth.key(1, synth.WK, 0, 0), synth.key(1, synth.WQ, 1, 0),
                  synth.key(1, synth.WQ, 0, 1), synth.key(2, synth.WQ, 0, 0)):
        b = synth.values(other, 0, 64, 1.0, synth.F32)
        assert not np.array_equal(a, b)
        assert abs(np.corrcoef(a, b)[0, 1]) < 0.5


def test_uniform_int_range():
    k = synth.key(5, synth.POSITIONS, 0, 0)
    v = synth.uniform_int(k, 0, 100_000, 512, 4096 - 512 + 1)
    assert v.min() >= 512 and v.max() <= 4096
    counts = np.bincount(v - 512, minlength=3585)
    chi2 = float(((counts - counts.mean()) ** 2 / counts.mean()).sum())
    dof = counts.size - 1
    assert abs(chi2 - dof) < 6 * (2 * dof) ** 0.5


def test_workload_recipe():
    assert wl.TINY.shape.head_dim == 32
    E, L, F, V = 4096, 32, 11008, 32000
    assert wl.LLAMA7B.shape.params_read_per_token() == E + L * (4 * E * E + 3 * F * E) + V * E
    # Mixtral: 4 attention matrices (GQA: q, o full; k, v a quarter) + router + 2 of 8 experts
    attn = 2 * E * E + 2 * 1024 * E
    assert wl.MIXTRAL.shape.params_read_per_token() == E + 32 * (attn + 8 * E + 2 * 3 * 14336 * E) + V * E
    assert wl.MISTRAL7B.shape.kv_cap == 4096
    assert wl.kv_prefill_range(wl.MISTRAL7B.shape, 8192) == (4096, 8192)
    toks = wl.prompt_tokens(wl.TINY)
    assert len(toks) == 16 and all(0 <= t < 1024 for t in toks)
    pos = wl.slot_positions(wl.LLAMA8B_BATCHED)
    assert len(pos) == 64 and all(512 <= p <= 4096 for p in pos)
