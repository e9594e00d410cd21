"""The seeded input recipe on the host: shapes, layouts, value distributions,
spike rate and reproducibility (the GPU tests draw the same recipe on the
device)."""
import numpy as np
import pytest
import torch

import synth


def _f(t):
    return t.float().numpy().astype(np.float64)


def test_shapes_layouts_and_dtypes():
    x = synth.make(synth.spec("swiglu_4096", M=64, N=96), with_dy=True)
    assert set(x) == {"gate", "up", "dy"}
    assert all(t.dtype == torch.bfloat16 and tuple(t.shape) == (64, 96) for t in x.values())
    y = synth.make(synth.spec("geglu_nvfp4", M=32, N=128), with_dy=True)
    assert tuple(y["x"].shape) == (32, 256) and tuple(y["dy"].shape) == (32, 128)
    with pytest.raises(KeyError):
        synth.spec("no_such_workload")


def test_reproducible_and_seeded_per_tensor_and_offset():
    sp = synth.spec("swiglu_4096", M=32, N=64)
    a, b = synth.make(sp, with_dy=True), synth.make(sp, with_dy=True)
    assert all(torch.equal(a[k], b[k]) for k in a)
    assert not torch.equal(a["gate"], a["up"]) and not torch.equal(a["up"], a["dy"])
    c = synth.make(sp, with_dy=True, seed_offset=1)
    assert not torch.equal(a["gate"], c["gate"])


def test_value_distributions():
    g = _f(synth.make(synth.spec("swiglu_4096", M=512, N=512))["gate"])
    assert abs(g.mean()) < 0.01 and abs(g.std() - 1.0) < 0.01
    d = _f(synth.make(synth.spec("geglu_8192", M=512, N=512), with_dy=True)["dy"])
    assert abs(d.std() - 0.1) < 0.002                      # dY = 0.1 N(0,1)
    x = _f(synth.make(synth.spec("geglu_nvfp4", M=256, N=512))["x"])
    assert abs(x.std() - 2.0) < 0.02                       # X = 2 N(0,1)


def test_spikes():
    sp = synth.spec("swiglu_131072", M=256)                # 256 x 8192 per tensor
    x = synth.make(sp, with_dy=True)
    for k, t in x.items():
        v = _f(t)
        spikes = np.abs(v) == 60.0
        rate = spikes.mean()
        assert 0.0008 < rate < 0.0012, (k, rate)           # 0.1 % of the elements
        assert (v[spikes] > 0).any() and (v[spikes] < 0).any()
        assert abs(v[~spikes].std() - 1.0) < 0.01
    # each tensor has its own spike pattern
    assert not np.array_equal(_f(x["gate"]) == 60.0, _f(x["up"]) == 60.0)


def test_host_bits_are_the_bf16_patterns():
    t = torch.tensor([1.0, -2.0, 0.0, -0.0], dtype=torch.bfloat16)
    assert synth.to_host_bits(t).tolist() == [0x3F80, 0xC000, 0x0000, 0x8000]
