"""The two checkpoint writers agree: the torch writer that generates the
benchmark's large layers on the device (synth.quantise_pack_torch) produces the
same words and scales as the numpy writer the parity tests use, on the same
float weights. Both are the quantiser + packer (outside the path); this pins
the benchmark's inputs to the rule the tests and the oracle are built on."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("fmt,act_order,dtype,K,N,group", [
    ("awq", False, "bf16", 512, 256, 128),
    ("awq", False, "fp16", 256, 64, 32),
    ("gptq", False, "bf16", 384, 96, 64),
    ("gptq", True, "fp16", 1024, 128, 64),
    ("gptq", True, "bf16", 768, 64, 128),
])
def test_torch_writer_matches_numpy_writer(fmt, act_order, dtype, K, N, group):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng([7, K, N])
    w = rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)
    w[:, 3] = 0.0125           # a constant column: scale 1 in both writers
    gi = synth.act_order_gidx(rng, K, group) if act_order else None
    q, z, s = synth._quantise_minmax(w, group, gi, dtype)
    if fmt == "awq":
        qw, qz = synth._pack_awq(q), synth._pack_awq(z)
    else:
        qw, qz = synth._pack_rows_std(q), synth._pack_cols_std(z)
    tq, tz, ts = synth.quantise_pack_torch(torch.from_numpy(w), group, dtype, fmt,
                                           None if gi is None else torch.from_numpy(gi))
    assert np.array_equal(tq.numpy(), qw)
    assert np.array_equal(tz.numpy(), qz)
    assert np.array_equal(ts.view(torch.int16).numpy().view(np.uint16), s)


def test_torch_layer_is_seeded():
    torch = pytest.importorskip("torch")
    a = synth.make_layer_torch(3, 256, 128, 128, "bf16", device="cpu")
    b = synth.make_layer_torch(3, 256, 128, 128, "bf16", device="cpu")
    c = synth.make_layer_torch(4, 256, 128, 128, "bf16", device="cpu")
    assert all(torch.equal(x, y) for x, y in zip(a[:3], b[:3]))
    assert not torch.equal(a[0], c[0])
    g = synth.make_layer_torch(3, 512, 64, 128, "fp16", fmt="gptq", act_order=True, device="cpu")[3]
    assert np.array_equal(np.bincount(g.numpy(), minlength=4), np.full(4, 128))
