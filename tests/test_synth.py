"""The seeded input generator: determinism, shapes, and bf16 rounding equal to torch's own
float32 -> bfloat16 conversion (round to nearest even)."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = synth.round_bf16(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    bits = synth.bf16_bits(got)
    assert np.array_equal(synth.bits_to_f32(bits), got)
    assert np.array_equal(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy(), got)


def test_requests_are_seeded_and_independent():
    wl = synth.small_workload(1, B=3, N=64, t=63)
    a = synth.gen_request(wl, 1)
    b = synth.gen_requests(wl, requests=[0, 1])[1]
    for k in a:
        assert np.array_equal(a[k], b[k])
    c = synth.gen_request(wl, 2)
    assert not np.array_equal(a["kv"], c["kv"])
    assert a["kv"].shape == (64, 512) and a["q"].shape == (1, 64, 512) and a["w"].shape == (1, 64)
    # bf16 storage: every stored value is bf16-representable
    assert np.array_equal(synth.round_bf16(a["kv"]), a["kv"])
    sh = synth.gen_shared(wl)
    assert sh["bias"].shape == (8, 512) and sh["idx_bias"].shape == (8, 128) and sh["sink"].shape == (64,)


def test_workload_shapes():
    w4 = synth.WORKLOADS[4]
    assert (w4.t + 1) // w4.ratio == 262144 and w4.N - 262144 * 4 == 3
    w3 = synth.WORKLOADS[3]
    assert w3.hca and w3.n_entries == 2048
    assert synth.WORKLOADS[0].storage == "f32"
