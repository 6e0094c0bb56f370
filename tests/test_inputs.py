"""The seeded input generator (CPU): reproducible, sliceable, and exactly in the target dtype."""
import numpy as np
import torch

import gdr_inputs as gi


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(
        -20, 20, 100000), np.array([0.0, -0.0, 1.0, 65504.0, 1e-38, 3.0e38], np.float32)])
    x = x.astype(np.float32)
    ours = gi.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)
    bits = gi.bf16_bits(ours)
    back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(back, ours)


def test_blocks_reproducible_and_sliceable():
    wl = gi.custom(seqlens=[5, 9, 3], H=3, d_k=16, d_v=8, dtype="bf16", s0="normal")
    full = gi.gen_full(wl, threads=4)
    sub = gi.gen_full(wl, heads=[2], seqs=[1], threads=1)
    cu = full["cu_seqlens"]
    for name in ("q", "k", "v", "alpha", "beta"):
        np.testing.assert_array_equal(sub[name][:, 0], full[name][cu[1]:cu[2], 2])
    np.testing.assert_array_equal(sub["S0"][0, 0], full["S0"][1, 2])
    again = gi.gen_full(wl, threads=2)
    for name in full:
        np.testing.assert_array_equal(full[name], again[name])
    # values are exactly bf16
    for name in ("q", "k", "v"):
        np.testing.assert_array_equal(gi.bf16_round(full[name]), full[name])


def test_distributions():
    wl = gi.custom(seqlens=[4000], H=2, d_k=64, d_v=64, dtype="f32", s0="normal")
    a = gi.gen_full(wl)
    np.testing.assert_allclose(np.linalg.norm(a["k"], axis=-1), 1.0, atol=1e-5)
    np.testing.assert_allclose(np.linalg.norm(a["q"], axis=-1), 1.0, atol=1e-5)
    assert 0 < a["alpha"].min() and a["alpha"].max() < 1
    assert abs(np.mean(-np.log(a["alpha"])) - 0.029) < 0.005
    assert 0 < a["beta"].min() and a["beta"].max() < 1 and abs(a["beta"].mean() - 0.5) < 0.02
    assert abs(a["v"].std() - 1.0) < 0.02 and abs(a["S0"].std() - 0.1) < 0.01


def test_named_workloads():
    wl = gi.workload("varlen_n64_h16")
    assert wl.n_seqs == 64 and wl.seqlens.min() >= 128 and wl.seqlens.max() < 65536
    assert 400_000 < wl.total_tokens < 1_000_000
    assert gi.workload("kda_b1_h32_t32768").total_tokens == 32768
    d = gi.gen_decode_step(gi.workload("decode_n256_h32"), 3)
    assert d["q"].shape == (256, 32, 128) and d["alpha"].shape == (256, 32, 128)


def test_parity_metrics():
    # the element-wise metric sees a single wrong element that the row norm hides, and the
    # fp32 bound asserts it; the bf16 bound keeps the row-normwise metric alone
    from tests.parity import TOL, err_rows, rel_elem, rel_rows
    rng = np.random.default_rng(0)
    ref = rng.normal(size=(8, 128))
    got = ref.copy()
    got[3, 5] += 5e-4 * abs(ref[3, 5]) + 1e-12
    assert rel_rows(got, ref) < 1e-4 < rel_elem(got, ref)
    assert err_rows(got, ref, TOL["f32"]) > TOL["f32"]
    assert err_rows(got, ref, TOL["bf16"]) == rel_rows(got, ref)
    # elements near zero are judged against 1e-3 x the RMS, not their own size
    ref2 = np.ones((2, 4))
    ref2[0, 0] = 0.0
    got2 = ref2.copy()
    got2[0, 0] = 1e-8
    assert rel_elem(got2, ref2) < 1e-4
