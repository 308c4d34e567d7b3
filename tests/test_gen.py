"""The seeded generators: determinism, per-request regeneration, storage rounding."""
import numpy as np
import torch

import gen


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * 10).astype(np.float32)
    ours = gen.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(gen.bf16_bits_to_f32(ours), torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_requests_regenerate_alone_and_are_deterministic():
    full = gen.make_asymspec_batch("spiky", 7, 6, 2, 300, gen.BF16, identical_frac=0.5)
    part = gen.make_asymspec_batch("spiky", 7, 6, 2, 300, gen.BF16, identical_frac=0.5, requests=[4, 1])
    for j, r in enumerate([4, 1]):
        np.testing.assert_array_equal(part.a[j], full.a[r])
        np.testing.assert_array_equal(part.b[j], full.b[r])
        np.testing.assert_array_equal(part.t[j], full.t[r])
        np.testing.assert_array_equal(part.drafts[j], full.drafts[r])
    assert full.identical.sum() == 3
    for r in range(6):
        assert np.array_equal(full.a[r], full.b[r]) == bool(full.identical[r])
    again = gen.make_asymspec_batch("spiky", 7, 6, 2, 300, gen.BF16, identical_frac=0.5)
    np.testing.assert_array_equal(again.t, full.t)


def test_gumbel_zipf_mask_and_drafts():
    b = gen.make_asymspec_batch("gumbel_zipf", 3, 2, 2, 5000, gen.BF16)
    frac = np.mean(b.a != b.b)
    assert 0.15 < frac < 0.25
    for r in range(2):
        for i in range(2):
            assert b.drafts[r, i] == np.argmax(gen.widen(b.a[r, i], gen.BF16))


def test_rapid_batch():
    b = gen.make_rapid_batch(1234, 2, 3, 1000)
    assert b.z.dtype == np.float32 and b.q.dtype == np.float32
    np.testing.assert_allclose(b.q.astype(np.float64).sum(-1), 1.0, atol=1e-5)
    assert np.all((b.drafts >= 0) & (b.drafts < 1000))


def test_parallel_generation_matches_serial():
    s = gen.make_asymspec_batch("gumbel_zipf", 9, 10, 1, 200, gen.BF16)
    p = gen.make_asymspec_batch("gumbel_zipf", 9, 10, 1, 200, gen.BF16, processes=2)
    np.testing.assert_array_equal(s.t, p.t)
    np.testing.assert_array_equal(s.drafts, p.drafts)
