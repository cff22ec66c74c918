"""Pins of the oracle's YaRN rotary embedding (CPU only).

"SnapKitty Transformer 8B" names YaRN-scaled rotary embeddings with a 32x
factor for 204800-token sequences; the definition comes from the YaRN paper
(Peng et al. 2023, section 3: NTK-by-parts interpolation and the attention
temperature) on RoFormer's rotary embedding.  Nothing on the pages prints a
value, so the oracle is pinned by what the mathematics fixes: the factor-1
case is plain RoPE, the ramp's closed form where alpha = 1 and beta = s, the
ramp's two ends, hand-computed rotations, norm preservation, and scores that
depend only on the distance between positions.  Planted mistakes in the
oracle's YaRN code are each caught by one of these pins.
"""
import math

import numpy as np
import pytest

import oracle
from causal_grouped_query_gqa_b300.inputs import make_inputs


def test_factor_one_is_plain_rope():
    """s = 1: h_i = theta_i = base^(-2i/d) whatever the ramp, and no temperature."""
    d, base = 64, 10000.0
    f = oracle.yarn_freqs(d, base, 1.0, 6400, 1.0, 32.0)
    theta = np.array([base ** (-2.0 * i / d) for i in range(d // 2)])
    np.testing.assert_allclose(f, theta, rtol=1e-15)
    assert oracle.yarn_mscale(1.0) == 1.0


def test_ramp_closed_form_when_alpha_one_beta_s():
    """With alpha = 1 and beta = s, inside the ramp gamma = (r - 1) / (s - 1), so
    h = theta ((1 - gamma) / s + gamma) = theta r / s = L theta^2 / (2 pi s).  d = 4, base 10^4:
    pair 0 has theta = 1, r = 6400 / (2 pi) = 1018.6 > 32, so h_0 = 1; pair 1 has
    theta = 0.01, r = 64 / (2 pi) = 10.19 (inside the ramp), so
    h_1 = 6400 * 1e-4 / (64 pi) = 0.01 / pi."""
    f = oracle.yarn_freqs(4, 10000.0, 32.0, 6400, 1.0, 32.0)
    assert f[0] == 1.0
    assert abs(f[1] - 0.01 / math.pi) < 1e-17


def test_ramp_ends():
    """r < alpha: full interpolation, h = theta / s; r > beta: none, h = theta.
    d = 64, base 10^4, L = 6400: pair 31 has r = 6400 * 10^(-62/16) / (2 pi) =
    0.14 < 1; pair 0 has r = 1018.6 > 32."""
    d, base, s, L = 64, 10000.0, 32.0, 6400
    f = oracle.yarn_freqs(d, base, s, L, 1.0, 32.0)
    theta31 = base ** (-62.0 / 64.0)
    assert L * theta31 / (2 * math.pi) < 1.0
    assert abs(f[31] - theta31 / s) <= 1e-18
    assert f[0] == 1.0
    # in between the frequencies fall strictly with the pair index
    assert np.all(np.diff(f) < 0)


def test_temperature_of_the_paper():
    """sqrt(1/t) = 0.1 ln s + 1: 1.3466 at s = 32 (ln 32 = 5 ln 2 = 3.4657)."""
    assert abs(oracle.yarn_mscale(32.0) - (0.1 * 5 * 0.6931471805599453 + 1.0)) < 1e-15


def test_rotation_hand_values():
    """A unit vector in pair 0 at position m turns to (cos m h_0, sin m h_0), the
    other pairs untouched; position 0 is the identity."""
    f = np.array([1.0, 0.5])
    x = np.zeros((4, 4))
    x[:, 0] = 1.0
    x[:, 3] = 2.0
    out = oracle.rope_rotate(x[None], f)[0]
    # m = 3, pair 0: cos 3 = -0.98999249660, sin 3 = 0.14112000806
    np.testing.assert_allclose(out[3, :2], [-0.98999249660, 0.14112000806], atol=1e-11)
    # m = 2, pair 1 (h = 0.5): (0, 2) turns to (-2 sin 1, 2 cos 1) = (-1.68294196962, 1.08060461174)
    np.testing.assert_allclose(out[2, 2:], [-1.68294196962, 1.08060461174], atol=1e-11)
    np.testing.assert_array_equal(out[0], x[0])


def test_rotation_preserves_pair_norms():
    f = oracle.yarn_freqs()
    x = np.random.default_rng(0).standard_normal((3, 50, 64))
    y = oracle.rope_rotate(x, f)
    nx = np.hypot(x[..., 0::2], x[..., 1::2])
    ny = np.hypot(y[..., 0::2], y[..., 1::2])
    np.testing.assert_allclose(ny, nx, rtol=1e-13)


def test_scores_depend_on_distance_only():
    """rot(q, m) . rot(k, n) == rot(q, m + c) . rot(k, n + c)."""
    f = oracle.yarn_freqs()
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n, c in [(7, 3, 100), (5000, 4990, 123456), (0, 0, 204799)]:
        a = oracle.rope_rotate(q[None, None], f, positions=[m])[0, 0] @ \
            oracle.rope_rotate(k[None, None], f, positions=[n])[0, 0]
        b = oracle.rope_rotate(q[None, None], f, positions=[m + c])[0, 0] @ \
            oracle.rope_rotate(k[None, None], f, positions=[n + c])[0, 0]
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_yarn_attention_keeps_t1_and_row_sums():
    """Causal attention over rotated q, k still returns out[0] = V[0] (test T1),
    and its LSE is that of the tempered scores of the rotated inputs."""
    q, k, v = (t.double().numpy() for t in make_inputs(1, 2, 1, 40, seed=3))
    o, lse = oracle.attn_fwd_yarn(q, k, v, rounded=False)
    np.testing.assert_allclose(o[0, :, 0], np.repeat(v[0, :1, 0], 2, axis=0), atol=1e-12)
    f = oracle.yarn_freqs()
    t = oracle.yarn_mscale(32.0) ** 2 / 8.0
    qr, kr = oracle.rope_rotate(q, f), oracle.rope_rotate(k, f)
    i = 17
    s = t * (qr[0, 1, i] @ kr[0, 0, :i + 1].T)
    assert abs(lse[0, 1, i] - (s.max() + math.log(np.exp(s - s.max()).sum()))) < 1e-12


def test_round_bf16_ties_and_library_cast():
    """Ties go to the even neighbour: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6,
    -(1 + 2^-8) -> -1; exact bf16 values, zeros and infinities are unchanged; and
    on random values the result equals torch's float32 -> bfloat16 cast."""
    import torch
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1.5, 0.0, -0.0, np.inf, 2 ** -130])
    y = oracle.round_bf16(x)
    assert list(y[:6]) == [1.0, 1 + 2 ** -6, -1.0, 1.5, 0.0, 0.0]
    assert y[6] == np.inf
    r = np.random.default_rng(5).standard_normal(10000) * 37.0
    ref = torch.from_numpy(r.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(r.astype(np.float32).astype(np.float64)), ref)


YARN_MUTANTS = {
    "sin_sign": ("out[r * d + 2 * i] = x0 * c - x1 * s;", "out[r * d + 2 * i] = x0 * c + x1 * s;"),
    "ramp_reversed": ("freq[i] = (1.0 - gamma) * theta / factor + gamma * theta;",
                      "freq[i] = gamma * theta / factor + (1.0 - gamma) * theta;"),
    "half_dim_exponent": ("double theta = pow(base, -2.0 * i / d);",
                          "double theta = pow(base, -1.0 * i / d);"),
    "wavelength_not_2pi": ("double wavelength = 2.0 * acos(-1.0) / theta;",
                           "double wavelength = 1.0 / theta;"),
    "temperature_log2": ("return 0.1 * log(factor) + 1.0;", "return 0.1 * log2(factor) + 1.0;"),
    "round_half_up": ("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "round_truncates": ("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0u;"),
}


@pytest.mark.parametrize("name", sorted(YARN_MUTANTS))
def test_planted_yarn_mistake_is_caught(name, tmp_path):
    import os
    old, new = YARN_MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(c_path), out=str(tmp_path / f"lib{name}.so")))
    saved = oracle._lib
    oracle._lib = lib
    failures = 0
    try:
        for pin in (test_factor_one_is_plain_rope, test_ramp_closed_form_when_alpha_one_beta_s,
                    test_ramp_ends, test_temperature_of_the_paper, test_rotation_hand_values,
                    test_rotation_preserves_pair_norms, test_scores_depend_on_distance_only,
                    test_round_bf16_ties_and_library_cast):
            try:
                pin()
            except AssertionError:
                failures += 1
    finally:
        oracle._lib = saved
    assert failures > 0, f"no pin caught the planted mistake {name}"
