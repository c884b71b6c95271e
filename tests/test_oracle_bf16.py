"""The oracle's float64 -> bfloat16 rounding, pinned to hand cases and to
torch's float32 -> bfloat16 conversion (a library routine) on values that are
exact in float32."""
import numpy as np
import torch

import oracle.draft_attn_oracle as orc


def test_hand_cases():
    u = 2.0 ** -7                      # bf16 spacing just above 1
    cases = {
        1.0: 1.0,
        1.0 + u / 2: 1.0,              # tie -> even (1.0)
        1.0 + 3 * u / 2: 1.0 + 2 * u,  # tie -> even (mantissa ...10)
        1.0 + u / 2 + 1e-12: 1.0 + u,  # above the tie
        -(1.0 + 3 * u / 2): -(1.0 + 2 * u),
        0.0: 0.0,
        3.0: 3.0,
        2.0 ** -130: 2.0 ** -130,      # bf16 subnormal, exact
        2.0 ** -134: 0.0,              # half the smallest subnormal: tie -> 0
    }
    for x, want in cases.items():
        assert orc.round_to_bf16(np.array([x]))[0] == want, x


def test_against_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-38).astype(np.float32),
                        (rng.standard_normal(2000) * 1e30).astype(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)
