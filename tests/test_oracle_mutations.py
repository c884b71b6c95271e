"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch every one of them: a pin set that lets a dropped term, a wrong sign, an
off-by-one or a transposed operand through would not be worth trusting."""
import math

import numpy as np
import pytest

import oracle.draft_attn_oracle as orc
from tests import oracle_pins as pins

# a planted mistake may produce NaN or inf on the way to a failing pin
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rope_sign(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    a = orc.rope_angles(pos, d, theta)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)


def _rope_adjacent_pairs(x, pos, theta):
    # interleaved (x_2i, x_2i+1) pairing instead of rotate-half
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    a = orc.rope_angles(pos, d, theta)
    c, s = np.cos(a), np.sin(a)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xo * c + xe * s
    return out


def _fold_sinks_also_far(mode, L, W=0, n_sink=0):
    # FOLD with sinks, the sinks counted twice: local and far
    sel = _select_keys(mode, L, W, n_sink)
    if mode == "fold":
        sel = dict(sel, far=np.arange(0, max(0, L - W), dtype=np.int64))
    return sel


def _fold_sinks_ignored(mode, L, W=0, n_sink=0):
    return _select_keys(mode, L, W, 0 if mode == "fold" else n_sink)


_select_keys = orc.select_keys
_e4m3_encode = orc.e4m3_encode


def _e4m3_ties_away(x):
    # an exact midpoint goes to the larger magnitude instead of the even code
    codes = _e4m3_encode(x)
    a = np.abs(np.asarray(x, dtype=np.float32).astype(np.float64))
    mag = codes & 0x7F
    v = np.abs(orc.e4m3_decode(mag))
    nxt = np.abs(orc.e4m3_decode(np.minimum(mag + 1, 0x7E)))
    mid = (a > v) & (a - v == nxt - a)
    return np.where(mid, codes + 1, codes).astype(np.uint8)


def _e4m3_subnormals_flushed(x):
    codes = _e4m3_encode(x)
    return np.where((codes & 0x78) == 0, codes & 0x80, codes).astype(np.uint8)


def _e4m3_no_saturation(x):
    codes = _e4m3_encode(x)
    big = np.abs(np.asarray(x, dtype=np.float32)) >= 464
    return np.where(big, codes | 0x7F, codes).astype(np.uint8)   # overflow to NaN


def _side_fp8_unscaled(k_raw, scale):
    return orc.e4m3_decode(orc.side_fp8_codes(k_raw, scale))


def _logits_chunk_positions_restart(q_rot, k_raw, key_pos, theta, chunk):
    # every chunk after the first takes the first chunk's key positions
    n = k_raw.shape[0]
    out = np.empty((n, q_rot.shape[0]), dtype=np.float64)
    key_pos = np.broadcast_to(np.asarray(key_pos, dtype=np.int64), (n,))
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        kr = orc.rope(np.asarray(k_raw[a:b], dtype=np.float64), key_pos[0:b - a], theta)
        out[a:b] = kr @ q_rot.T
    return out


def _logits_chunk_shifted(q_rot, k_raw, key_pos, theta, chunk):
    # the keys of chunk c are written one row late (an off-by-one slice)
    n = k_raw.shape[0]
    out = np.zeros((n, q_rot.shape[0]), dtype=np.float64)
    key_pos = np.broadcast_to(np.asarray(key_pos, dtype=np.int64), (n,))
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        kr = orc.rope(np.asarray(k_raw[a:b], dtype=np.float64), key_pos[a:b], theta)
        lo = a + 1 if a else a
        out[lo:b] = (kr @ q_rot.T)[: b - lo]
    return out


def _weighted_sum_chunk_values_restart(w, v, chunk):
    # every chunk's weights meet the first chunk's values
    o = np.zeros((w.shape[1], v.shape[1]), dtype=np.float64)
    for a in range(0, w.shape[0], chunk):
        b = min(w.shape[0], a + chunk)
        o += w[a:b].T @ np.asarray(v[0:b - a], dtype=np.float64)
    return o


def _append_at_next_position(k_new, pos, theta):
    return orc.rope(np.asarray(k_new, dtype=np.float64),
                    np.asarray(pos, dtype=np.int64)[..., None] + 1, theta)


def _append_pos_wrong_axis(k_new, pos, theta):
    # positions broadcast over the head axis instead of the token axis
    k = np.asarray(k_new, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.int64)
    p = np.resize(pos.reshape(-1), k.shape[:-1])
    return orc.rope(k, p, theta)

MUTATIONS = {
    "rope_sign": ("rope", _rope_sign),
    "rope_pairing": ("rope", _rope_adjacent_pairs),
    "inv_freq_missing_2": ("rope_inv_freq",
                           lambda d, theta: np.power(float(theta), -np.arange(d // 2) / d)),
    "nope_ignored": ("rope_inv_freq",
                     lambda d, theta: np.power(float(theta or 1e4), -2.0 * np.arange(d // 2) / d)),
    "window_off_by_one": ("window_start", lambda L, W: max(0, L - W + 1)),
    "tree_bit_off_by_one": ("tree_filter", lambda pos, L, nt, m: (
        np.asarray(pos, dtype=np.int64) if m is None or nt <= 0 else np.asarray(
            [j for j in pos if j < L - nt or (int(m) >> int(j - (L - nt) + 1)) & 1], dtype=np.int64))),
    "fold_sinks_also_far": ("select_keys", _fold_sinks_also_far),
    "e4m3_ties_away": ("e4m3_encode", _e4m3_ties_away),
    "e4m3_subnormals_flushed": ("e4m3_encode", _e4m3_subnormals_flushed),
    "e4m3_no_saturation": ("e4m3_encode", _e4m3_no_saturation),
    "side_fp8_scale_dropped": ("side_fp8_keys", _side_fp8_unscaled),
    "fold_sinks_ignored": ("select_keys", _fold_sinks_ignored),
    "far_position_off_by_one": ("fold_far_position", lambda L, W: L - W),
    "gamma_no_clamp": ("sharp_gamma", lambda n, b, r: 1.0 + b * math.log(max(n, 1) / r)),
    "gamma_log2": ("sharp_gamma", lambda n, b, r: max(1.0, 1 + b * math.log2(max(n, 1) / r))),
    "softmax_no_normalise": ("_softmax",
                             lambda s: np.exp(s - s.max(axis=0, keepdims=True)) if s.shape[0] else s),
    "weighted_sum_drop_last_chunk": ("_weighted_sum",
                                     lambda w, v, chunk: (w[:-1].T @ np.asarray(v[:-1], dtype=np.float64))),
    "page_slot_transposed": ("page_slot",
                             lambda pos, bt, P=64: (np.asarray(bt)[np.asarray(pos) % P],
                                                    np.asarray(pos) // P,
                                                    np.asarray(bt)[np.asarray(pos) % P] * P + np.asarray(pos) // P)),
    "logits_chunk_positions_restart": ("_logits", _logits_chunk_positions_restart),
    "logits_chunk_off_by_one": ("_logits", _logits_chunk_shifted),
    "weighted_sum_chunk_values_restart": ("_weighted_sum", _weighted_sum_chunk_values_restart),
    "append_at_next_position": ("append_rotated_keys", _append_at_next_position),
    "append_pos_wrong_axis": ("append_rotated_keys", _append_pos_wrong_axis),
}


def _run_all():
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(orc, attr, bad)
    failed = _run_all()
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_unmutated_oracle_passes_all():
    assert _run_all() == []
