"""Pins for the float64 oracle: checks against facts that do not come from the
oracle itself (an independent complex-number formulation of RoPE, pure-Python
brute force over tiny inputs, closed forms and invariants the pages fix).

Each check takes the oracle module, so the mutation tests can run the same
checks against an oracle with a planted mistake and see at least one fail.
"""
from __future__ import annotations

import cmath
import math

import numpy as np

# --------------------------------------------------------------------------
# Independent pure-Python formulations (no numpy, no oracle code)
# --------------------------------------------------------------------------


def bf_rope(x, pos, theta):
    """RoPE as complex multiplication: z_i = x_i + i x_{i+d/2} times
    exp(i * pos * theta^(-2i/d)) (RoFormer's complex form, rotate-half pairing)."""
    d = len(x)
    h = d // 2
    out = [0.0] * d
    for i in range(h):
        z = complex(x[i], x[i + h]) * cmath.exp(1j * pos * theta ** (-2.0 * i / d))
        out[i], out[i + h] = z.real, z.imag
    return out


def bf_member(mode, j, L, W, n_sink):
    """Which segment key j belongs to, by the plain definitions: None, 'loc' or
    'far'."""
    if not 0 <= j < L:
        return None
    if mode in ("full", "sharp"):
        return "loc"
    if mode == "window":
        return "loc" if (j < n_sink or j >= L - W) else None
    # fold: the window and the sinks are local, every other older key is far
    return "loc" if (j >= L - W or j < n_sink) else "far"


def bf_e4m3(x):
    """Nearest E4M3 value of a Python float by its binade: spacing 2^(E-3) in
    [2^E, 2^(E+1)), E >= -6 (2^-9 in the subnormal range), Python's round()
    (half to even on the multiple of the spacing, which is the code's last
    mantissa bit), magnitudes saturating at 448."""
    sign = math.copysign(1.0, x)
    a = min(abs(x), 448.0)
    if a == 0.0:
        return sign * 0.0
    _, e = math.frexp(a)                 # a in [2^(e-1), 2^e)
    spacing = 2.0 ** (max(e - 1, -6) - 3)
    return sign * min(round(a / spacing) * spacing, 448.0)


def bf_side_fp8(k, s):
    """Far key as an FP8 side cache with scale s returns it."""
    return [bf_e4m3(float(np.float32(x) / np.float32(s))) * float(np.float32(s)) for x in k]


def bf_attend_row(mode, q, p, K, V, L, W=0, n_sink=0, alpha=1.0, lam=0.0,
                  beta=0.0, n_ref=4096, theta=1e4, n_tree=0, tree_mask=None, far_key=None):
    """One query row by brute force: per-key loops, math.exp, Python floats.
    far_key optionally maps a raw key to the key the far memory sees."""
    d = len(q)
    c = 1.0 / math.sqrt(d)
    qr = bf_rope(q, p, theta)
    segs = {"loc": [], "far": []}
    for j in range(L):
        m = bf_member(mode, j, L, W, n_sink)
        # a draft-tree key counts only if the query's mask bit for it is set
        if m is not None and tree_mask is not None and j >= L - n_tree:
            if not (tree_mask >> (j - (L - n_tree))) & 1:
                m = None
        if m is not None:
            segs[m].append(j)
    gamma = 1.0
    if mode == "sharp" and segs["loc"]:
        gamma = max(1.0, 1.0 + beta * math.log(len(segs["loc"]) / n_ref))

    def seg_out(js, key_pos, mult, kmap=None):
        if not js:
            return [0.0] * d, []
        logits = []
        for j in js:
            kr = bf_rope(kmap(K[j]) if kmap else K[j], key_pos(j), theta)
            logits.append(mult * c * sum(a * b for a, b in zip(qr, kr)))
        mx = max(logits)
        e = [math.exp(s - mx) for s in logits]
        z = sum(e)
        w = [x / z for x in e]
        o = [sum(w[n] * V[j][i] for n, j in enumerate(js)) for i in range(d)]
        return o, w

    o_loc, w_loc = seg_out(segs["loc"], lambda j: j, gamma)
    if mode != "fold":
        return o_loc, w_loc, []
    pf = L - W - 1
    o_far, w_far = seg_out(segs["far"], lambda j: pf, alpha, far_key)
    lam_eff = lam if segs["far"] else 0.0
    o = [(1 - lam_eff) * a + lam_eff * b for a, b in zip(o_loc, o_far)]
    return o, [(1 - lam_eff) * w for w in w_loc], [lam_eff * w for w in w_far]


# --------------------------------------------------------------------------
# Checks (raise AssertionError on failure)
# --------------------------------------------------------------------------


def check_rope_complex(orc):
    rng = np.random.default_rng(11)
    for d, theta in ((8, 1e4), (16, 1e6), (64, 1e4)):
        for pos in (0, 1, 7, 4096, 131075, 1048581):
            x = rng.standard_normal(d)
            got = orc.rope(x, pos, theta)
            want = np.array(bf_rope(list(x), pos, theta))
            assert np.max(np.abs(got - want)) < 1e-9, (d, theta, pos)


def check_rope_d2(orc):
    # d = 2: a single pair with inv_freq 1, i.e. a plane rotation by pos radians.
    for pos in (0, 1, 2, 3, 100):
        x = np.array([0.3, -1.7])
        a = float(pos)
        want = np.array([0.3 * math.cos(a) + 1.7 * math.sin(a),
                         -1.7 * math.cos(a) + 0.3 * math.sin(a)])
        assert np.allclose(orc.rope(x, pos, 1e4), want, atol=1e-14)


def check_inv_freq(orc):
    assert np.allclose(orc.rope_inv_freq(4, 1e4), [1.0, 0.01], rtol=1e-15)
    assert np.allclose(orc.rope_inv_freq(8, 1e4), [1.0, 0.1, 0.01, 0.001], rtol=1e-14)
    assert np.allclose(orc.rope_inv_freq(4, 1e6), [1.0, 1e-3], rtol=1e-14)


def check_selection(orc):
    cases = [(0, 4, 2), (1, 4, 2), (5, 4, 0), (10, 4, 2), (10, 8, 2), (10, 10, 3),
             (10, 12, 0), (64, 16, 4), (65, 64, 4), (200, 63, 5), (7, 3, 10)]
    for L, W, ns in cases:
        for mode in ("full", "window", "fold", "sharp"):
            sel = orc.select_keys(mode, L, W, ns if mode in ("window", "fold") else 0)
            want_loc = [j for j in range(L)
                        if bf_member(mode, j, L, W, ns) == "loc"]
            want_far = [j for j in range(L)
                        if bf_member(mode, j, L, W, ns) == "far"]
            assert list(sel["loc"]) == want_loc, (mode, L, W, ns)
            assert list(sel["far"]) == want_far, (mode, L, W, ns)


def check_brute_force(orc):
    rng = np.random.default_rng(5)
    d = 8
    configs = [
        dict(mode="full", L=37), dict(mode="full", L=1),
        dict(mode="window", L=50, W=16, n_sink=3), dict(mode="window", L=20, W=32, n_sink=4),
        dict(mode="window", L=40, W=10, n_sink=0),
        dict(mode="fold", L=45, W=12, alpha=2.0, lam=0.5),
        dict(mode="fold", L=30, W=7, alpha=0.7, lam=0.25),
        dict(mode="fold", L=9, W=12, alpha=2.0, lam=0.5),
        dict(mode="fold", L=45, W=12, n_sink=4, alpha=2.0, lam=0.5),
        dict(mode="fold", L=15, W=12, n_sink=4, alpha=1.5, lam=0.5),
        dict(mode="fold", L=45, W=12, alpha=2.0, lam=0.5, fp8=0.05),
        dict(mode="fold", L=40, W=9, n_sink=3, alpha=2.0, lam=0.5, fp8=0.004),
        dict(mode="sharp", L=60, beta=0.4, n_ref=8),
        dict(mode="sharp", L=5, beta=0.4, n_ref=8),
    ]
    for cfg in configs:
        L = cfg["L"]
        K = rng.standard_normal((L, d))
        V = rng.standard_normal((L, d))
        q = rng.standard_normal(d)
        p = L + int(rng.integers(0, 3))
        prm = orc.Params(mode=cfg["mode"], window=cfg.get("W", 0), n_sink=cfg.get("n_sink", 0),
                         alpha=cfg.get("alpha", 1.0), far_mix=cfg.get("lam", 0.0),
                         scale_slope=cfg.get("beta", 0.0), scale_ref=cfg.get("n_ref", 4096),
                         rope_theta=1e4, side_fp8_scale=cfg.get("fp8", 0.0))
        got = orc.attend_group(q[None], p, K, V, L, prm)[0]
        s8 = cfg.get("fp8", 0.0)
        want, _, _ = bf_attend_row(cfg["mode"], list(q), p, K.tolist(), V.tolist(), L,
                                   W=cfg.get("W", 0), n_sink=cfg.get("n_sink", 0),
                                   alpha=cfg.get("alpha", 1.0), lam=cfg.get("lam", 0.0),
                                   beta=cfg.get("beta", 0.0), n_ref=cfg.get("n_ref", 4096),
                                   far_key=(lambda k: bf_side_fp8(k, s8)) if s8 else None)
        assert np.max(np.abs(got - np.array(want))) < 1e-12, cfg


def check_closed_forms(orc):
    rng = np.random.default_rng(9)
    d = 16
    K = rng.standard_normal((40, d))
    V = rng.standard_normal((40, d))
    # one visible key -> its value
    for mode in ("full", "window", "sharp", "fold"):
        prm = orc.Params(mode=mode, window=4, n_sink=0, alpha=2.0, far_mix=0.5)
        o = orc.attend_group(rng.standard_normal(d)[None], 3, K, V, 1, prm)[0]
        assert np.allclose(o, V[0], atol=1e-14), mode
    # zero query: every logit equal -> mean of the selected values
    q0 = np.zeros((1, d))
    assert np.allclose(orc.attend_group(q0, 40, K, V, 40, orc.Params("full"))[0],
                       V.mean(0), atol=1e-13)
    prm = orc.Params("window", window=10, n_sink=3)
    idx = list(range(3)) + list(range(30, 40))
    assert np.allclose(orc.attend_group(q0, 40, K, V, 40, prm)[0], V[idx].mean(0), atol=1e-13)
    prm = orc.Params("fold", window=10, alpha=3.0, far_mix=0.3)
    want = 0.7 * V[30:40].mean(0) + 0.3 * V[:30].mean(0)
    assert np.allclose(orc.attend_group(q0, 40, K, V, 40, prm)[0], want, atol=1e-13)
    # two keys: weights are a logistic function of the logit difference.
    Kt = np.zeros((2, d)); Vt = np.zeros((2, d))
    Kt[0, 0] = 1.0; Kt[1, 1] = 1.0       # at positions 0 and 1, theta large -> d/2.. dims
    Vt[0, 2] = 1.0; Vt[1, 3] = 1.0
    q = np.zeros(d); q[0] = 2.0
    # with p = 0 and theta huge, only pair 0 rotates (by j radians); key 0 is at 0.
    prm = orc.Params("full", rope_theta=1e30)
    o = orc.attend_group(q[None], 0, Kt, Vt, 2, prm)[0]
    c = 1.0 / math.sqrt(d)
    s0 = c * 2.0 * 1.0                      # <q, k0> with no rotation
    s1 = c * 2.0 * 0.0                      # k1 = e_1 stays e_1 (pair 1 angle ~ 0)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert abs(o[2] - w0) < 1e-12 and abs(o[3] - (1 - w0)) < 1e-12
    # a dominant key: q aligned with one rotated key and scaled up -> its value
    p = 40
    j = 17
    kr = orc.rope(K[j], j, 1e4)
    qd = orc.rope(kr * 200.0, -p, 1e4)      # un-rotate so that RoPE(q, p) = 200 kr
    o = orc.attend_group(qd[None], p, K, V, 40, orc.Params("full"))[0]
    assert np.allclose(o, V[j], atol=1e-6)


def check_weights_sum(orc):
    rng = np.random.default_rng(3)
    d = 8
    K = rng.standard_normal((300, d)) * 3
    V = rng.standard_normal((300, d))
    for prm in (orc.Params("full"), orc.Params("window", window=40, n_sink=4),
                orc.Params("fold", window=50, alpha=2.0, far_mix=0.5),
                orc.Params("sharp", scale_slope=0.05, scale_ref=16)):
        o, w = orc.attend_group(rng.standard_normal((3, d)), 300, K, V, 300, prm,
                                return_weights=True)
        total = sum(ww.sum(axis=0) for _, ww in w.values())
        assert np.allclose(total, 1.0, atol=1e-12), prm.mode
        for _, ww in w.values():
            assert (ww >= 0).all()
        # o must be the weight-average of the values
        o2 = sum(ww.T @ V[idx] for idx, ww in w.values())
        assert np.allclose(o, o2, atol=1e-12)


def check_mode_equivalences(orc):
    rng = np.random.default_rng(4)
    d = 16
    L = 90
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal((4, d))
    full = orc.attend_group(q, L, K, V, L, orc.Params("full"))
    # window with W >= L is full attention (with or without sinks)
    for W, ns in ((L, 0), (L + 5, 3), (L - 2, 4)):
        o = orc.attend_group(q, L, K, V, L, orc.Params("window", window=W, n_sink=ns))
        assert np.allclose(o, full, atol=1e-13), (W, ns)
    # fold with an empty far memory (L <= W) is window attention without sinks
    for W in (L, L + 1, 200):
        o = orc.attend_group(q, L, K, V, L, orc.Params("fold", window=W, alpha=3.0, far_mix=0.5))
        w = orc.attend_group(q, L, K, V, L, orc.Params("window", window=W, n_sink=0))
        assert np.allclose(o, w, atol=1e-13)
    # fold with lambda = 0 is window attention over the last W keys (and the
    # same sinks); with sinks and an empty far memory it is that window too
    for ns in (0, 4):
        o = orc.attend_group(q, L, K, V, L,
                             orc.Params("fold", window=30, n_sink=ns, alpha=3.0, far_mix=0.0))
        w = orc.attend_group(q, L, K, V, L, orc.Params("window", window=30, n_sink=ns))
        assert np.allclose(o, w, atol=1e-13), ns
    o = orc.attend_group(q, L, K, V, L, orc.Params("fold", window=L - 4, n_sink=4, alpha=3.0,
                                                   far_mix=0.7))
    w = orc.attend_group(q, L, K, V, L, orc.Params("window", window=L - 4, n_sink=4))
    assert np.allclose(o, w, atol=1e-13)
    # sharp with slope 0, or with |S| <= N_ref (clamp), is plain attention
    o = orc.attend_group(q, L, K, V, L, orc.Params("sharp", scale_slope=0.0, scale_ref=4))
    assert np.allclose(o, full, atol=1e-13)
    o = orc.attend_group(q, L, K, V, L, orc.Params("sharp", scale_slope=0.3, scale_ref=L))
    assert np.allclose(o, full, atol=1e-13)
    # sharp equals full attention of the query scaled by gamma (closed form)
    beta, nref = 0.3, 10
    gamma = 1.0 + beta * math.log(L / nref)
    o = orc.attend_group(q, L, K, V, L, orc.Params("sharp", scale_slope=beta, scale_ref=nref))
    assert np.allclose(o, orc.attend_group(gamma * q, L, K, V, L, orc.Params("full")),
                       atol=1e-13)
    assert abs(orc.sharp_gamma(int(round(nref * math.e ** 2)), beta, nref)
               - (1 + beta * math.log(round(nref * math.e ** 2) / nref))) < 1e-15


def check_fold_shared_position(orc):
    """Far logits use keys rotated at P_far = L-W-1.  Pinned through the
    relative-position identity <R(p)q, R(P)k> = <R(p-P)q, k> (RoPE's rotation
    matrices compose), computed here from the complex form."""
    rng = np.random.default_rng(8)
    d, L, W, alpha = 8, 40, 12, 2.5
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    p = L
    pf = L - W - 1
    # far-only output: lambda = 1
    o = orc.attend_group(q[None], p, K, V, L, orc.Params("fold", window=W, alpha=alpha, far_mix=1.0))[0]
    qd = bf_rope(list(q), p - pf, 1e4)
    c = 1.0 / math.sqrt(d)
    logits = [alpha * c * sum(a * b for a, b in zip(qd, K[j])) for j in range(L - W)]
    mx = max(logits)
    e = [math.exp(s - mx) for s in logits]
    want = sum(e[j] * V[j] for j in range(L - W)) / sum(e)
    assert np.allclose(o, want, atol=1e-12)
    sl = orc.selection_list("fold", L, p, orc.Params("fold", window=W))
    far = sl["segment"] == orc.SEG_FAR
    assert (sl["key_rope_pos"][far] == pf).all()
    assert (sl["q_rope_pos"][far] == p - pf).all()
    assert (sl["key_rope_pos"][~far] == sl["position"][~far]).all()
    assert (sl["q_rope_pos"][~far] == p).all()


def check_gqa(orc):
    rng = np.random.default_rng(12)
    B, n_q, H_q, H_kv, d, L = 1, 2, 6, 3, 8, 20
    q = rng.standard_normal((B, n_q, H_q, d))
    K = rng.standard_normal((L, H_kv, d))
    V = rng.standard_normal((L, H_kv, d))
    prm = orc.Params("full")
    out = orc.attend(q, [[L, L + 1]], [K], [V], [L], prm)
    for t in range(n_q):
        for h in range(H_q):
            g = h // (H_q // H_kv)
            o = orc.attend_group(q[0, t, h][None], L + t, K[:, g], V[:, g], L, prm)[0]
            assert np.allclose(out[0, t, h], o, atol=1e-14), (t, h)


def check_page_slot(orc):
    bt = [5, 2, 7, 0]
    P = 4
    pos = np.arange(16)
    phys, slot, flat = orc.page_slot(pos, bt, P)
    for j in range(16):
        assert phys[j] == bt[j // P] and slot[j] == j % P and flat[j] == bt[j // P] * P + j % P


def check_tree_masks(orc):
    """Draft-tree masks: brute force per key, every mode; an all-ones mask is
    no mask; a mask hiding every tree key is attention over the cache part."""
    rng = np.random.default_rng(17)
    d, L, nt = 8, 50, 6
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    for mode, kw, bkw in (("full", {}, {}), ("window", dict(window=12, n_sink=2), dict(W=12, n_sink=2)),
                          ("fold", dict(window=10, alpha=2.0, far_mix=0.3),
                           dict(W=10, alpha=2.0, lam=0.3)),
                          ("fold", dict(window=10, n_sink=3, alpha=2.0, far_mix=0.3),
                           dict(W=10, n_sink=3, alpha=2.0, lam=0.3)),
                          ("sharp", dict(scale_slope=0.4, scale_ref=8), dict(beta=0.4, n_ref=8))):
        for mask in (0b101001, 0b1, 0b111111, 0):
            prm = orc.Params(mode=mode, n_tree=nt, rope_theta=1e4, **kw)
            got = orc.attend_group(q[None], L + 1, K, V, L, prm, tree_mask=mask)[0]
            want, _, _ = bf_attend_row(mode, list(q), L + 1, K.tolist(), V.tolist(), L,
                                       n_tree=nt, tree_mask=mask, **bkw)
            assert np.max(np.abs(got - np.array(want))) < 1e-12, (mode, mask)
        prm = orc.Params(mode=mode, n_tree=nt, **kw)
        allv = orc.attend_group(q[None], L, K, V, L, prm, tree_mask=(1 << nt) - 1)
        assert np.array_equal(allv, orc.attend_group(q[None], L, K, V, L, prm))
    prm = orc.Params("full", n_tree=nt)
    none = orc.attend_group(q[None], L, K, V, L, prm, tree_mask=0)
    assert np.allclose(none, orc.attend_group(q[None], L, K, V, L - nt, orc.Params("full")),
                       atol=1e-14)
    sl = orc.selection_list("full", L, L, prm, tree_mask=0b100)
    assert list(sl["position"]) == list(range(L - nt)) + [L - nt + 2]


def check_nope(orc):
    """rope_theta = 0 is NoPE: the plain softmax-attention definition with no
    rotation, written out here per key (full, window, FOLD)."""
    rng = np.random.default_rng(21)
    d, L = 8, 40
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    c = 1.0 / math.sqrt(d)

    def plain(js, mult):
        s = [mult * c * sum(q[i] * K[j][i] for i in range(d)) for j in js]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        return np.array([sum(e[n] * V[j][i] for n, j in enumerate(js)) / sum(e) for i in range(d)])

    got = orc.attend_group(q[None], 977, K, V, L, orc.Params("full", rope_theta=0.0))[0]
    assert np.allclose(got, plain(range(L), 1.0), atol=1e-12)
    got = orc.attend_group(q[None], 5, K, V, L,
                           orc.Params("window", window=10, n_sink=2, rope_theta=0.0))[0]
    assert np.allclose(got, plain(list(range(2)) + list(range(30, 40)), 1.0), atol=1e-12)
    got = orc.attend_group(q[None], L, K, V, L,
                           orc.Params("fold", window=10, alpha=2.0, far_mix=0.4, rope_theta=0.0))[0]
    want = 0.6 * plain(range(30, 40), 1.0) + 0.4 * plain(range(30), 2.0)
    assert np.allclose(got, want, atol=1e-12)


def check_e4m3(orc):
    import torch
    # every code's value against torch's float8_e4m3fn, and a few closed values
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    for c, v in ((0x00, 0.0), (0x01, 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0), (0x7E, 448.0),
                 (0xFE, -448.0), (0x3C, 1.5)):
        assert orc.e4m3_decode([c])[0] == v, hex(c)
    # encoding against the pure-Python binade rounding: ties, subnormals,
    # saturation, signed zeros, and a log-uniform spread over the range
    rng = np.random.default_rng(21)
    mags = np.exp2(rng.uniform(-12, 9.5, 4000))
    xs = (mags * rng.choice([-1.0, 1.0], 4000)).astype(np.float32)
    special = np.float32([0.0, -0.0, 1.0625, 1.1875, -1.0625, 3 * 2.0 ** -10, 2.0 ** -10,
                          -(2.0 ** -11), 447.0, 448.0, 463.0, 464.0, 470.0, 1e6, -1e6,
                          2.0 ** -6 - 2.0 ** -11, 15.5, 17.0])
    xs = np.concatenate([xs, special])
    enc = orc.e4m3_encode(xs)
    dec = orc.e4m3_decode(enc)
    for x, c, v in zip(xs, enc, dec):
        w = bf_e4m3(float(x))
        assert v == w and math.copysign(1.0, v) == math.copysign(1.0, w), (float(x), int(c), v, w)
    # torch rounds the same way inside the saturation limit
    m = np.abs(xs) < 464
    t = torch.from_numpy(xs[m]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(enc[m], t)
    # the side cache's keys: the float32 quotient's code times the scale
    k = rng.standard_normal(64)
    for s in (0.05, 1.0, 0.003):
        want = [bf_e4m3(float(np.float32(x) / np.float32(s))) * float(np.float32(s)) for x in k]
        assert np.array_equal(orc.side_fp8_keys(k, s), np.array(want)), s


def check_append_rotated_keys(orc):
    """The rotated cache's keys: every (token, head) against the complex form
    at its own position, for a [B, n_new, H_kv, d] append with positions
    [B, n_new] near the ends of the workloads' ranges."""
    rng = np.random.default_rng(31)
    positions = [[0, 4095, 4096], [131075, 1048581, 63]]
    for theta in (1e4, 1e6):
        k = rng.standard_normal((2, 3, 4, 16))
        got = orc.append_rotated_keys(k, np.array(positions), theta)
        assert got.shape == k.shape
        for b in range(2):
            for t in range(3):
                for h in range(4):
                    want = bf_rope(list(k[b, t, h]), positions[b][t], theta)
                    assert np.max(np.abs(got[b, t, h] - np.array(want))) < 1e-9, (theta, b, t, h)
    # one token, one head: the same single rotation
    k1 = rng.standard_normal((1, 1, 1, 8))
    got = orc.append_rotated_keys(k1, np.array([[7]]), 1e4)[0, 0, 0]
    assert np.max(np.abs(got - np.array(bf_rope(list(k1[0, 0, 0]), 7, 1e4)))) < 1e-12


def check_chunked_paths(orc):
    """The oracle walks long selections in chunks of keys.  With chunks far
    smaller than the selection (7, 16 and 64 keys, so that every case crosses
    several chunk boundaries, ragged tail included) the result must still be
    the brute-force one, in every mode."""
    rng = np.random.default_rng(37)
    d = 8
    configs = [
        dict(mode="full", L=37), dict(mode="window", L=50, W=16, n_sink=3),
        dict(mode="window", L=58, W=40, n_sink=9),
        dict(mode="fold", L=45, W=12, alpha=2.0, lam=0.5),
        dict(mode="fold", L=45, W=12, n_sink=4, alpha=2.0, lam=0.5),
        dict(mode="fold", L=52, W=9, n_sink=3, alpha=2.0, lam=0.5, fp8=0.004),
        dict(mode="sharp", L=60, beta=0.4, n_ref=8),
        dict(mode="full", L=200, chunks=(64,)), dict(mode="fold", L=200, W=70, alpha=1.5,
                                                     lam=0.4, chunks=(64,)),
    ]
    for cfg in configs:
        L = cfg["L"]
        K = rng.standard_normal((L, d))
        V = rng.standard_normal((L, d))
        q = rng.standard_normal((2, d))
        p = L + 1
        s8 = cfg.get("fp8", 0.0)
        prm = orc.Params(mode=cfg["mode"], window=cfg.get("W", 0), n_sink=cfg.get("n_sink", 0),
                         alpha=cfg.get("alpha", 1.0), far_mix=cfg.get("lam", 0.0),
                         scale_slope=cfg.get("beta", 0.0), scale_ref=cfg.get("n_ref", 4096),
                         rope_theta=1e4, side_fp8_scale=s8)
        want = [bf_attend_row(cfg["mode"], list(q[r]), p, K.tolist(), V.tolist(), L,
                              W=cfg.get("W", 0), n_sink=cfg.get("n_sink", 0),
                              alpha=cfg.get("alpha", 1.0), lam=cfg.get("lam", 0.0),
                              beta=cfg.get("beta", 0.0), n_ref=cfg.get("n_ref", 4096),
                              far_key=(lambda k: bf_side_fp8(k, s8)) if s8 else None)[0]
                for r in range(2)]
        for chunk in cfg.get("chunks", (7, 16)):
            got = orc.attend_group(q, p, K, V, L, prm, chunk=chunk)
            assert np.max(np.abs(got - np.array(want))) < 1e-12, (cfg, chunk)


ALL_CHECKS = [check_e4m3, check_tree_masks, check_nope, check_rope_complex, check_rope_d2, check_inv_freq, check_selection,
              check_brute_force, check_closed_forms, check_weights_sum,
              check_mode_equivalences, check_fold_shared_position, check_gqa,
              check_page_slot, check_append_rotated_keys, check_chunked_paths]
