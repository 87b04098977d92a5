"""Pins for the oracle's eight elementwise optimizer rules.

Each rule is checked two ways, neither of which re-types the rule itself:
* against torch.optim run on the CPU in float64 (AdamW, NAdam, RAdam, RMSprop,
  Adagrad, SGD, SGD-momentum), over several steps, including RAdam's
  rectified branch;
* against closed forms that the published methods reduce to at step 1 or in
  special cases (the explainer's Technical Summary §3 "Generality" names the
  rules; Lion has no torch.optim counterpart, so closed forms pin it).
"""

import zlib

import numpy as np
import pytest
import torch

from oracle import optimizers as opt

RTOL = 2e-6


def _f32(x):
    return float(np.float32(x))


def _run_oracle(kind, hp, grads, w0, s1=None, s2=None):
    w = w0.astype(np.float32)
    traj = []
    for t, g in enumerate(grads, start=1):
        sc = opt.step_scalars(kind, hp, t)
        w, s1, s2 = opt.apply_rule(kind, sc, w, g, s1, s2)
        traj.append((w.copy(), None if s1 is None else s1.copy(), None if s2 is None else s2.copy()))
    return traj


def _run_torch(make_opt, grads, w0, state_keys):
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    o = make_opt([p])
    traj = []
    for g in grads:
        p.grad = torch.from_numpy(g.astype(np.float64))
        o.step()
        st = o.state[p]
        traj.append((p.detach().numpy().copy(),) + tuple(
            None if k is None else st[k].numpy().copy() for k in state_keys))
    return traj


def _grads(n_steps, shape=(64, 64), seed=0, scale=1e-2):
    rng = np.random.default_rng(seed)
    return [(rng.standard_normal(shape) * scale).astype(np.float32) for _ in range(n_steps)]


def _close(a, b, rtol=RTOL, atol=1e-12):
    """Relative closeness, with an absolute floor at rtol times the array's scale
    (float32 rounding of values that pass near zero is relative to that scale)."""
    b = np.asarray(b, dtype=np.float64)
    floor = max(atol, rtol * float(np.abs(b).max()))
    np.testing.assert_allclose(a.astype(np.float64), b, rtol=rtol, atol=floor)


CASES = [
    ("adamw", opt.ADAMW, opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
     lambda h: (lambda ps: torch.optim.AdamW(ps, lr=h["lr"], betas=(h["beta1"], h["beta2"]),
                                             eps=h["eps"], weight_decay=h["weight_decay"],
                                             foreach=False)),
     ("exp_avg", "exp_avg_sq")),
    ("nadam", opt.NADAM, opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
     lambda h: (lambda ps: torch.optim.NAdam(ps, lr=h["lr"], betas=(h["beta1"], h["beta2"]),
                                             eps=h["eps"], weight_decay=h["weight_decay"],
                                             momentum_decay=0.004, foreach=False)),
     ("exp_avg", "exp_avg_sq")),
    ("radam", opt.RADAM, opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
     lambda h: (lambda ps: torch.optim.RAdam(ps, lr=h["lr"], betas=(h["beta1"], h["beta2"]),
                                             eps=h["eps"], weight_decay=h["weight_decay"],
                                             foreach=False)),
     ("exp_avg", "exp_avg_sq")),
    ("radam_b2_0.9", opt.RADAM, opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.9, eps=1e-8),
     lambda h: (lambda ps: torch.optim.RAdam(ps, lr=h["lr"], betas=(h["beta1"], h["beta2"]),
                                             eps=h["eps"], foreach=False)),
     ("exp_avg", "exp_avg_sq")),
    ("rmsprop", opt.RMSPROP, opt.Hparams(lr=1e-3, alpha=0.99, eps=1e-8),
     lambda h: (lambda ps: torch.optim.RMSprop(ps, lr=h["lr"], alpha=h["alpha"], eps=h["eps"],
                                               foreach=False)),
     (None, "square_avg")),
    ("adagrad", opt.ADAGRAD, opt.Hparams(lr=1e-2, eps=1e-10),
     lambda h: (lambda ps: torch.optim.Adagrad(ps, lr=h["lr"], eps=h["eps"], foreach=False)),
     (None, "sum")),
    ("sgd", opt.SGD, opt.Hparams(lr=1e-2),
     lambda h: (lambda ps: torch.optim.SGD(ps, lr=h["lr"], foreach=False)),
     (None, None)),
    ("sgd_momentum", opt.SGD_MOMENTUM, opt.Hparams(lr=1e-2, momentum=0.9),
     lambda h: (lambda ps: torch.optim.SGD(ps, lr=h["lr"], momentum=h["momentum"],
                                           foreach=False)),
     ("momentum_buffer", None)),
    ("sgd_momentum_l2", opt.SGD_MOMENTUM, opt.Hparams(lr=1e-2, momentum=0.9, weight_decay=0.05),
     lambda h: (lambda ps: torch.optim.SGD(ps, lr=h["lr"], momentum=h["momentum"],
                                           weight_decay=h["weight_decay"], foreach=False)),
     ("momentum_buffer", None)),
    ("adagrad_l2", opt.ADAGRAD, opt.Hparams(lr=1e-2, eps=1e-10, weight_decay=0.1),
     lambda h: (lambda ps: torch.optim.Adagrad(ps, lr=h["lr"], eps=h["eps"],
                                               weight_decay=h["weight_decay"], foreach=False)),
     (None, "sum")),
]


@pytest.mark.parametrize("name,kind,hp,make,keys", CASES, ids=[c[0] for c in CASES])
def test_rule_matches_torch_optim_float64(name, kind, hp, make, keys):
    steps = 8  # crosses RAdam's rectification threshold (rho_t > 5 from step 6)
    grads = _grads(steps, seed=zlib.crc32(name.encode()))
    rng = np.random.default_rng(1)
    w0 = (rng.standard_normal((64, 64)) * 0.02).astype(np.float32)
    z = np.zeros_like(w0)
    ours = _run_oracle(kind, hp, grads, w0, z if opt.USES_S1[kind] else None,
                       z if opt.USES_S2[kind] else None)
    theirs = _run_torch(make(hp.f32()), grads, w0, keys)
    for t, ((w, s1, s2), ref) in enumerate(zip(ours, theirs), start=1):
        _close(w, ref[0])
        if keys[0] is not None:
            _close(s1, ref[1], atol=1e-15)
        if keys[1] is not None:
            _close(s2, ref[2], atol=1e-18)


def test_radam_branch_switches_at_step_6_for_beta2_0999():
    hp = opt.Hparams(beta2=0.999)
    flags = [opt.step_scalars(opt.RADAM, hp, t)["rectified"] for t in range(1, 9)]
    assert flags == [False] * 5 + [True] * 3


# ---------------------------------------------------------------- closed forms

def _g():
    rng = np.random.default_rng(5)
    g = (rng.standard_normal((32, 32)) * 1e-2).astype(np.float32)
    g[0, 0] = 0.0
    return g


def test_adamw_step1_closed_form():
    """Step 1: m_hat = g, v_hat = g^2, so w' = w (1 - lr wd) - lr g / (|g| + eps)."""
    hp = opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    g, w = _g(), np.full((32, 32), 0.5, dtype=np.float32)
    h = hp.f32()
    w1, m1, v1 = opt.apply_rule(opt.ADAMW, opt.step_scalars(opt.ADAMW, hp, 1), w, g,
                                np.zeros_like(g), np.zeros_like(g))
    g64 = g.astype(np.float64)
    ref = 0.5 * (1 - h["lr"] * h["weight_decay"]) - h["lr"] * g64 / (np.abs(g64) + h["eps"])
    _close(w1, ref, rtol=1e-6)
    _close(m1, (1 - h["beta1"]) * g64, rtol=1e-6)
    _close(v1, (1 - h["beta2"]) * g64 ** 2, rtol=1e-6)


def test_lion_step1_and_special_cases():
    """Lion: step 1 gives w' = w (1 - lr wd) - lr sign(g), m' = (1 - b2) g.
    With b1 = 0 the direction is sign(g_t) at every step; with b2 = 0 the
    momentum is the last gradient, so step 2 uses sign(b1 g1 + (1 - b1) g2)."""
    rng = np.random.default_rng(9)
    g1 = (rng.standard_normal((32, 32)) * 1e-2).astype(np.float32)
    g2 = (rng.standard_normal((32, 32)) * 1e-2).astype(np.float32)
    g1[0, 0] = 0.0
    w = np.full((32, 32), 0.25, dtype=np.float32)
    hp = opt.Hparams(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=0.1)
    h = hp.f32()
    w1, m1, _ = opt.apply_rule(opt.LION, opt.step_scalars(opt.LION, hp, 1), w, g1,
                               np.zeros_like(w), None)
    _close(w1, 0.25 * (1 - h["lr"] * h["weight_decay"]) - h["lr"] * np.sign(g1), rtol=1e-7)
    _close(m1, (1 - h["beta2"]) * g1.astype(np.float64), rtol=1e-6)
    assert w1[0, 0] == np.float32(np.float32(0.25) * np.float32(1 - h["lr"] * h["weight_decay"]))

    hp0 = opt.Hparams(lr=1e-4, beta1=0.0, beta2=0.99)
    sc = opt.step_scalars(opt.LION, hp0, 2)
    w2, _, _ = opt.apply_rule(opt.LION, sc, w, g2, (g1 * np.float32(7)).astype(np.float32), None)
    _close(w2, 0.25 - hp0.f32()["lr"] * np.sign(g2), rtol=1e-7)

    hpb = opt.Hparams(lr=1e-4, beta1=0.9, beta2=0.0)
    _, m_after1, _ = opt.apply_rule(opt.LION, opt.step_scalars(opt.LION, hpb, 1), w, g1,
                                    np.zeros_like(w), None)
    assert np.array_equal(m_after1, g1)
    w2b, _, _ = opt.apply_rule(opt.LION, opt.step_scalars(opt.LION, hpb, 2), w, g2, m_after1, None)
    direction = np.sign(0.9 * g1.astype(np.float64) + 0.1 * g2.astype(np.float64))
    _close(w2b, 0.25 - hpb.f32()["lr"] * direction, rtol=1e-7)


def test_sgd_closed_form_is_exact():
    g, w = _g(), np.full((32, 32), 0.5, dtype=np.float32)
    w1, _, _ = opt.apply_rule(opt.SGD, opt.step_scalars(opt.SGD, opt.Hparams(lr=1.0), 1), w, g)
    assert np.array_equal(w1, (w - g).astype(np.float32))


def test_adagrad_rmsprop_sgdm_step1_closed_forms():
    g, w = _g(), np.full((32, 32), 0.5, dtype=np.float32)
    g64 = g.astype(np.float64)
    z = np.zeros_like(g)
    hp = opt.Hparams(lr=1e-2, eps=1e-10)
    w1, _, v1 = opt.apply_rule(opt.ADAGRAD, opt.step_scalars(opt.ADAGRAD, hp, 1), w, g, None, z)
    _close(w1, 0.5 - hp.f32()["lr"] * g64 / (np.abs(g64) + hp.f32()["eps"]), rtol=1e-6)
    assert np.array_equal(v1, g * g)
    hp = opt.Hparams(lr=1e-3, alpha=0.99, eps=1e-8)
    h = hp.f32()
    w1, _, _ = opt.apply_rule(opt.RMSPROP, opt.step_scalars(opt.RMSPROP, hp, 1), w, g, None, z)
    ref = 0.5 - h["lr"] * g64 / (np.sqrt(1 - h["alpha"]) * np.abs(g64) + h["eps"])
    _close(w1, ref, rtol=1e-6)
    hp = opt.Hparams(lr=1e-2, momentum=0.9)
    w1, b1, _ = opt.apply_rule(opt.SGD_MOMENTUM, opt.step_scalars(opt.SGD_MOMENTUM, hp, 1), w, g, z)
    assert np.array_equal(b1, g)
    g2 = (g * np.float32(-3)).astype(np.float32)
    _, b2, _ = opt.apply_rule(opt.SGD_MOMENTUM, opt.step_scalars(opt.SGD_MOMENTUM, hp, 2), w1, g2, b1)
    _close(b2, 0.9 * g64 - 3 * g64, rtol=1e-6, atol=1e-12)


def test_nadam_and_radam_step1_closed_forms():
    """NAdam step 1: sqrt(v / c2) = |g|, so the update is lr sign(g) times
    (1 + mu2 (1 - b1) / (1 - mu1 mu2)).  RAdam step 1 (unrectified): w - lr g."""
    g, w = _g(), np.full((32, 32), 0.5, dtype=np.float32)
    g64 = g.astype(np.float64)
    z = np.zeros_like(g)
    hp = opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
    h = hp.f32()
    mu1 = h["beta1"] * (1 - 0.5 * 0.96 ** 0.004)
    mu2 = h["beta1"] * (1 - 0.5 * 0.96 ** 0.008)
    w1, _, _ = opt.apply_rule(opt.NADAM, opt.step_scalars(opt.NADAM, hp, 1), w, g, z, z)
    d = np.abs(g64) + h["eps"]
    ref = 0.5 - h["lr"] * g64 / d - h["lr"] * mu2 * (1 - h["beta1"]) / (1 - mu1 * mu2) * g64 / d
    _close(w1, ref, rtol=1e-6)
    w1, _, _ = opt.apply_rule(opt.RADAM, opt.step_scalars(opt.RADAM, hp, 1), w, g, z, z)
    _close(w1, 0.5 - h["lr"] * g64, rtol=1e-6)


def test_decoupled_vs_l2_weight_decay():
    """Zero gradient isolates the decay: AdamW/Lion shrink w by (1 - lr wd);
    SGD with L2 decay moves it by lr * wd * w."""
    w = np.full((4, 64), 0.5, dtype=np.float32)
    z = np.zeros_like(w)
    hp = opt.Hparams(lr=1e-2, weight_decay=0.1)
    w1, _, _ = opt.apply_rule(opt.ADAMW, opt.step_scalars(opt.ADAMW, hp, 1), w, z, z, z)
    assert np.all(w1 == np.float32(0.5) * np.float32(1 - hp.f32()["lr"] * hp.f32()["weight_decay"]))
    w1, _, _ = opt.apply_rule(opt.SGD, opt.step_scalars(opt.SGD, hp, 1), w, z)
    _close(w1, np.full(w.shape, 0.5 - hp.f32()["lr"] * hp.f32()["weight_decay"] * 0.5), rtol=1e-7)
