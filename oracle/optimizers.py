"""The eight elementwise optimizer rules FORGE fuses, in float32.

The explainer's Technical Summary §3 ("Generality") lists the rules: AdamW,
NAdam, RAdam, Lion, RMSprop, AdaGrad, SGD and SGD-momentum; §2 ("Exactness")
says the tile-fused step leaves the update logic unchanged, so each rule is the
published method.  The pages give no equations; these are the textbook forms,
with the conventions of torch.optim where a published method leaves a choice:

  AdamW    Loshchilov & Hutter, "Decoupled Weight Decay Regularization" (2019)
  NAdam    Dozat, "Incorporating Nesterov Momentum into Adam" (2016), with the
           momentum-decay schedule mu_t = b1 (1 - 0.5 * 0.96^(0.004 t))
  RAdam    Liu et al., "On the Variance of the Adaptive Learning Rate and
           Beyond" (2020), rectification when rho_t > 5
  Lion     Chen et al., "Symbolic Discovery of Optimization Algorithms" (2023)
  RMSprop  Tieleman & Hinton (2012), lecture 6.5
  AdaGrad  Duchi, Hazan & Singer (2011), diagonal form
  SGD, SGD-momentum (heavy ball, dampening 0)

Weight decay: decoupled (w <- w (1 - lr wd)) for AdamW and Lion; added to the
gradient (g <- g + wd w) for the others, as torch.optim does by default.

Arithmetic: every scalar that depends only on the step and the hyper-parameters
is formed on the host in float64 from the float32 hyper-parameters and rounded
once to float32 (bias corrections enter as reciprocals where that saves a
per-element division: AdamW scales sqrt(v) by 1/sqrt(1 - b2^t), NAdam scales
v by 1/(1 - b2^t)); every per-element operation is one IEEE float32 operation
in the order written in each rule below (no fused multiply-add).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""

import math
from dataclasses import dataclass

import numpy as np

ADAMW, NADAM, RADAM, LION, RMSPROP, ADAGRAD, SGD, SGD_MOMENTUM = range(8)
NAMES = ["adamw", "nadam", "radam", "lion", "rmsprop", "adagrad", "sgd", "sgd_momentum"]

NADAM_MOMENTUM_DECAY = 0.004

# Which state buffers a rule keeps: s1 = first moment / momentum (may be
# negative), s2 = second moment / accumulated square (never negative).
USES_S1 = {ADAMW: True, NADAM: True, RADAM: True, LION: True, RMSPROP: False,
           ADAGRAD: False, SGD: False, SGD_MOMENTUM: True}
USES_S2 = {ADAMW: True, NADAM: True, RADAM: True, LION: False, RMSPROP: True,
           ADAGRAD: True, SGD: False, SGD_MOMENTUM: False}


@dataclass
class Hparams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    alpha: float = 0.99      # RMSprop smoothing constant
    momentum: float = 0.0    # SGD-momentum coefficient

    def f32(self):
        """The hyper-parameters as the float32 values a caller passes."""
        return {k: float(np.float32(getattr(self, k))) for k in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "alpha", "momentum")}


def _f(x: float) -> np.float32:
    return np.float32(x)


def step_scalars(kind: int, hp: Hparams, step: int) -> dict:
    """Per-step scalars (float64 on the host, rounded once to float32)."""
    assert step >= 1
    h = hp.f32()
    lr, b1, b2, eps, wd = h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"]
    t = float(step)
    sc = {"l2": _f(wd)}
    if kind == ADAMW:
        c1 = 1.0 - b1 ** t
        c2 = 1.0 - b2 ** t
        sc.update(decay=_f(1.0 - lr * wd), b1=_f(b1), omb1=_f(1.0 - b1), b2=_f(b2),
                  omb2=_f(1.0 - b2), step_size=_f(lr / c1), inv_sqrt_c2=_f(1.0 / math.sqrt(c2)),
                  eps=_f(eps))
    elif kind == NADAM:
        c2 = 1.0 - b2 ** t
        mu = [b1 * (1.0 - 0.5 * 0.96 ** (i * NADAM_MOMENTUM_DECAY)) for i in range(1, step + 2)]
        mu_t, mu_next = mu[step - 1], mu[step]
        prod_t = 1.0
        for i in range(step):
            prod_t *= mu[i]
        prod_next = prod_t * mu_next
        sc.update(b1=_f(b1), omb1=_f(1.0 - b1), b2=_f(b2), omb2=_f(1.0 - b2), inv_c2=_f(1.0 / c2),
                  eps=_f(eps), coef_g=_f(lr * (1.0 - mu_t) / (1.0 - prod_t)),
                  coef_m=_f(lr * mu_next / (1.0 - prod_next)))
    elif kind == RADAM:
        c1 = 1.0 - b1 ** t
        c2 = 1.0 - b2 ** t
        rho_inf = 2.0 / (1.0 - b2) - 1.0
        rho_t = rho_inf - 2.0 * t * (b2 ** t) / c2
        rect = rho_t > 5.0
        sc.update(b1=_f(b1), omb1=_f(1.0 - b1), b2=_f(b2), omb2=_f(1.0 - b2), eps=_f(eps),
                  rectified=bool(rect), sqrt_c2=_f(math.sqrt(c2)))
        if rect:
            r = math.sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf /
                          ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t))
            sc["step_size"] = _f(lr * r / c1)
        else:
            sc["step_size"] = _f(lr / c1)
    elif kind == LION:
        sc.update(decay=_f(1.0 - lr * wd), lr=_f(lr), b1=_f(b1), omb1=_f(1.0 - b1),
                  b2=_f(b2), omb2=_f(1.0 - b2))
    elif kind == RMSPROP:
        a = h["alpha"]
        sc.update(alpha=_f(a), oma=_f(1.0 - a), lr=_f(lr), eps=_f(eps))
    elif kind == ADAGRAD:
        sc.update(lr=_f(lr), eps=_f(eps))
    elif kind == SGD:
        sc.update(lr=_f(lr))
    elif kind == SGD_MOMENTUM:
        sc.update(lr=_f(lr), mom=_f(h["momentum"]))
    else:
        raise ValueError(f"unknown optimizer kind {kind}")
    return sc


def _sign(c: np.ndarray) -> np.ndarray:
    """sign with sign(0) = 0 and NaN propagated."""
    return np.where(c > 0, np.float32(1), np.where(c < 0, np.float32(-1),
                    np.where(c == 0, np.float32(0), np.float32(np.nan)))).astype(np.float32)


def apply_rule(kind: int, sc: dict, w, g, s1=None, s2=None):
    """One elementwise step.  All arrays float32 of one shape; returns (w, s1, s2).

    w is the float32 value of the weight before the step, g the float32
    gradient, s1/s2 the float32 state values (after dequantisation for INT8
    states).  Returned states are None for buffers the rule does not keep."""
    w = np.asarray(w, dtype=np.float32)
    g = np.asarray(g, dtype=np.float32)
    if kind in (NADAM, RADAM, RMSPROP, ADAGRAD, SGD, SGD_MOMENTUM) and sc["l2"] != 0:
        g = g + sc["l2"] * w
    if kind == ADAMW:
        m = sc["b1"] * s1 + sc["omb1"] * g
        v = sc["b2"] * s2 + sc["omb2"] * (g * g)
        denom = np.sqrt(v) * sc["inv_sqrt_c2"] + sc["eps"]
        w = w * sc["decay"] - sc["step_size"] * (m / denom)
        return w, m, v
    if kind == NADAM:
        m = sc["b1"] * s1 + sc["omb1"] * g
        v = sc["b2"] * s2 + sc["omb2"] * (g * g)
        denom = np.sqrt(v * sc["inv_c2"]) + sc["eps"]
        w = w - sc["coef_g"] * (g / denom)
        w = w - sc["coef_m"] * (m / denom)
        return w, m, v
    if kind == RADAM:
        m = sc["b1"] * s1 + sc["omb1"] * g
        v = sc["b2"] * s2 + sc["omb2"] * (g * g)
        if sc["rectified"]:
            denom = np.sqrt(v) + sc["eps"]
            w = w - sc["step_size"] * ((m * sc["sqrt_c2"]) / denom)
        else:
            w = w - sc["step_size"] * m
        return w, m, v
    if kind == LION:
        c = sc["b1"] * s1 + sc["omb1"] * g
        w = w * sc["decay"] - sc["lr"] * _sign(c)
        m = sc["b2"] * s1 + sc["omb2"] * g
        return w, m, None
    if kind == RMSPROP:
        v = sc["alpha"] * s2 + sc["oma"] * (g * g)
        denom = np.sqrt(v) + sc["eps"]
        w = w - sc["lr"] * (g / denom)
        return w, None, v
    if kind == ADAGRAD:
        v = s2 + g * g
        denom = np.sqrt(v) + sc["eps"]
        w = w - sc["lr"] * (g / denom)
        return w, None, v
    if kind == SGD:
        return w - sc["lr"] * g, None, None
    if kind == SGD_MOMENTUM:
        b = sc["mom"] * s1 + g
        w = w - sc["lr"] * b
        return w, b, None
    raise ValueError(f"unknown optimizer kind {kind}")
