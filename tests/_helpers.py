"""Shared test utilities: input construction, oracle/GPU adapters, tolerance checks.

Tolerances:
* exact FP32 inputs (integer-grid data, oracle-supplied gradients): bit-exact;
* realistic data, one step from a common state: an *interval oracle*.  The GPU
  sums the T token products on the tensor cores in FP32 (T/16 accumulator
  updates), the oracle in float64; the FORGE explainer's §2 "Exactness" names
  the summation order as the only difference.  The oracle is evaluated at
  g - d, g and g + d, where d bounds the tensor-core summation error per
  element, and every GPU output must lie in the hull of the three results
  widened by the base tolerance: FP32 values 1e-7 + 1e-5 |x|, BF16 weights one
  ULP (stochastic rounding turns a sub-ULP difference into a whole ULP), INT8
  codes one step.  In addition >= 99.9 % of BF16 weights must be within 1 ULP
  of the central result;
* free-running multi-step BF16 trajectories: >= 99.9 % within 1 ULP, all
  within 2 ULP measured at the weight scale;
* dX (bf16): |gpu - exact| <= 1 bf16 ULP of the exact value plus the same
  summation bound over the N reduction terms.
"""

import numpy as np
import torch

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import quant, rounding
from optimizer_tcgen05_dw_gb300 import inputs

NAME_TO_KIND = {n: i for i, n in enumerate(opt.NAMES)}
SUM_ERR = 2.0 ** -20  # relative FP32 summation bound used for exclusions


def oracle_hparams(hp: dict) -> opt.Hparams:
    return opt.Hparams(**hp)


def to_bits(t):
    return inputs.bf16_to_bits(t)


class Problem:
    """One layer: inputs per step, initial state, and both trajectories."""

    def __init__(self, T, N, K, w_dtype, s_dtype, opt_name, hp, seed=1, grid=False,
                 x_std=1.0, dy_std=1e-3, w_std=0.02, m_std=1e-4, v_std=1e-6, steps=2,
                 device_inputs=False, qblock=64):
        self.T, self.N, self.K = T, N, K
        self.qblock = qblock  # INT8 states: elements per absmax block
        self.w_dtype, self.s_dtype, self.opt, self.hp = w_dtype, s_dtype, opt_name, hp
        self.kind = NAME_TO_KIND[opt_name]
        self.seed = seed
        self.steps = steps
        gen_dev = "cuda" if device_inputs else "cpu"
        self.X, self.dY = [], []
        for s in range(steps):
            if grid:
                X = inputs.integer_grid((T, K), -4, 4, 0, inputs.layer_seed(seed, 0, s, 1), device=gen_dev)
                dY = inputs.integer_grid((T, N), -4, 4, -12, inputs.layer_seed(seed, 0, s, 2), device=gen_dev)
            else:
                X = inputs.normal((T, K), x_std, inputs.layer_seed(seed, 0, s, 1), device=gen_dev)
                dY = inputs.normal((T, N), dy_std, inputs.layer_seed(seed, 0, s, 2), device=gen_dev)
            self.X.append(X)
            self.dY.append(dY)
        W = inputs.normal((N, K), w_std, inputs.layer_seed(seed, 0, 0, 3), torch.float32)
        m = inputs.normal((N, K), m_std, inputs.layer_seed(seed, 0, 0, 4), torch.float32)
        v = inputs.abs_normal((N, K), v_std, inputs.layer_seed(seed, 0, 0, 5))
        st = {"w_dtype": w_dtype, "s_dtype": s_dtype,
              "W": W.numpy() if w_dtype == "fp32" else rounding.bf16_bits_rne(W.numpy())}
        if opt.USES_S1[self.kind]:
            if s_dtype == "int8":
                st["s1"], st["s1_scale"] = quant.quantize_blocks(m.numpy(), signed=True, block=qblock)
            elif s_dtype == "bf16":
                st["s1"] = rounding.bf16_bits_rne(m.numpy())
            else:
                st["s1"] = m.numpy()
        if opt.USES_S2[self.kind]:
            if s_dtype == "int8":
                st["s2"], st["s2_scale"] = quant.quantize_blocks(v.numpy(), signed=False, block=qblock)
            elif s_dtype == "bf16":
                st["s2"] = rounding.bf16_bits_rne(v.numpy())
            else:
                st["s2"] = v.numpy()
        self.state0 = st

    # ---- GPU side
    def gpu_state(self):
        return self.upload(self.state0)

    def run_gpu(self, fused=True, want_dx=False, state=None):
        from optimizer_tcgen05_dw_gb300 import api
        g = self.gpu_state() if state is None else state
        dxs = []
        for s in range(self.steps):
            X, dY = self.X[s].cuda(), self.dY[s].cuda()
            dX = torch.empty((self.T, self.K), dtype=torch.bfloat16, device="cuda") if want_dx else None
            if fused:
                api.forge_linear_bwd_step(X, dY, g["W"], self.opt, self.hp, s + 1, self.seed,
                                          g.get("s1"), g.get("s2"), g.get("s1_scale"),
                                          g.get("s2_scale"), dX=dX)
            else:
                if want_dx:
                    api.forge_linear_dgrad(dY, g["W"], dX)
                dW = torch.empty((self.N, self.K), dtype=torch.float32, device="cuda")
                api.forge_unfused_wgrad(X, dY, dW)
                api.forge_unfused_opt_step(dW, g["W"], self.opt, self.hp, s + 1, self.seed,
                                           g.get("s1"), g.get("s2"), g.get("s1_scale"),
                                           g.get("s2_scale"))
            dxs.append(dX)
        api.forge_get_device_status()
        torch.cuda.synchronize()
        return g, dxs

    def upload(self, st):
        dev = "cuda"
        W = (torch.from_numpy(np.ascontiguousarray(st["W"])) if self.w_dtype == "fp32"
             else inputs.bits_to_bf16(st["W"])).to(dev)
        out = {"W": W}
        for k in ("s1", "s2", "s1_scale", "s2_scale"):
            if st.get(k) is not None:
                if self.s_dtype == "bf16" and k in ("s1", "s2"):
                    out[k] = inputs.bits_to_bf16(st[k]).to(dev)
                else:
                    out[k] = torch.from_numpy(np.ascontiguousarray(st[k])).to(dev)
        return out

    def per_step_from_common_state(self):
        """Every step starts both sides from the oracle's (central) state; the
        GPU result of that step must lie in the oracle's interval."""
        from optimizer_tcgen05_dw_gb300 import api
        st = {k: v for k, v in self.state0.items()}
        hp = oracle_hparams(self.hp)
        for s in range(self.steps):
            g_dev = self.upload(st)
            Xb, dYb = to_bits(self.X[s]), to_bits(self.dY[s])
            api.forge_linear_bwd_step(self.X[s].cuda(), self.dY[s].cuda(), g_dev["W"], self.opt,
                                      self.hp, s + 1, self.seed, g_dev.get("s1"), g_dev.get("s2"),
                                      g_dev.get("s1_scale"), g_dev.get("s2_scale"))
            api.forge_get_device_status()
            g = ls.weight_gradient(Xb, dYb)
            iv = oracle_interval(self.kind, hp, s + 1, self.seed, g, st, self.w_dtype,
                                 self.s_dtype, 0, 0, self.K, grad_error_bound(Xb, dYb), self.qblock)
            assert_in_interval(g_dev, iv, self.w_dtype, self.s_dtype, f"step {s + 1}", self.qblock)
            st = dict(st)
            st.update({k: iv[0][0][k] for k in ("W", "s1", "s2", "s1_scale", "s2_scale")})
        return st

    # ---- oracle side
    def run_oracle(self, want_dx=False):
        st = {k: (None if v is None else (v.copy() if isinstance(v, np.ndarray) else v))
              for k, v in self.state0.items()}
        hp = oracle_hparams(self.hp)
        dxs, sens = [], np.zeros((self.N, self.K), dtype=bool)
        self.w_before = []  # the weights each step starts from (dX reads them)
        for s in range(self.steps):
            Xb, dYb = to_bits(self.X[s]), to_bits(self.dY[s])
            self.w_before.append(st["W"])
            sens |= self.sensitive(Xb, dYb, st)
            if self.qblock == 64:
                out = ls.linear_bwd_step(Xb, dYb, st, self.kind, hp, s + 1, self.seed, want_dx=want_dx)
            else:  # the same step with another INT8 block width
                out = {}
                if want_dx:
                    out["dX"] = ls.input_gradient(dYb, ls.weights_for_dx(st["W"], self.w_dtype))
                out.update(ls.update_block(self.kind, hp, s + 1, self.seed, ls.weight_gradient(Xb, dYb),
                                           st["W"], self.w_dtype, st.get("s1"), st.get("s2"),
                                           st.get("s1_scale"), st.get("s2_scale"), self.s_dtype,
                                           0, 0, self.K, block=self.qblock))
            dxs.append(out.get("dX"))
            st.update({k: out[k] for k in ("W", "s1", "s2", "s1_scale", "s2_scale")})
        return st, dxs, sens

    def sensitive(self, Xb, dYb, st):
        """Elements whose update flips within the FP32 summation error of g."""
        X = rounding.bf16_bits_to_f32(Xb).astype(np.float64)
        dY = rounding.bf16_bits_to_f32(dYb).astype(np.float64)
        g = dY.T @ X
        bound = SUM_ERR * (np.abs(dY).T @ np.abs(X)) + 1e-30
        mask = np.abs(g) <= bound
        if self.kind == opt.LION and st.get("s1") is not None:
            if self.s_dtype == "fp32":
                m = st["s1"]
            elif self.s_dtype == "bf16":
                m = rounding.bf16_bits_to_f32(st["s1"])
            else:
                m = quant.dequantize_blocks(st["s1"], st["s1_scale"], True, block=self.qblock)
            b1 = np.float32(self.hp.get("beta1", 0.9))
            c = b1 * m.astype(np.float64) + (1 - b1) * g
            mask |= np.abs(c) <= bound
        return mask


def gpu_np(t):
    if t.dtype == torch.bfloat16:
        return to_bits(t)
    return t.detach().cpu().numpy()


def assert_bitexact(gpu, ref, what):
    a, b = gpu_np(gpu), np.asarray(ref)
    if a.dtype == np.float32:
        same = (a == b) | (np.isnan(a) & np.isnan(b))
    else:
        same = a == b
    bad = np.argwhere(~same)
    assert bad.size == 0, f"{what}: {len(bad)} of {a.size} differ; first at {bad[:3].tolist()}: " \
        f"gpu={a[tuple(bad[0])]} ref={b[tuple(bad[0])]}"


def assert_fp32_close(gpu, ref, what, exclude=None, rtol=1e-5, atol=1e-7):
    a = gpu_np(gpu).astype(np.float64)
    b = np.asarray(ref, dtype=np.float64)
    ok = np.abs(a - b) <= atol + rtol * np.abs(b)
    if exclude is not None:
        ok |= exclude
    bad = np.argwhere(~ok)
    assert bad.size == 0, f"{what}: {len(bad)} of {a.size} outside tolerance; first " \
        f"{bad[:3].tolist()}: gpu={a[tuple(bad[0])]} ref={b[tuple(bad[0])]}"


def _ulp_at(mag):
    """bf16 ULP size at magnitude mag (normal range)."""
    mag = np.maximum(np.asarray(mag, dtype=np.float64), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(mag)) - 7)


def assert_bf16_close(gpu, ref_bits, what, exclude=None, free_running=False):
    """<= 1 ULP on >= 99.9 % of elements, <= 2 ULP on all non-excluded ones.

    One step from a common state (free_running=False): ULPs are the bf16 grid
    steps between the two values.  A free-running multi-step trajectory
    (free_running=True): once one stochastic rounding decision differs, the
    trajectories stay one ULP apart in absolute terms, and a weight that later
    passes near zero turns that gap into many ULPs of a smaller binade, so the
    ULP is taken at the larger of the two values and the RMS weight."""
    a_bits = gpu_np(gpu)
    d = rounding.bf16_ulp_distance(a_bits, ref_bits)
    frac1 = float((d <= 1).mean())
    assert frac1 >= 0.999, f"{what}: only {frac1:.5f} of elements within 1 ULP"
    if free_running:
        a = rounding.bf16_bits_to_f32(a_bits).astype(np.float64)
        b = rounding.bf16_bits_to_f32(ref_bits).astype(np.float64)
        rms = float(np.sqrt(np.mean(b * b)))
        d = np.abs(a - b) / _ulp_at(np.maximum(np.maximum(np.abs(a), np.abs(b)), rms))
    far = d > 2
    if exclude is not None:
        far &= ~exclude
    bad = np.argwhere(far)
    assert bad.size == 0, f"{what}: {len(bad)} elements beyond 2 ULP; first {bad[:3].tolist()} " \
        f"({d[tuple(bad[0])]} ULP)"


def block_mask(mask, block=64):
    """Element mask -> the same mask widened to whole blocks of `block` elements."""
    N, K = mask.shape
    b = mask.reshape(N, K // block, block).any(axis=2)
    return np.repeat(b, block, axis=1), b


def assert_int8_close(gpu_codes, gpu_scale, ref_codes, ref_scale, what, exclude=None, block=64):
    a = gpu_np(gpu_codes).astype(np.int64)
    b = np.asarray(ref_codes).astype(np.int64)
    ex_el, ex_blk = (None, None) if exclude is None else block_mask(exclude, block)
    diff = np.abs(a - b) > 1
    if ex_el is not None:
        diff &= ~ex_el
    bad = np.argwhere(diff)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ by more than one step"
    assert_fp32_close(gpu_scale, ref_scale, what + " scale", exclude=ex_blk)


def assert_dx_close(gpu_dx, dYb, Wb, what):
    dY = rounding.bf16_bits_to_f32(dYb).astype(np.float64)
    W = rounding.bf16_bits_to_f32(Wb).astype(np.float64)
    exact = dY @ W
    n_red = W.shape[0]
    bound = 2.0 ** -24 * (np.ceil(n_red / 16.0) * 3.0 * np.sqrt((dY * dY) @ (W * W)) +
                          4.0 * np.abs(exact))
    a = rounding.bf16_bits_to_f32(gpu_np(gpu_dx)).astype(np.float64)
    ulp = np.maximum(np.abs(exact), 1e-38)
    ulp = 2.0 ** (np.floor(np.log2(ulp)) - 7)
    ok = np.abs(a - exact) <= ulp + bound
    bad = np.argwhere(~ok)
    assert bad.size == 0, f"{what}: {len(bad)} of {a.size} outside; first {bad[:3].tolist()}: " \
        f"gpu={a[tuple(bad[0])]} exact={exact[tuple(bad[0])]}"


# ---------------------------------------------------------------- interval oracle

def grad_error_bound(Xb, dYb):
    """Per-element bound on |g_gpu - g_exact| for g = sum_t dY[t,n] X[t,k]:
    ceil(T/16) FP32 accumulator updates, each off by at most one rounding of a
    partial sum no larger than 3x the random-walk scale sqrt(sum_t (dY X)^2),
    plus the final rounding of g."""
    X = rounding.bf16_bits_to_f32(Xb).astype(np.float64)
    dY = rounding.bf16_bits_to_f32(dYb).astype(np.float64)
    T = X.shape[0]
    rw = np.sqrt((dY * dY).T @ (X * X))
    g = dY.T @ X
    return 2.0 ** -24 * (np.ceil(T / 16.0) * 3.0 * rw + 4.0 * np.abs(g)) + 1e-30


def oracle_interval(kind, hp, step, seed, g, st_block, w_dtype, s_dtype, n0, k0, K, delta, block=64):
    """Oracle results for one block of W at four gradients: g, g - delta,
    g + delta, and the point of [g - delta, g + delta] nearest zero (where a
    squared gradient is smallest).  Returns (outs, fp32_states): outs[i] is
    the oracle's update_block result, fp32_states[i] the float32 moments the
    rule produced before any INT8 quantisation."""
    g64 = g.astype(np.float64)
    near0 = np.clip(0.0, g64 - delta, g64 + delta)
    points = [g64, g64 - delta, g64 + delta, near0]
    outs, fp32 = [], []
    wf = (rounding.bf16_bits_to_f32(st_block["W"]) if w_dtype == "bf16"
          else np.asarray(st_block["W"], dtype=np.float32))
    uses1, uses2 = opt.USES_S1[kind], opt.USES_S2[kind]
    if s_dtype == "int8":
        m0 = quant.dequantize_blocks(st_block["s1"], st_block["s1_scale"], True, block) if uses1 else None
        v0 = quant.dequantize_blocks(st_block["s2"], st_block["s2_scale"], False, block) if uses2 else None
    elif s_dtype == "bf16":
        m0 = rounding.bf16_bits_to_f32(st_block["s1"]) if uses1 else None
        v0 = rounding.bf16_bits_to_f32(st_block["s2"]) if uses2 else None
    else:
        m0, v0 = st_block.get("s1"), st_block.get("s2")
    sc = opt.step_scalars(kind, hp, step)
    for pt in points:
        gg = pt.astype(np.float32)
        outs.append(ls.update_block(kind, hp, step, seed, gg, st_block["W"], w_dtype,
                                    st_block.get("s1"), st_block.get("s2"),
                                    st_block.get("s1_scale"), st_block.get("s2_scale"),
                                    s_dtype, n0, k0, K, block=block))
        _, m1, v1 = opt.apply_rule(kind, sc, wf, gg, m0, v0)
        fp32.append({"s1": m1, "s2": v1})
    return outs, fp32


def _hull(vals):
    v = np.stack([np.asarray(x, dtype=np.float64) for x in vals])
    return v.min(axis=0), v.max(axis=0)


def _fp32_in(g, lo, hi):
    return (g >= lo - (1e-7 + 1e-5 * np.abs(lo))) & (g <= hi + (1e-7 + 1e-5 * np.abs(hi)))


def assert_in_interval(gpu_state, interval, w_dtype, s_dtype, what, block=64):
    """GPU outputs inside the hull of the oracle's interval results, widened
    by the base tolerance (see module docstring)."""
    outs, fp32 = interval
    central = outs[0]
    a = gpu_np(gpu_state["W"])
    if w_dtype == "bf16":
        d = rounding.bf16_ulp_distance(a, central["W"])
        frac1 = float((d <= 1).mean())
        assert frac1 >= 0.999, f"{what} W: only {frac1:.5f} within 1 ULP of the central result"
        lo, hi = _hull([rounding.bf16_bits_to_f32(o["W"]) for o in outs])
        af = rounding.bf16_bits_to_f32(a).astype(np.float64)
        ok = (af >= lo - _ulp_at(np.abs(lo))) & (af <= hi + _ulp_at(np.abs(hi)))
    else:
        lo, hi = _hull([o["W"] for o in outs])
        af = a.astype(np.float64)
        ok = _fp32_in(af, lo, hi)
    bad = np.argwhere(~ok)
    assert bad.size == 0, f"{what} W: {len(bad)} of {a.size} outside the interval; first " \
        f"{bad[:3].tolist()}: gpu={af[tuple(bad[0])]} interval=[{lo[tuple(bad[0])]}, {hi[tuple(bad[0])]}]"
    for key, signed in (("s1", True), ("s2", False)):
        if central.get(key) is None:
            continue
        g = gpu_np(gpu_state[key])
        lo, hi = _hull([f[key] for f in fp32])          # float32 moment, per element
        if s_dtype == "bf16":  # nearest-even bf16 of a value in the hull: within 1 ULP of it
            gf = rounding.bf16_bits_to_f32(g).astype(np.float64)
            ok = (gf >= lo - _ulp_at(np.abs(lo))) & (gf <= hi + _ulp_at(np.abs(hi)))
            bad = np.argwhere(~ok)
            assert bad.size == 0, f"{what} {key}: {len(bad)} of {g.size} outside the interval; " \
                f"first {bad[:3].tolist()}: gpu={gf[tuple(bad[0])]} [{lo[tuple(bad[0])]}, {hi[tuple(bad[0])]}]"
            continue
        if s_dtype != "int8":
            gf = g.astype(np.float64)
            ok = _fp32_in(gf, lo, hi)
            bad = np.argwhere(~ok)
            assert bad.size == 0, f"{what} {key}: {len(bad)} of {g.size} outside the interval; " \
                f"first {bad[:3].tolist()}: gpu={gf[tuple(bad[0])]} [{lo[tuple(bad[0])]}, {hi[tuple(bad[0])]}]"
            continue
        # INT8: the block absmax lies between the largest per-element lower
        # magnitude and the largest upper magnitude; each dequantised code lies
        # within half a quantisation step of its element's interval.
        R, C = lo.shape
        lo_b, hi_b = lo.reshape(R, C // block, block), hi.reshape(R, C // block, block)
        min_mag = np.where((lo_b > 0) | (hi_b < 0), np.minimum(np.abs(lo_b), np.abs(hi_b)), 0.0)
        max_mag = np.maximum(np.abs(lo_b), np.abs(hi_b))
        a_lo, a_hi = min_mag.max(axis=2), max_mag.max(axis=2)
        gs = gpu_np(gpu_state[key + "_scale"]).astype(np.float64)
        ok = (gs >= a_lo * (1 - 1e-5)) & (gs <= a_hi * (1 + 1e-5) + 1e-30)
        bad = np.argwhere(~ok)
        assert bad.size == 0, f"{what} {key} scale: {len(bad)} outside the interval; first " \
            f"{bad[:3].tolist()}: gpu={gs[tuple(bad[0])]} [{a_lo[tuple(bad[0])]}, {a_hi[tuple(bad[0])]}]"
        step = gs / (127.0 if signed else 255.0)
        deq = g.astype(np.float64).reshape(R, C // block, block) * step[..., None]
        half = 0.5 * step[..., None] * (1 + 1e-5) + 1e-30
        ok = (deq >= lo_b - half - 1e-5 * np.abs(lo_b)) & (deq <= hi_b + half + 1e-5 * np.abs(hi_b))
        bad = np.argwhere(~ok)
        assert bad.size == 0, f"{what} {key}: {len(bad)} codes further than half a step " \
            f"from the interval; first {bad[:3].tolist()}"
