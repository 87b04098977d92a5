"""Column-parallel tensor-parallel FORGE step (Technical Summary §2 "Distributed
Training Compatibility": a weight shard's gradient is complete on its own
device, so the fused step stays exact under tensor parallelism).

CPU: two gloo ranks run the partition and the partial-dX all-reduce of
optimizer_tcgen05_dw_gb300.tp with the shard compute supplied by the test (the
oracle on the rank's rows); the gathered shards must equal the unsharded
oracle step bit for bit and dX must lie within the rounding of the partials.
GPU: P = 2 shards stepped one after the other through the C ABI
(forge_linear_bwd_step_shard) must equal the unsharded library step bit for
bit in W and the states; the partial dX tiles summed must match its dX within
the same rounding bound."""

import ctypes
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import rounding
from optimizer_tcgen05_dw_gb300 import api, inputs, tp
from optimizer_tcgen05_dw_gb300.build import build

HP = dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_shard_step(X, dY, W, opt_name, hp, step, seed, row_offset, s1=None, s2=None,
                       s1_scale=None, s2_scale=None, dX=None):
    """The shard's FORGE step computed by the oracle on CPU tensors (bf16 W,
    fp32 moments), in place, with the rows' indices in the whole matrix."""
    Xb, dYb, Wb = inputs.bf16_to_bits(X), inputs.bf16_to_bits(dY), inputs.bf16_to_bits(W)
    if dX is not None:
        dX.copy_(inputs.bits_to_bf16(ls.input_gradient(dYb, Wb)))
    g = ls.weight_gradient(Xb, dYb)
    out = ls.update_block(opt.NAMES.index(opt_name), opt.Hparams(**hp), step, seed, g, Wb, "bf16",
                          s1.numpy(), s2.numpy(), None, None, "fp32", row_offset, 0, W.shape[1])
    W.copy_(inputs.bits_to_bf16(out["W"]))
    s1.copy_(torch.from_numpy(out["s1"]))
    s2.copy_(torch.from_numpy(out["s2"]))


def _full_problem(T, N, K, seed):
    X = inputs.normal((T, K), 1.0, seed)
    dY = inputs.normal((T, N), 1e-3, seed + 1)
    W = inputs.normal((N, K), 0.02, seed + 2)
    m = inputs.normal((N, K), 1e-4, seed + 3, torch.float32)
    v = inputs.abs_normal((N, K), 1e-6, seed + 4)
    return X, dY, W, m, v


def _dx_bound_ok(dx_tp_bits, partial_bits, exact_bits):
    """|dX_tp - exact| <= half an ulp of each partial (their own rounding) +
    half an ulp of the result (the final rounding); exact = correctly rounded
    bf16 of the exact sum, so one more half ulp of it."""
    f = lambda b: rounding.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    ulp = lambda x: 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126))) - 7)  # noqa: E731
    got, ex = f(dx_tp_bits), f(exact_bits)
    bound = 0.5 * ulp(got) + 0.5 * ulp(ex) + sum(0.5 * ulp(f(p)) for p in partial_bits)
    return np.all(np.abs(got - ex) <= bound * (1 + 1e-12))


def _rank_main(rank, world, port, T, N, K, seed, step, result_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, dY, W, m, v = _full_problem(T, N, K, seed)
        row0, rows = tp.shard_rows(N, world, rank)
        Wr, mr, vr = tp.shard(W, world, rank), tp.shard(m, world, rank), tp.shard(v, world, rank)
        dYr = tp.shard(dY, world, rank, dim=1)
        dX = torch.empty((T, K), dtype=torch.bfloat16)
        got_row0 = tp.column_parallel_bwd_step(X, dYr, Wr, "adamw", HP, step, seed, mr, vr, dX=dX,
                                               world=world, rank=rank, step_fn=_oracle_shard_step)
        assert got_row0 == row0
        # this rank's own partial (from its pre-update rows), for the rounding bound
        partial = ls.input_gradient(inputs.bf16_to_bits(dYr), inputs.bf16_to_bits(tp.shard(W, world, rank)))
        gathered = {}
        for name, t in (("W", Wr.view(torch.int16).to(torch.int32)), ("m", mr), ("v", vr)):
            parts = [torch.empty_like(t) for _ in range(world)]
            dist.all_gather(parts, t)
            gathered[name] = torch.cat(parts, 0)
        pt = torch.from_numpy(partial.astype(np.int32))
        parts = [torch.empty_like(pt) for _ in range(world)]
        dist.all_gather(parts, pt)
        if rank == 0:
            result_q.put({"W": gathered["W"].numpy().astype(np.uint16), "m": gathered["m"].numpy(),
                          "v": gathered["v"].numpy(), "dX": inputs.bf16_to_bits(dX),
                          "partials": [p.numpy().astype(np.uint16) for p in parts]})
    finally:
        dist.destroy_process_group()


def test_shard_rows_partition():
    assert tp.shard_rows(1024, 2, 1) == (512, 512)
    assert tp.shard_rows(14336, 8, 7, align=64) == (12544, 1792)
    with pytest.raises(ValueError):
        tp.shard_rows(1000, 3, 0)
    with pytest.raises(ValueError):
        tp.shard_rows(1024, 2, 2)
    # every row owned exactly once
    owned = sorted(r for k in range(4) for r in range(*(lambda a, b: (a, a + b))(*tp.shard_rows(256, 4, k))))
    assert owned == list(range(256))


def test_two_gloo_ranks_equal_the_unsharded_oracle_step():
    T, N, K, seed, step = 48, 64, 32, 5, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, T, N, K, seed, step, q)) for r in range(2)]
    for p in procs:
        p.start()
    import queue
    res = None
    for _ in range(600):  # up to 5 minutes, but stop as soon as a rank has failed
        try:
            res = q.get(timeout=0.5)
            break
        except queue.Empty:
            if any(p.exitcode not in (None, 0) for p in procs):
                break
    for p in procs:
        p.join(timeout=120)
        if p.exitcode is None:
            p.kill()
        assert p.exitcode == 0
    assert res is not None
    X, dY, W, m, v = _full_problem(T, N, K, seed)
    ref = ls.linear_bwd_step(inputs.bf16_to_bits(X), inputs.bf16_to_bits(dY),
                             {"W": inputs.bf16_to_bits(W), "w_dtype": "bf16", "s_dtype": "fp32",
                              "s1": m.numpy(), "s2": v.numpy()},
                             opt.ADAMW, opt.Hparams(**HP), step, seed, want_dx=True)
    assert np.array_equal(res["W"], ref["W"])
    assert np.array_equal(res["m"], ref["s1"])
    assert np.array_equal(res["v"], ref["s2"])
    assert _dx_bound_ok(res["dX"], res["partials"], ref["dX"])


def test_dx_bound_catches_a_wrong_partial():
    """The dX check fails when one shard's partial is dropped from the sum."""
    T, N, K = 16, 32, 16
    X, dY, W, m, v = _full_problem(T, N, K, 11)
    exact = ls.input_gradient(inputs.bf16_to_bits(dY), inputs.bf16_to_bits(W))
    p0 = ls.input_gradient(inputs.bf16_to_bits(tp.shard(dY, 2, 0, 1)), inputs.bf16_to_bits(tp.shard(W, 2, 0)))
    p1 = ls.input_gradient(inputs.bf16_to_bits(tp.shard(dY, 2, 1, 1)), inputs.bf16_to_bits(tp.shard(W, 2, 1)))
    f = lambda b: rounding.bf16_bits_to_f32(b)  # noqa: E731
    summed = rounding.bf16_bits_rne((f(p0) + f(p1)).astype(np.float32))
    assert _dx_bound_ok(summed, [p0, p1], exact)
    assert not _dx_bound_ok(p0, [p0, p1], exact)


def test_shard_entry_point_rejects_a_negative_offset():
    build()
    L = api.lib()
    fake = 1 << 20
    lin = api.ForgeLinear(64, 128, 256, fake, fake, None)
    st = api.ForgeState(fake, api.W_BF16_SR, api.STATE_FP32, fake, fake, None, None)
    hp = api.hparams(lr=1e-3)
    r = L.forge_linear_bwd_step_shard(ctypes.byref(lin), ctypes.byref(st), 0, ctypes.byref(hp), 1, 0, -128, None)
    assert r == 1 and b"row_offset" in L.forge_last_error_message()


@pytest.mark.gpu
@pytest.mark.parametrize("s_dtype,T,N,K", [("fp32", 512, 1024, 768), ("int8", 320, 512, 384),
                                           ("fp32", 200, 256, 136)])
def test_two_shards_in_sequence_equal_the_unsharded_step(cuda_device, s_dtype, T, N, K):
    """P = 2 row shards stepped one after the other on one GPU (each through
    forge_linear_bwd_step_shard, dX into its own partial) against one
    unsharded forge_linear_bwd_step: W and the states bit-equal, and the
    partials summed within their rounding of the unsharded dX's exact value."""
    build()
    api.forge_set_step_fusion(True)
    dev = cuda_device
    seed = 23
    X = inputs.normal((T, K), 1.0, seed, torch.bfloat16, dev)
    dY = inputs.normal((T, N), 1e-3, seed + 1, torch.bfloat16, dev)
    W0 = inputs.normal((N, K), 0.02, seed + 2, torch.bfloat16, dev)
    hp = dict(HP)

    def state():
        if s_dtype == "int8":
            m = torch.empty((N, K), dtype=torch.int8, device=dev)
            v = torch.empty((N, K), dtype=torch.uint8, device=dev)
            ms = torch.empty((N, K // 64), device=dev)
            vs = torch.empty((N, K // 64), device=dev)
            api.forge_quantize_state(inputs.normal((N, K), 1e-4, seed + 3, torch.float32, dev), m, ms, True)
            api.forge_quantize_state(inputs.abs_normal((N, K), 1e-6, seed + 4, torch.float32, dev), v, vs, False)
            return [W0.clone(), m, v, ms, vs]
        return [W0.clone(), torch.zeros((N, K), device=dev), torch.zeros((N, K), device=dev), None, None]

    full = state()
    dX_full = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    shards = [[None if t is None else tp.shard(t, 2, r) for t in state()] for r in range(2)]
    partials = [torch.empty((T, K), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    for step in (1, 2):
        W_pre = full[0].clone()
        api.forge_linear_bwd_step(X, dY, full[0], "adamw", hp, step, seed, *full[1:], dX=dX_full)
        for r in range(2):
            tp.column_parallel_bwd_step(X, tp.shard(dY, 2, r, dim=1), shards[r][0], "adamw", hp, step, seed,
                                        *shards[r][1:], dX=partials[r], world=2, rank=r)
        api.forge_get_device_status()
        for i, name in enumerate(("W", "s1", "s2", "s1_scale", "s2_scale")):
            if full[i] is None:
                continue
            cat = torch.cat([shards[0][i], shards[1][i]], 0)
            assert torch.equal(cat, full[i]), f"step {step}: {name}"
    # dX of the last step: each partial is dY_r W_r from the shard's pre-update
    # rows, within one bf16 ulp plus the FP32 summation bound of its exact
    # value; the partials summed in FP32 and rounded once must lie within
    # those bounds plus half an ulp of the exact whole dX
    f = lambda t: rounding.bf16_bits_to_f32(inputs.bf16_to_bits(t)).astype(np.float64)  # noqa: E731
    ulp = lambda x: 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126))) - 7)  # noqa: E731
    dY64, W64 = f(dY), f(W_pre)
    bound = np.zeros((T, K))
    exact = np.zeros((T, K))
    for r in range(2):
        row0, rows = tp.shard_rows(N, 2, r)
        d, w = dY64[:, row0:row0 + rows], W64[row0:row0 + rows]
        ex_r = d @ w
        exact += ex_r
        bound += ulp(ex_r) + 2.0 ** -24 * (np.ceil(rows / 16.0) * 3.0 * np.sqrt((d * d) @ (w * w)) +
                                           4.0 * np.abs(ex_r))
        assert np.all(np.abs(f(partials[r]) - ex_r) <= ulp(ex_r) + bound), f"partial {r}"
    summed = (f(partials[0]) + f(partials[1])).astype(np.float32)
    got = rounding.bf16_bits_to_f32(rounding.bf16_bits_rne(summed)).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound + 0.5 * ulp(got))
