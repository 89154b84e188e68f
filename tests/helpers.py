"""Shared test plumbing: seeded inputs on both sides, and the parity bar.

Inputs come only from synth/ (bit-identical on host and device).  Expected values
come only from oracle/.  Nothing here computes any part of the block.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import synth
from synth import configs as C

# Parity bar (the stated tolerances):
#   fp32: max |err| <= 1e-4 * max |ref|
#   bf16: for every row, max_i |err| <= 2e-2 * RMS(ref row)
FP32_TOL = 1e-4
BF16_TOL = 2e-2


def assert_parity(got: np.ndarray, ref: np.ndarray, dtype: int, what: str = "", tol: float | None = None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if dtype == synth.F32:
        t = FP32_TOL if tol is None else tol
        err = np.max(np.abs(got - ref)) if got.size else 0.0
        bound = t * max(np.max(np.abs(ref)) if ref.size else 0.0, 1e-30)
        assert err <= bound, f"{what}: max|err| {err:.3e} > {bound:.3e}"
        return err / max(bound / t, 1e-30)
    t = BF16_TOL if tol is None else tol
    g2 = got.reshape(-1, got.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    rms = np.sqrt(np.mean(r2 * r2, axis=-1))
    err = np.max(np.abs(g2 - r2), axis=-1)
    rel = err / np.maximum(rms, 1e-30)
    worst = int(np.argmax(rel)) if rel.size else 0
    assert np.all(err <= t * rms), f"{what}: row {worst} max|err|/RMS = {rel[worst]:.3e} > {t}"
    return float(rel.max()) if rel.size else 0.0


def assert_sublayer_parity(got_y, ref_y, x, dtype: int, what: str = ""):
    """The sublayer contributions y - x against the oracle's, per row: within 2e-2 of the
    contribution's RMS plus the rounding of the stored output (half a bf16 ulp of y, <= 2^-8 |y|;
    f32 outputs get 2^-23 |y|)."""
    got_y, ref_y, x = (np.asarray(a, dtype=np.float64) for a in (got_y, ref_y, x))
    dg = (got_y - x).reshape(-1, x.shape[-1])
    dr = (ref_y - x).reshape(-1, x.shape[-1])
    ry = np.abs(ref_y.reshape(-1, x.shape[-1]))
    rms = np.sqrt(np.mean(dr * dr, axis=-1, keepdims=True))
    ulp = 2.0 ** -8 if dtype != synth.F32 else 2.0 ** -23
    bound = BF16_TOL * rms + ulp * ry + 1e-30
    ratio = np.abs(dg - dr) / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert np.all(ratio <= 1.0), f"{what}: row {worst[0]} col {worst[1]} err/bound = {ratio[worst]:.3f}"


# ----------------------------------------------------------------------- device side
def torch_dtype(dtype: int):
    import torch
    return torch.float32 if dtype == synth.F32 else torch.bfloat16


def dev_tensor(dtype: int, shape, seed: int, tid: int, mean: float, std: float, offset: int = 0):
    import torch
    shape = (shape,) if isinstance(shape, int) else tuple(shape)
    t = torch.empty(shape, dtype=torch_dtype(dtype), device="cuda")
    synth.device_fill(t.data_ptr(), dtype, t.numel(), seed, tid, mean, std, offset,
                      torch.cuda.current_stream().cuda_stream)
    return t


def to_f64(t) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def host_tensor(dtype: int, shape, seed: int, tid: int, mean: float, std: float, offset: int = 0):
    return synth.host_f64(dtype, tuple(shape), seed, tid, mean, std, offset)


# ----------------------------------------------------------------------- a layer's weights
def layer_weights(wl: C.Workload, layer: int = 0, host: bool = True, device: bool = True):
    """(device dict, oracle BlockWeights) for one layer of workload wl."""
    dev, hst = {}, {}
    for name, tid, shape, mean, std in C.tensor_specs(wl, layer):
        if device:
            dev[name] = dev_tensor(wl.dtype, shape, wl.seed, tid, mean, std)
        if host:
            hst[name] = host_tensor(wl.dtype, shape, wl.seed, tid, mean, std)
    return dev, (O.BlockWeights(**hst) if host else None)


def oracle_dims(wl: C.Workload, **over) -> O.Dims:
    d = dict(B=wl.B, S=wl.S, d_model=wl.d_model, n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim,
             d_ff=wl.d_ff, theta_base=wl.theta_base, eps=wl.eps)
    d.update(over)
    return O.Dims(**d)


def sample_rows(S: int, n: int = 64) -> np.ndarray:
    """n rows spread over [0, S), always including 0 and S-1."""
    if S <= n:
        return np.arange(S)
    r = np.unique(np.concatenate([[0, S - 1], np.linspace(0, S - 1, n - 2).round().astype(int)]))
    return r
