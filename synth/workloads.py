"""Materialise a workload's seeded inputs on the device (torch tensors) or on the host
(fp64 numpy arrays of the stored values).  Only draws numbers; computes nothing of the block."""
from __future__ import annotations

import numpy as np

from . import BF16, F32, LAYER_STRIDE, TID_X, device_fill, host_f64
from . import configs as C


def _torch_dtype(dtype):
    import torch
    return torch.float32 if dtype == F32 else torch.bfloat16


def device_tensor(dtype, shape, seed, tid, mean, std, offset=0, out=None):
    import torch
    t = out if out is not None else torch.empty(tuple(shape), dtype=_torch_dtype(dtype), device="cuda")
    device_fill(t.data_ptr(), dtype, t.numel(), seed, tid, mean, std, offset, torch.cuda.current_stream().cuda_stream)
    return t


def device_layer(wl: C.Workload, layer: int = 0) -> dict:
    return {name: device_tensor(wl.dtype, shape, wl.seed, tid, mean, std)
            for name, tid, shape, mean, std in C.tensor_specs(wl, layer)}


def host_layer(wl: C.Workload, layer: int = 0) -> dict:
    return {name: host_f64(wl.dtype, shape, wl.seed, tid, mean, std)
            for name, tid, shape, mean, std in C.tensor_specs(wl, layer)}


def device_x(wl: C.Workload):
    name, tid, shape, mean, std = C.x_spec(wl)
    return device_tensor(wl.dtype, shape, wl.seed, tid, mean, std)


def host_x(wl: C.Workload, b: int | None = None) -> np.ndarray:
    """All of x [B, S, d], or sequence b only [S, d]."""
    name, tid, shape, mean, std = C.x_spec(wl)
    if b is None:
        return host_f64(wl.dtype, shape, wl.seed, tid, mean, std)
    n = wl.S * wl.d_model
    return host_f64(wl.dtype, (wl.S, wl.d_model), wl.seed, tid, mean, std, offset=b * n)


def cache_tid(which: str, layer: int) -> int:
    from . import TID_KCACHE, TID_VCACHE
    return (TID_KCACHE if which == "k" else TID_VCACHE) + LAYER_STRIDE * layer


def device_caches(wl: C.Workload, cap: int):
    """K and V caches [n_layers, B, cap, n_kv, hd]; every position drawn N(0, 1)."""
    import torch
    shape = (wl.n_layers, wl.B, cap, wl.n_kv, wl.head_dim)
    out = []
    for which in ("k", "v"):
        t = torch.empty(shape, dtype=_torch_dtype(wl.dtype), device="cuda")
        for l in range(wl.n_layers):
            device_tensor(wl.dtype, shape[1:], wl.seed, cache_tid(which, l), 0.0, 1.0, out=t[l])
        out.append(t)
    return out


def host_cache(wl: C.Workload, which: str, layer: int, b: int, cap: int, length: int) -> np.ndarray:
    """Positions 0..length-1 of sequence b's cache in one layer: [length, n_kv, hd]."""
    row = wl.n_kv * wl.head_dim
    return host_f64(wl.dtype, (length, wl.n_kv, wl.head_dim), wl.seed, cache_tid(which, layer), 0.0, 1.0,
                    offset=b * cap * row)


def device_final(wl: C.Workload):
    return [device_tensor(wl.dtype, shape, wl.seed, tid, mean, std) for _, tid, shape, mean, std in C.final_specs(wl)]


def host_final(wl: C.Workload):
    return [host_f64(wl.dtype, shape, wl.seed, tid, mean, std) for _, tid, shape, mean, std in C.final_specs(wl)]


def device_x_emb(wl: C.Workload):
    return device_tensor(wl.dtype, (wl.B, wl.d_model), wl.seed, TID_X, 0.0, 1.0)


def host_x_emb(wl: C.Workload, rows) -> np.ndarray:
    d = wl.d_model
    return np.stack([host_f64(wl.dtype, (d,), wl.seed, TID_X, 0.0, 1.0, offset=int(b) * d) for b in rows])


def device_embed(wl: C.Workload):
    """The [vocab, d_model] token embedding table, rows N(0, 1)."""
    from . import TID_EMBED
    return device_tensor(wl.dtype, (wl.vocab, wl.d_model), wl.seed, TID_EMBED, 0.0, 1.0)


def host_embed_rows(wl: C.Workload, tokens) -> np.ndarray:
    from . import TID_EMBED
    d = wl.d_model
    return np.stack([host_f64(wl.dtype, (d,), wl.seed, TID_EMBED, 0.0, 1.0, offset=int(t) * d) for t in tokens])
