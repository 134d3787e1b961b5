"""Helpers for the GPU tests: inputs from datagen, runs through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

import datagen
import oracle
import soft_clustering_gb300 as G
from soft_clustering_gb300.torch_api import Assigner, GMMState

TORCH_STORE = {datagen.F32: torch.float32, datagen.F16: torch.float16, datagen.BF16: torch.bfloat16}


def to_device(bits: np.ndarray, xdtype: int) -> torch.Tensor:
    """Stored bits (host) -> device tensor of the stored dtype, same bytes."""
    if xdtype == datagen.F32:
        t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_STORE[xdtype])
    return t.cuda()


def make_state(wl, chunk_rows=None):
    return GMMState(wl.N, wl.D, wl.K, wl.cov_type, wl.dtype, chunk_rows=chunk_rows)


def set_opts(state: GMMState, opts):
    for k, v in (opts or {}).items():
        setattr(state.opts, k, v)


def gpu_step(state: GMMState, Xd, params, want_lse=False, opts=None):
    set_opts(state, opts)
    state.set_params(*params)
    lse = torch.empty(state.N, dtype=torch.float32, device="cuda") if want_lse else None
    state.step(Xd, lse=lse)
    st = state.device_status()
    pi, mu, cov = state.params_numpy()
    out = dict(status=st, pi=pi, mu=mu, cov=cov, ll=float(state.loglik.item()),
               flags=state.flags.cpu().numpy())
    if want_lse:
        out["lse"] = lse.cpu().numpy().astype(np.float64)
    return out


def f32(params):
    return tuple(np.asarray(p, dtype=np.float32) for p in params)


def oracle_step(bits, xdtype, params, cov_type, opts=None, want_lse=False):
    pi, mu, cov = (np.asarray(p, dtype=np.float64) for p in params)
    return oracle.em_step(bits, pi, mu, cov, cov_type, xdtype=xdtype, opts=opts, want_lse=want_lse)
