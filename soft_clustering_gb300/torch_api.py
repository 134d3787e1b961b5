"""Torch-owned buffers around the C ABI: what a user holds to run EM.

``GMMState`` allocates the parameters, the workspace and the small outputs
as torch tensors on one device and calls ``gmm_em_step`` /
``gmm_em_step_host`` / ``gmm_assign_topm`` on the current torch stream.  No
arithmetic happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (GMM_BF16, GMM_COV_FULL, GMM_COV_DIAG, GMM_F16, GMM_F32, gmm_assign_topm,
               gmm_default_opts, gmm_em_step, gmm_em_step_host, gmm_ivf_lists,
               gmm_ivf_lists_ws_bytes, gmm_last_device_status, gmm_prepare, gmm_prepared_bytes,
               gmm_workspace_bytes, gmm_workspace_bytes_host)

TORCH_XDTYPE = {torch.float32: GMM_F32, torch.float16: GMM_F16, torch.bfloat16: GMM_BF16}


def cov_shape(cov_type, K, D):
    if cov_type == GMM_COV_FULL:
        return (K, D, D)
    if cov_type == GMM_COV_DIAG:
        return (K, D)
    return (K,)


class GMMState:
    """Parameters + workspace for EM on N x D points with K components."""

    def __init__(self, N, D, K, cov_type, xdtype, device="cuda", chunk_rows=None):
        self.N, self.D, self.K, self.cov_type, self.xdtype = int(N), int(D), int(K), cov_type, xdtype
        self.device = torch.device(device)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.pi = torch.zeros(K, **f32)
        self.mu = torch.zeros(K, D, **f32)
        self.cov = torch.zeros(cov_shape(cov_type, K, D), **f32)
        self.chunk_rows = chunk_rows
        if chunk_rows:
            self.ws_bytes = gmm_workspace_bytes_host(N, D, K, cov_type, xdtype, chunk_rows)
        else:
            self.ws_bytes = gmm_workspace_bytes(N, D, K, cov_type, xdtype)
        if self.ws_bytes == 0:
            raise ValueError("unsupported sizes N=%d D=%d K=%d" % (N, D, K))
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.loglik = torch.zeros(1, dtype=torch.float64, device=self.device)
        self.flags = torch.zeros(K, dtype=torch.int32, device=self.device)
        self.opts = gmm_default_opts()

    def set_params(self, pi, mu, cov):
        for dst, src in ((self.pi, pi), (self.mu, mu), (self.cov, cov)):
            t = torch.as_tensor(np.asarray(src) if not torch.is_tensor(src) else src)
            dst.copy_(t.reshape(dst.shape).to(torch.float32))

    def params_numpy(self):
        return (self.pi.cpu().numpy().astype(np.float64), self.mu.cpu().numpy().astype(np.float64),
                self.cov.cpu().numpy().astype(np.float64))

    def step(self, X, lse=None, stream=None):
        """One EM iteration on device-resident X (N x D); async."""
        return gmm_em_step(X, self.xdtype, self.N, self.D, self.K, self.pi, self.mu, self.cov,
                           self.cov_type, self.ws, self.ws_bytes, self.loglik, lse=lse,
                           flags=self.flags, opts=self.opts, stream=stream)

    def step_host(self, X_host, loglik_host=None, stream=None):
        """One EM iteration with X in (pinned) host memory; synchronous."""
        return gmm_em_step_host(X_host, self.xdtype, self.N, self.D, self.K, self.pi, self.mu,
                                self.cov, self.cov_type, self.ws, self.ws_bytes, self.chunk_rows,
                                self.loglik, loglik_host=loglik_host, flags=self.flags,
                                opts=self.opts, stream=stream)

    def device_status(self, stream=None):
        return gmm_last_device_status(self.ws, stream)

    def fit(self, X, max_iters, tol=0.0, log=None):
        """EM on device-resident X from the current parameters until the
        log-likelihood's relative rise is at most tol, or max_iters steps;
        reads the log-likelihood and the component flags after each step.
        Returns the dict of em_loop.run_em (history, convergence, records)."""
        from . import em_loop
        return em_loop.run_em(lambda: self.step(X), lambda: self.loglik.item(), max_iters, tol,
                              read_flags=lambda: self.flags.cpu().numpy(), log=log)

    def save_checkpoint(self, path, iteration, ll_history=()):
        """Write the parameters (fp32, bit for bit), the iteration count and the
        log-likelihood history; waits for the device work queued so far."""
        from . import checkpoint
        checkpoint.save(path, self.pi.cpu().numpy(), self.mu.cpu().numpy(),
                        self.cov.cpu().numpy(), self.cov_type, iteration, ll_history)

    def load_checkpoint(self, path):
        """Set the parameters from a checkpoint of this shape; returns
        (iteration, ll_history)."""
        from . import checkpoint
        c = checkpoint.load(path)
        if (c["D"], c["K"], c["cov_type"]) != (self.D, self.K, self.cov_type):
            raise ValueError("checkpoint is for D=%d K=%d cov=%d, state is D=%d K=%d cov=%d"
                             % (c["D"], c["K"], c["cov_type"], self.D, self.K, self.cov_type))
        self.set_params(c["pi"], c["mu"], c["cov"])
        return c["iteration"], c["ll_history"]


class Assigner:
    """Prepared parameters + outputs for top-m assignment of N points."""

    def __init__(self, N, D, K, cov_type, xdtype, m, device="cuda"):
        self.N, self.D, self.K, self.cov_type, self.xdtype, self.m = N, D, K, cov_type, xdtype, m
        self.device = torch.device(device)
        self.prepared = torch.empty(gmm_prepared_bytes(D, K, cov_type), dtype=torch.uint8,
                                    device=self.device)
        self.flags = torch.zeros(K, dtype=torch.int32, device=self.device)
        self.ids = torch.empty(N, m, dtype=torch.int32, device=self.device)
        self.gamma = torch.empty(N, m, dtype=torch.float32, device=self.device)
        self.lse = torch.empty(N, dtype=torch.float32, device=self.device)
        self.ws_bytes = gmm_workspace_bytes(N, D, K, cov_type, xdtype)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)

    def prepare(self, pi, mu, cov, opts=None, stream=None):
        f = lambda a, shape: torch.as_tensor(np.asarray(a, dtype=np.float32)).reshape(shape).to(self.device)
        self._p = (f(pi, (self.K,)), f(mu, (self.K, self.D)),
                   f(cov, cov_shape(self.cov_type, self.K, self.D)))
        return gmm_prepare(*self._p, self.D, self.K, self.cov_type, self.prepared, self.flags,
                           opts=opts, stream=stream)

    def assign(self, X, with_lse=True, stream=None):
        return gmm_assign_topm(X, self.xdtype, self.N, self.D, self.K, self.prepared,
                               self.cov_type, self.m, self.ids, self.gamma,
                               self.lse if with_lse else None, self.ws, self.ws_bytes,
                               stream=stream)

    def device_status(self, stream=None):
        return gmm_last_device_status(self.ws, stream)

    def inverted_lists(self, gamma_min, stream=None):
        """IVF lists from the last assignment: (offsets [K+1] int64, point
        indices int32, gamma float32), device tensors; a point joins its best
        component's list and every other of its top-m with gamma >= gamma_min."""
        dev = self.device
        offsets = torch.empty(self.K + 1, dtype=torch.int64, device=dev)
        pts = torch.empty(self.N * self.m, dtype=torch.int32, device=dev)
        gam = torch.empty(self.N * self.m, dtype=torch.float32, device=dev)
        wsb = gmm_ivf_lists_ws_bytes(self.N, self.m, self.K)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        gmm_ivf_lists(self.ids, self.gamma, self.N, self.m, self.K, gamma_min, offsets, pts, gam,
                      ws, wsb, stream=stream)
        return offsets, pts, gam
