"""Device-resident MoE layers built from the seeded synthetic workloads.

Host tensors come from ``workloads`` (the shared seeded generators); every expert is packed
into its bundle by the library's ``moe_pack_bundle`` and copied to the GPU (or kept in pinned
host memory for the expert-slot cache).  Device memory is allocated with torch; all layer
arithmetic runs in libmoe.
"""
from __future__ import annotations

import ctypes as C
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import workloads as wl

from . import (GATING, WDTYPE, moe_bundle_bytes, moe_checksum64, moe_host_bundle, moe_layer,
               moe_layer_forward, moe_layer_workspace_size, moe_pack_bundle,
               moe_pack_bundle_nvfp4)

_POOL = ThreadPoolExecutor(max_workers=max(1, min(16, len(os.sched_getaffinity(0)))))


def pack_expert(cfg: wl.MoEConfig, layer: int, e: int, dst: np.ndarray, shared=False) -> None:
    """Generate expert (layer, e) and pack it into the host byte array ``dst``."""
    w = wl.expert(cfg, layer, e, shared=shared)
    I = cfg.Is if shared else cfg.I
    if cfg.wdtype == "nvfp4":
        moe_pack_bundle_nvfp4(cfg.H, I, w.wg, w.wu, w.wd, w.sg, w.su, w.sd, w.gs, dst)
    else:
        moe_pack_bundle(cfg.H, I, cfg.wdtype, w.wg, w.wu, w.wd, w.sg, w.su, w.sd, dst)


def host_bundles(cfg: wl.MoEConfig, layer: int, experts, pinned=True, shared=False) -> torch.Tensor:
    """[n, bundle_bytes] uint8 host tensor of packed bundles (pinned by default)."""
    I = cfg.Is if shared else cfg.I
    nb = moe_bundle_bytes(cfg.H, I, cfg.wdtype)
    out = torch.empty((len(experts), nb), dtype=torch.uint8, pin_memory=pinned)
    arr = out.numpy()
    list(_POOL.map(lambda ie: pack_expert(cfg, layer, ie[1], arr[ie[0]], shared),
                   enumerate(experts)))
    return out


class DeviceLayer:
    """One MoE layer of ``cfg`` with every routed bundle resident on the GPU (or, with
    ``cached=True``, only the router / shared expert resident: routed bundles come from an
    expert-slot cache)."""

    def __init__(self, cfg: wl.MoEConfig, layer: int = 0, device="cuda", cached=False,
                 bundles_override=None):
        self.cfg, self.layer = cfg, layer
        dev = torch.device(device)
        self.bundle_bytes = moe_bundle_bytes(cfg.H, cfg.I, cfg.wdtype)
        self.w_r = torch.from_numpy(wl.router(cfg, layer)).to(dev)
        b = wl.popularity_bias(cfg, layer)
        self.logit_bias = torch.from_numpy(b).to(dev) if (b is not None and cfg.bias_kind == "logit") else None
        self.sel_bias = torch.from_numpy(b).to(dev) if (b is not None and cfg.bias_kind == "select") else None
        ws = wl.shared_gate_vector(cfg, layer)
        self.w_gate = torch.from_numpy(ws.view(np.int16)).to(dev) if ws is not None else None
        self.shared = None
        if cfg.Is:
            self.shared = host_bundles(cfg, layer, [0], pinned=False, shared=True).to(dev)
        self.routed = None
        if not cached:
            hb = bundles_override if bundles_override is not None else host_bundles(cfg, layer, list(range(cfg.E)))
            self.routed = hb.to(dev)
        self._ptrs = (C.c_void_p * cfg.E)(*[
            (self.routed[e].data_ptr() if self.routed is not None else None) for e in range(cfg.E)])
        d = moe_layer()
        d.H, d.E, d.k, d.I, d.Is = cfg.H, cfg.E, cfg.k, cfg.I, cfg.Is
        d.gating, d.scale, d.wdtype = GATING[cfg.gating], cfg.scale, WDTYPE[cfg.wdtype]
        d.layer_index = layer
        d.shared_gate_sigmoid = 1 if cfg.shared_gate == "sigmoid" else 0
        d.w_r = self.w_r.data_ptr()
        d.logit_bias = self.logit_bias.data_ptr() if self.logit_bias is not None else None
        d.sel_bias = self.sel_bias.data_ptr() if self.sel_bias is not None else None
        d.w_gate = self.w_gate.data_ptr() if self.w_gate is not None else None
        d.shared_bundle = self.shared.data_ptr() if self.shared is not None else None
        d.bundles = None if cached else self._ptrs
        d.norm_eps = wl.STACK_NORM_EPS
        self.desc = d
        self.device = dev

    def workspace(self, T: int) -> torch.Tensor:
        n = moe_layer_workspace_size(self.desc, T)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)

    def forward(self, x: torch.Tensor, ws: torch.Tensor, out=None, forced_ids=None, residual=None,
                cache=None, stream=None, ids_out=None, w_out=None, phase_events=None,
                out_normed=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        st = moe_layer_forward(self.desc, x, T, forced_ids, residual, out, cache, ws, ws.numel(),
                               stream, ids_out=ids_out, w_out=w_out, phase_events=phase_events,
                               out_normed=out_normed)
        return out, st


def host_bundle_table(cfg: wl.MoEConfig, layers: int):
    """Pinned host bundles of every routed expert of ``layers`` layers plus the
    moe_host_bundle table (layer-major) with FNV-1a checksums, for an expert-slot cache."""
    nb = moe_bundle_bytes(cfg.H, cfg.I, cfg.wdtype)
    store = torch.empty((layers * cfg.E, nb), dtype=torch.uint8, pin_memory=True)
    arr = store.numpy()
    jobs = [(l, e) for l in range(layers) for e in range(cfg.E)]
    list(_POOL.map(lambda le: pack_expert(cfg, le[0], le[1], arr[le[0] * cfg.E + le[1]]), jobs))
    sums = list(_POOL.map(lambda i: moe_checksum64(arr[i], nb), range(len(jobs))))
    table = (moe_host_bundle * len(jobs))()
    for i in range(len(jobs)):
        table[i].ptr = store[i].data_ptr()
        table[i].bytes = nb
        table[i].checksum = sums[i]
    return store, table


def to_device_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit array -> int16 device tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """int16/bf16 device tensor -> uint16 bit array on the host."""
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy().view(np.uint16)
