"""Helpers for the GPU tests: device copies of numpy inputs and workspace views."""
from __future__ import annotations

import numpy as np

import bit_grouped_expert_gb300 as moe

DEV = "cuda:0"


def dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(DEV)


def host_u16(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def dev_weights(W: dict) -> dict:
    return {n: dev(v) for n, v in W.items()}


class Layer:
    """A plan + workspace for one layer configuration."""

    def __init__(self, H=2048, E=256, k=8, I=512, S=1, max_tokens=256, flags=0):
        import torch
        self.H, self.E, self.k, self.I, self.S = H, E, k, I, S
        self.plan = moe.moe_plan(moe.make_config(H, E, k, I, S, 64), max_tokens, flags)
        self.ws = torch.zeros(moe.moe_workspace_bytes(self.plan), dtype=torch.uint8, device=DEV)
        moe.moe_workspace_init(self.plan, self.ws)

    def view(self, T):
        return moe.moe_route_view(self.plan, self.ws, T)

    def ws_array(self, ptr, shape, dtype):
        import torch
        n = int(np.prod(shape))
        t = moe.workspace_tensor(self.ws, ptr, n, dtype)
        a = t.cpu().numpy().reshape(shape)
        if dtype == torch.int16:
            a = a.view(np.uint16)
        return a

    def routing(self, T):
        import torch
        v = self.view(T)
        E, k = self.E, self.k
        n_tiles = int(self.ws_array(v.n_tiles_d, (1,), torch.int32)[0])
        n_tiles2 = int(self.ws_array(v.n_tiles2_d, (1,), torch.int32)[0]) if v.block_rows2 else 0
        return {
            "keys": self.ws_array(v.keys_d, (T, E), torch.float32),
            "ids": self.ws_array(v.topk_id_d, (T, k), torch.int32),
            "w": self.ws_array(v.topk_w_d, (T, k), torch.float32),
            "counts": self.ws_array(v.counts_d, (E,), torch.int32),
            "offsets": self.ws_array(v.offsets_d, (E + 1,), torch.int32),
            "perm": self.ws_array(v.perm_d, (k * T,), torch.int32),
            "inv": self.ws_array(v.inv_d, (k * T,), torch.int32),
            "n_tiles": n_tiles,
            "blockmap": self.ws_array(v.blockmap_d, (max(n_tiles, 1), 4), torch.int32)[:n_tiles],
            "block_rows": v.block_rows,
            "n_tiles2": n_tiles2,
            "blockmap2": self.ws_array(v.blockmap2_d, (max(n_tiles2, 1), 4), torch.int32)[:n_tiles2],
            "block_rows2": v.block_rows2,
        }

    def status(self, reset=True):
        return moe.moe_device_status(self.plan, self.ws, reset=reset)
