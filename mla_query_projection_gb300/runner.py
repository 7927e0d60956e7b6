"""Torch-side plumbing around the C ABI: device buffers for one decode step.

PyTorch only allocates memory and provides the stream; the decode itself is
one ``mla_query_decode`` call into the CUDA library.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 BF16 bit patterns -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class DecodeStep:
    """Device copies of one workload's inputs and outputs plus a handle.

    ``fused_row=True`` packs q_a | kv_c | k_pe into one [B, 2112] row (strided
    inputs, the layout of a fused qkv activation).  ``hidden=True`` makes that
    row on the device instead: every ``decode`` first runs the qkv_a
    down-projection of ``inp["hidden"]`` through ``inp["w_qkv_a"]`` into it."""

    def __init__(self, inp: dict, device="cuda:0", fused_row: bool = False, q_c: bool = True,
                 weights: dict | None = None, hidden: bool = False):
        self.device = torch.device(device)
        dev = self.device
        self.batch = int(inp["q_a"].shape[0])
        self.heads = int(inp["w_uk"].shape[0])
        self.layout = int(inp["layout"])
        wsrc = weights if weights is not None else inp
        if weights is not None and isinstance(weights.get("w_qb"), torch.Tensor):
            self.w_qb, self.w_uk = weights["w_qb"], weights["w_uk"]
            self.gamma_q, self.gamma_kv = weights["gamma_q"], weights["gamma_kv"]
        else:
            self.w_qb = bf16_tensor(wsrc["w_qb"], dev)
            self.w_uk = bf16_tensor(wsrc["w_uk"], dev)
            self.gamma_q = bf16_tensor(wsrc["gamma_q"], dev)
            self.gamma_kv = bf16_tensor(wsrc["gamma_kv"], dev)
        Bn, H = self.batch, self.heads
        self.qkv_a = None
        if hidden:
            self.w_qkv_a = bf16_tensor(inp["w_qkv_a"], dev)
            self.hidden = bf16_tensor(inp["hidden"], dev)
            n, k = self.w_qkv_a.shape
            self.qkv_a = B.mla_qkv_a_create(n, k, self.w_qkv_a)
            fused_row = True
        if fused_row:
            row = np.zeros((Bn, 2112), dtype=np.uint16)
            row[:, :1536] = inp["q_a"]
            row[:, 1536:2048] = inp["kv_c"]
            row[:, 2048:] = inp["k_pe"]
            self.row = bf16_tensor(row, dev)
            self.q_a, self.kv_c, self.k_pe = self.row[:, :1536], self.row[:, 1536:2048], self.row[:, 2048:]
            self.strides = (2112, 2112, 2112)
        else:
            self.q_a = bf16_tensor(inp["q_a"], dev)
            self.kv_c = bf16_tensor(inp["kv_c"], dev)
            self.k_pe = bf16_tensor(inp["k_pe"], dev)
            self.strides = (0, 0, 0)
        self.slots = torch.from_numpy(np.asarray(inp["slots"], dtype=np.int64)).to(dev)
        self.cache = torch.from_numpy(np.ascontiguousarray(inp["cache"])).to(dev)
        self.num_pages, self.page_size = int(self.cache.shape[0]), int(self.cache.shape[1])
        self.k_scale = torch.tensor([inp["k_scale"]], dtype=torch.float32, device=dev)
        self.eps = float(inp["eps"])
        self.q_latent = torch.empty((Bn, H, 512), dtype=torch.bfloat16, device=dev)
        self.q_pe = torch.empty((Bn, H, 64), dtype=torch.bfloat16, device=dev)
        self.q_c = torch.empty((Bn, 1536), dtype=torch.bfloat16, device=dev) if q_c else None
        self.handle = B.mla_query_create(H, self.w_qb, self.w_uk, self.gamma_q, self.gamma_kv, self.eps)

    def decode(self, stream=None, batch=None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        if self.qkv_a is not None:
            rc = B.mla_qkv_a_run(self.qkv_a, self.batch if batch is None else batch, self.hidden, 0,
                                 self.row, 2112, s)
            if rc != B.MLA_OK:
                return rc
        return B.mla_query_decode(
            self.handle, self.batch if batch is None else batch,
            self.q_a, self.strides[0], self.kv_c, self.strides[1], self.k_pe, self.strides[2],
            self.slots, self.cache, self.num_pages, self.page_size, self.layout, self.k_scale,
            self.q_latent, self.q_pe, self.q_c, s,
        )

    def set_path(self, path: int) -> int:
        return B.mla_query_set_path(self.handle, path)

    def error_flags(self) -> int:
        return B.mla_query_get_error(self.handle, torch.cuda.current_stream(self.device))

    def results(self) -> dict:
        torch.cuda.synchronize(self.device)
        out = {
            "q_latent": bf16_bits(self.q_latent),
            "q_pe": bf16_bits(self.q_pe),
            "cache": self.cache.cpu().numpy(),
        }
        if self.q_c is not None:
            out["q_c"] = bf16_bits(self.q_c)
        if self.qkv_a is not None:
            out["qkv_row"] = bf16_bits(self.row)
        return out

    def close(self):
        if self.handle:
            torch.cuda.synchronize(self.device)
            B.mla_query_destroy(self.handle)
            self.handle = None
        if self.qkv_a is not None:
            B.mla_qkv_a_destroy(self.qkv_a)
            self.qkv_a = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
