"""Device-side set-up for one attention family: buffers, rotary tables, plan, and the
two calls of the path (prep, then attention) through the C ABI.

Only marshalling: torch allocates device memory and supplies the stream; every
computation runs in ``libpg.so``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import pg
from .workloads import FamilyInputs


def bits_to_device(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch bfloat16 tensor on ``device``."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def device_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class FamilyRun:
    """Everything one family's prep + attention needs, resident on the GPU."""

    def __init__(self, fi: FamilyInputs, device="cuda", stream=None, pool_bits=None,
                 rope_rows: int | None = None, ring_window: int | None = None):
        self.fi = fi
        f, b = fi.family, fi.batch
        self.D, self.Hq, self.Hkv = f.head_dim, f.num_qo_heads, f.num_kv_heads
        self.stream = stream
        self.q_raw = bits_to_device(fi.q_raw, device)
        self.k_raw = bits_to_device(fi.k_raw, device)
        self.v_raw = bits_to_device(fi.v_raw, device) if fi.v_raw is not None else None
        self.w_q = bits_to_device(fi.w_q, device)
        self.w_k = bits_to_device(fi.w_k, device)
        if pool_bits is None and fi.pool_fill == "sentinel":
            # a constant fill is cheaper to make on the device than to copy there
            self.pool = torch.full(fi.pool_shape, -1, dtype=torch.int16,
                                   device=device).view(torch.bfloat16)   # 0xFFFF
        else:
            self.pool = bits_to_device(fi.make_pool() if pool_bits is None else pool_bits, device)
        self.pool_desc = pg.pool_descriptor(self.pool)
        self.rope_rows = rope_rows or fi.rope_rows
        half = self.D // 2
        self.rope_cos = torch.empty(self.rope_rows, half, dtype=torch.float32, device=device)
        self.rope_sin = torch.empty(self.rope_rows, half, dtype=torch.float32, device=device)
        pg.check(pg.pg_rope_table(self.rope_cos, self.rope_sin, self.rope_rows, self.D,
                                  f.rope_theta, stream), "pg_rope_table")
        if ring_window is None:
            rc, self.plan = pg.pg_plan_paged_prefill(
                None, b.num_req, b.qo_indptr, b.kv_page_indptr, b.page_ids, b.last_page_len,
                b.start_pos, self.Hq, self.Hkv, self.D, b.page_size, stream)
        else:   # ring slot addressing for window-crossing requests
            rc, self.plan = pg.pg_plan_paged_prefill_ring(
                None, b.num_req, b.qo_indptr, b.kv_page_indptr, b.page_ids, b.start_pos,
                self.Hq, self.Hkv, self.D, b.page_size, ring_window, stream)
        pg.check(rc, "plan")
        T = b.num_tokens
        self.q_out = torch.empty(T, self.Hq, self.D, dtype=torch.bfloat16, device=device)
        self.out = torch.empty(T, self.Hq, self.D, dtype=torch.bfloat16, device=device)
        self.ws_bytes = pg.pg_workspace_bytes(self.plan)
        self.ws = (torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
                   if self.ws_bytes else None)

    # ---- the two calls of the path ----
    def prep_status(self) -> int:
        fi = self.fi
        if self.D == 256:
            return pg.pg_prep_paged_hd256(
                self.plan, self.pool_desc, fi.layer, self.q_raw, self.Hq * 256, self.k_raw,
                self.Hkv * 256, self.v_raw, self.Hkv * 256, self.w_q, self.w_k, fi.eps,
                self.rope_cos, self.rope_sin, self.rope_rows, self.q_out, self.stream)
        return pg.pg_prep_paged_hd512(
            self.plan, self.pool_desc, fi.layer, self.q_raw, self.Hq * 512, self.k_raw,
            self.Hkv * 512, self.w_q, self.w_k, fi.eps, self.rope_cos, self.rope_sin,
            self.rope_rows, self.q_out, self.stream)

    def attn_status(self, q=None, window_left=None) -> int:
        fi = self.fi
        w = fi.family.window_left if window_left is None else window_left
        fn = pg.pg_attn_paged_prefill if self.D == 256 else pg.pg_attn_paged_prefill_hd512
        return fn(self.plan, self.pool_desc, fi.layer, self.q_out if q is None else q, self.out,
                  w, fi.sm_scale, self.ws, self.ws_bytes, self.stream)

    def prep(self):
        pg.check(self.prep_status(), "prep")

    def attn(self, q=None, window_left=None):
        pg.check(self.attn_status(q, window_left), "attention")

    def close(self):
        if self.plan is not None:
            self.plan.close()
            self.plan = None
