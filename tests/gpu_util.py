"""Helpers for the GPU parity tests: move a seeded workload to the device,
run the library through its C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_decode_cache_gb300 import pa
from paged_kv_decode_cache_gb300 import workloads as W

# Attention tolerance (bf16 in, fp32 accumulate, bf16 out), element-wise:
# |gpu - ref| <= ATOL + RTOL * |ref|.
ATOL = 2e-3
RTOL = 1e-2
# Log-sum-exp tolerance (fp32 out, no bf16 rounding): |gpu - ref| <= LSE_ATOL + LSE_RTOL * |ref|.
LSE_ATOL = 2e-3
LSE_RTOL = 1e-3


def u16_to_dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().double().numpy()


class Dev:
    """Device copies of a workload's inputs (pools before this step's write)."""

    def __init__(self, w: W.DecodeWorkload):
        self.w = w
        self.q = u16_to_dev_bf16(w.q)
        self.k_cache = u16_to_dev_bf16(w.k_cache)
        self.v_cache = u16_to_dev_bf16(w.v_cache)
        self.block_tables = torch.from_numpy(w.block_tables).cuda()
        self.seq_lens = torch.from_numpy(w.seq_lens).cuda()
        self.k_new = u16_to_dev_bf16(w.k_new)
        self.v_new = u16_to_dev_bf16(w.v_new)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def write(self):
        if self.slot_mapping.numel():
            pa.pa_cache_write(self.k_new, self.v_new, self.slot_mapping, self.k_cache,
                              self.v_cache, status=self.status)

    def decode(self, with_lse=True):
        w = self.w
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda") if with_lse else None
        pa.pa_decode(out, lse, self.q, self.k_cache, self.v_cache, self.block_tables,
                     self.seq_lens, w.scale, status=self.status)
        return out, lse

    def splitkv(self, num_splits=0):
        w = self.w
        P = num_splits or pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_splitkv(out, lse, self.q, self.k_cache, self.v_cache, self.block_tables,
                             self.seq_lens, w.scale, num_splits=P, workspace=ws,
                             status=self.status)
        return out, lse, P

    def step(self, num_splits=0):
        """Fused write + decode (pa_decode_step)."""
        w = self.w
        P = num_splits or pa.pa_auto_num_splits(w.B, w.Hq, w.Hkv, w.D, w.max_blocks, w.block_size)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B, w.Hq, w.D, P)),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_step(out, lse, self.q, self.k_new, self.v_new, self.slot_mapping, self.k_cache,
                          self.v_cache, self.block_tables, self.seq_lens, w.scale, num_splits=P,
                          workspace=ws, status=self.status)
        return out, lse, P

    def mq(self, num_splits=0):
        """Causal multi-query decode (pa_decode_mq) of the workload's q_len queries."""
        w = self.w
        q_len = w.q_len
        q = self.q.view(w.B, q_len, w.Hq, w.D)
        P = num_splits
        if P == 0:
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            P = pa.pa_choose_num_splits_mq(w.B, q_len, w.Hq, w.Hkv, w.D, w.max_blocks,
                                           w.block_size, sms)
        ws = torch.zeros(max(1, pa.pa_splitkv_workspace_bytes(w.B * q_len, w.Hq, w.D, P)),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty((w.B, q_len, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, q_len, w.Hq), dtype=torch.float32, device="cuda")
        pa.pa_decode_mq(out, lse, q, self.k_cache, self.v_cache, self.block_tables, self.seq_lens,
                        w.scale, num_splits=P, workspace=ws, status=self.status)
        return out, lse, P

    def pools(self):
        f = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
        return f(self.k_cache), f(self.v_cache)

    def partial(self, P):
        w = self.w
        po = torch.empty((w.B, w.Hq, P, w.D), dtype=torch.float32, device="cuda")
        pl = torch.empty((w.B, w.Hq, P), dtype=torch.float32, device="cuda")
        pa.pa_decode_partial(po, pl, self.q, self.k_cache, self.v_cache, self.block_tables,
                             self.seq_lens, w.scale, P, status=self.status)
        return po, pl

    def status_value(self) -> int:
        return int(self.status.item())


def oracle_after_write(w: W.DecodeWorkload):
    """Apply this step's write to host copies of the pools; returns (k_cache, v_cache)."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    if w.slot_mapping.size:
        oracle.cache_write(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    return kc, vc


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "", atol: float = ATOL,
                 rtol: float = RTOL):
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
            f"{tuple(idx)}: got {got[tuple(idx)]!r} ref {ref[tuple(idx)]!r}; "
            f"max abs {err.max():.3g}")


def assert_lse_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf pattern differs"
    if fin.any():
        assert_close(got[fin], ref[fin], what + " lse", LSE_ATOL, LSE_RTOL)
