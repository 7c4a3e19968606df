"""Shared helpers for the GPU parity tests: run a workload through the CUDA
library (C ABI via the binding) and through the oracle, and compare.

Tolerances: attention out passes iff |gpu - ref| <= 1e-2 + 1e-2 * |ref| for
every element (bf16 output, fp32 accumulation), lse iff |gpu - ref| <= 1e-3;
the cache write and the page gather must match bit for bit.
"""
import numpy as np
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def dev(t):
    return None if t is None else t.to("cuda").contiguous()


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def assert_attention_close(out, lse, ref_out, ref_lse, what=""):
    got = out.detach().float().cpu().double().numpy()
    err = np.abs(got - ref_out)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    assert not bad.any(), (f"{what}: {int(bad.sum())} out elements outside tolerance; "
                           f"max abs err {err.max():.3e}")
    if lse is not None:
        gl = lse.detach().cpu().double().numpy()
        same_inf = np.isinf(gl) & np.isinf(ref_lse) & (np.sign(gl) == np.sign(ref_lse))
        # equal infinities count as no error (and are not subtracted); a NaN or an
        # unmatched infinity stays an error
        lerr = np.abs(np.where(same_inf, 0.0, gl) - np.where(same_inf, 0.0, ref_lse))
        assert np.all(lerr <= LSE_ATOL), f"{what}: lse max abs err {np.nanmax(lerr):.3e}"
    return float(err.max())


class DecodeRun:
    """Device copies of a DecodeInputs and the buffers one decode step needs."""

    def __init__(self, inp, max_context_len=None):
        self.inp = inp
        self.kc = dev(inp.k_cache)
        self.vc = dev(inp.v_cache)
        self.bt = dev(inp.block_tables)
        self.cl = dev(inp.context_lens)
        self.q = dev(inp.q)
        self.ks = dev(inp.k_scale)
        self.vs = dev(inp.v_scale)
        B, Hq, D = inp.q.shape
        self.max_ctx = max_context_len if max_context_len is not None else inp.max_context_len
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        nbytes = pgqa.decode_workspace_size(B, Hq, inp.num_kv_heads, D, max(self.max_ctx, 1))
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def append(self):
        inp = self.inp
        pgqa.kv_cache_write(dev(inp.step_key), dev(inp.step_value), dev(inp.step_slots), self.kc,
                            self.vc, k_scale=self.ks, v_scale=self.vs, dev_status=self.status)

    def decode(self):
        pgqa.paged_attention_decode(self.out, self.lse, self.q, self.kc, self.vc, self.bt, self.cl,
                                    self.inp.scale, self.max_ctx, k_scale=self.ks,
                                    v_scale=self.vs, workspace=self.ws, dev_status=self.status)

    def status_code(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def oracle_cache_after_append(inp):
    dt = oracle.BF16 if inp.cache_dtype == "bf16" else oracle.E4M3
    return oracle.kv_cache_write(inp.step_key, inp.step_value, inp.step_slots, inp.k_cache,
                                 inp.v_cache, dtype=dt, k_scale=inp.k_scale, v_scale=inp.v_scale)


def oracle_decode(inp, kc=None, vc=None):
    dt = oracle.BF16 if inp.cache_dtype == "bf16" else oracle.E4M3
    kc = inp.k_cache if kc is None else kc
    vc = inp.v_cache if vc is None else vc
    return oracle.paged_decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale,
                               dtype=dt, k_scale=inp.k_scale, v_scale=inp.v_scale)
