"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import software_pipelined_tiled_gemm_gb300 as sg
from tests import tolerance

_TD = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_device(A: torch.Tensor, B: torch.Tensor, dtype: str, epilogue=None, stages=4,
               variant="pipelined", c_offset=0, a_offset=0, b_offset=0, fill=0xFFFF, bias=None,
               **tuning):
    """Run C = epi(A.B^T) on cuda:0 through gemm_run (C = epi(A.B) with B of
    shape (K, N) when tuning has b_kn=1).

    *_offset place the operand `offset` elements into a larger allocation (to
    exercise unaligned base addresses); C's surroundings are filled with the
    `fill` pattern and returned so callers can check nothing outside C was
    written.  Returns (C_cpu, plan_info, canary_ok)."""
    M, K = A.shape
    N = B.shape[1] if tuning.get("b_kn") else B.shape[0]
    dev = torch.device("cuda", 0)

    def place(x, off):
        buf = torch.empty(x.numel() + off + 64, dtype=x.dtype, device=dev)
        buf.view(torch.int16).fill_(0x5A5A)
        view = buf[off:off + x.numel()]
        view.copy_(x.reshape(-1).to(dev))
        return buf, view

    _, a = place(A, a_offset)
    _, b = place(B, b_offset)
    bias_ptr = 0
    if bias is not None:
        _, bd = place(bias, 0)
        bias_ptr = bd.data_ptr()
    # C holds the input type, or fp32 for a plan with out_f32.
    c_dtype = torch.float32 if tuning.get("out_f32") else _TD[dtype]
    cbuf = torch.empty(M * N + c_offset + 64, dtype=c_dtype, device=dev)
    cbuf.view(torch.int16).fill_(np.int16(np.uint16(fill).view(np.int16)).item())
    c = cbuf[c_offset:c_offset + M * N]
    plan = sg.Plan(M, N, K, dtype, epilogue, stages, variant, 0, **tuning)
    try:
        stream = torch.cuda.current_stream(dev)
        plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), stream.cuda_stream, bias_ptr)
        torch.cuda.synchronize(dev)
        ds, detail = plan.check()
        assert ds == 0, "device status %d detail %#x" % (ds, detail)
        info = plan.info()
    finally:
        plan.close()
    out = c.view(M, N).cpu()
    around = torch.cat([cbuf[:c_offset], cbuf[c_offset + M * N:]]).view(torch.int16).cpu()
    canary_ok = bool((around.numpy().view(np.uint16) == np.uint16(fill)).all())
    return out, info, canary_ok


def check_full(A, B, dtype, C, epilogue=None, bias=None):
    ref = oracle.gemm_nt(A, B, dtype, epilogue=epilogue, bias=bias)
    got = oracle.decode(bits(C), dtype)
    return tolerance.compare(got, ref, dtype), ref, got


def check_sampled(A, B, dtype, C, rows, cols, epilogue=None, bias=None):
    ref = oracle.gemm_nt_entries(A, B, dtype, rows, cols, epilogue=epilogue, bias=bias)
    got = oracle.decode(bits(C)[rows, cols], dtype)
    return tolerance.compare(got, ref, dtype)


def sample_positions(M, N, count, seed=0, tile_m=128, tile_n=256):
    """Random positions plus every tile-boundary row/column corner and the last
    row/column (partial tiles)."""
    rng = np.random.default_rng(seed)
    r = list(rng.integers(0, M, count))
    c = list(rng.integers(0, N, count))
    edge_r = sorted({0, M - 1} | {x for m in range(tile_m, M, tile_m) for x in (m - 1, m)})
    edge_c = sorted({0, N - 1} | {x for n in range(64, N, 64) for x in (n - 1, n)})
    for i in edge_r[:64]:
        for j in (0, N - 1, N // 2):
            r.append(i)
            c.append(j)
    for j in edge_c[:256]:
        for i in (0, M - 1):
            r.append(i)
            c.append(j)
    return np.array(r, dtype=np.int64), np.array(c, dtype=np.int64)
