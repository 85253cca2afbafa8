"""Shared helpers of the GPU tests: run one decode step through the C ABI (via the thin
binding) and compute the oracle's answer for the same seeded inputs."""
from __future__ import annotations

import os
from contextlib import contextmanager

import numpy as np
import torch

import oracle
import workloads as W

BF16_ATOL, BF16_RTOL = 2e-3, 1e-2  # bf16 KV: |gpu - ref| <= atol + rtol * |ref|
FP8_ATOL = 3e-2  # E4M3 KV, against the oracle on the dequantised cache
FP32_ATOL, FP32_RTOL = 1e-4, 1e-4  # fp32 output: the kernel's own arithmetic only
# E4M3 pools through the cascade's prefix pass: the softmax weights enter its P V product as
# fp16 (relative rounding 2^-11 each) and their rounded sum is the denominator, so the
# output moves by at most 2^-11 / (1 - 2^-11) * max_t |V_t - out| <= 2^-10 * max |V| of the
# row's values (the codes and q enter exactly); plus the fp32 arithmetic's own error.
FP16_WEIGHT_REL = 2.0 ** -10


def fp16_weight_atol(vmax: float) -> float:
    """Absolute bound for attention with fp16 softmax weights over values |V| <= vmax."""
    return FP16_WEIGHT_REL * vmax + FP32_ATOL


@contextmanager
def split_tokens(n):
    """Force the context partition length (tokens) the library uses."""
    old = os.environ.get("PKV_SPLIT_TOKENS")
    if n is None:
        os.environ.pop("PKV_SPLIT_TOKENS", None)
    else:
        os.environ["PKV_SPLIT_TOKENS"] = str(n)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("PKV_SPLIT_TOKENS", None)
        else:
            os.environ["PKV_SPLIT_TOKENS"] = old


def to_dev(w: W.Workload, dev="cuda"):
    return {
        "q": w.q.to(dev), "k_cache": w.k_cache.to(dev), "v_cache": w.v_cache.to(dev),
        "k_new": w.k_new.to(dev), "v_new": w.v_new.to(dev), "slot_mapping": w.slot_mapping.to(dev),
        "block_tables": w.block_tables.to(dev), "context_lens": w.context_lens.to(dev),
        "scales": None if w.scales is None else w.scales.to(dev),
    }


def gpu_step(w: W.Workload, out_dtype=torch.float32, append=True, t=None):
    """Append (optional) then decode on the GPU; returns (device tensors, out)."""
    import paged_kv_cache_17_gb300 as pkv

    t = t or to_dev(w)
    if append:
        pkv.paged_kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"],
                            scales=t["scales"])
    out = torch.empty(t["q"].shape, dtype=out_dtype, device=t["q"].device)
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                               w.cfg.softmax_scale, out, scales=t["scales"],
                               max_context_len=int(w.context_lens.max()))
    torch.cuda.synchronize()
    return t, out


def oracle_pools_after_append(w: W.Workload, append=True):
    a = w.np()
    kc, vc = a["k_cache"], a["v_cache"]
    if append:
        rc = oracle.append(kc, vc, a["k_new"], a["v_new"], a["slot_mapping"], w.kv_dtype_code, a["scales"])
        assert rc == 0
    return a, kc, vc


def pool_bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu()
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def assert_close(got: np.ndarray, ref: np.ndarray, kind: str, what: str = ""):
    err = np.abs(got - ref)
    if kind == "bf16":
        bad = err > BF16_ATOL + BF16_RTOL * np.abs(ref)
    elif kind == "fp8":
        bad = err > FP8_ATOL
    elif kind == "fp32":
        bad = err > FP32_ATOL + FP32_RTOL * np.abs(ref)
    elif isinstance(kind, float):  # an absolute bound given by the caller
        bad = err > kind
    else:
        raise ValueError(kind)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside the {kind} tolerance; "
                             f"max abs err {err.max():.3e}; first bad {idx.tolist()}")
    return float(err.max()) if err.size else 0.0


def e4m3_vmax(v_codes: np.ndarray, scales: np.ndarray) -> float:
    """Largest |decoded V| in an E4M3 pool [blocks][16][Hkv][D] with V scales scales[1]."""
    import torch

    vals = torch.from_numpy(np.ascontiguousarray(v_codes)).view(torch.float8_e4m3fn).float().abs()
    per_head = vals.amax(dim=(0, 1, 3)).numpy() * np.asarray(scales)[1]
    return float(per_head.max())
