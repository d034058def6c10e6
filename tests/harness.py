"""Move a workload to the device and run one step through the C ABI.

The metadata the kernels receive is built by the product's runner-side
builder (``paged_kv_attention_17_gb300.metadata``); the oracle builds its own
independently (``oracle.flatten``).  Inputs come from ``workloads`` only.
"""

from __future__ import annotations

import numpy as np
import torch

import paged_kv_attention_17_gb300 as pkv
from paged_kv_attention_17_gb300 import metadata


def to_torch(x: np.ndarray, dtype: str, device) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def device_inputs(w, device="cuda", requests=None) -> dict:
    reqs = w.requests if requests is None else requests
    meta = metadata.build(reqs, w.block_size)
    e4m3 = getattr(w, "kv_dtype", None) == "e4m3"

    def cache(pool):
        # E4M3 caches travel as their uint8 codes
        return torch.from_numpy(np.ascontiguousarray(pool)).to(device) if e4m3 \
            else to_torch(pool, w.dtype, device)

    d = {
        "w": w,
        "meta": meta,
        "q": to_torch(w.q, w.dtype, device),
        "k_new": to_torch(w.k_new, w.dtype, device),
        "v_new": to_torch(w.v_new, w.dtype, device),
        "k_cache": cache(w.k_pool),
        "v_cache": cache(w.v_pool),
        "qsl": torch.from_numpy(meta["query_start_loc"]).to(device),
        "seq_lens": torch.from_numpy(meta["seq_lens"]).to(device),
        "block_table": torch.from_numpy(meta["block_table"]).to(device),
        "slot_mapping": torch.from_numpy(meta["slot_mapping"]).to(device),
    }
    return d


def run_fused_step(d, num_splits=0, with_lse=True, causal=None, flag=None):
    """pkv_write_attention_varlen of the step.  Returns (out, lse, flag)."""
    w, meta = d["w"], d["meta"]
    dev = d["q"].device
    if flag is None:
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev) if with_lse else None
    if getattr(w, "kv_dtype", None) == "e4m3":
        pkv.pkv_write_attention_varlen_e4m3(
            d["k_new"], d["v_new"], d["slot_mapping"], d["q"], d["k_cache"], d["v_cache"], out,
            d["qsl"], d["seq_lens"], d["block_table"], meta["max_query_len"], meta["max_seq_len"],
            w.softmax_scale, w.k_scale, w.v_scale, causal=w.causal if causal is None else causal,
            num_splits=num_splits, lse_out=lse, error_flag=flag)
        return out, lse, flag
    pkv.pkv_write_attention_varlen(d["k_new"], d["v_new"], d["slot_mapping"], d["q"],
                                   d["k_cache"], d["v_cache"], out, d["qsl"], d["seq_lens"],
                                   d["block_table"], meta["max_query_len"], meta["max_seq_len"],
                                   w.softmax_scale, causal=w.causal if causal is None else causal,
                                   num_splits=num_splits, lse_out=lse, error_flag=flag)
    return out, lse, flag


def run_step(d, num_splits=0, write=True, with_lse=True, causal=None, workspace=None,
             flag=None, out=None):
    """pkv_write of the new tokens, then pkv_attention_varlen (their E4M3 forms
    for a workload with an E4M3 cache).  Returns (out, lse, flag)."""
    w, meta = d["w"], d["meta"]
    dev = d["q"].device
    e4m3 = getattr(w, "kv_dtype", None) == "e4m3"
    if flag is None:
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
    if write:
        if e4m3:
            pkv.pkv_write_e4m3(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                               d["v_cache"], w.k_scale, w.v_scale, error_flag=flag)
        else:
            pkv.pkv_write(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                          error_flag=flag)
    if out is None:
        out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev) if with_lse else None
    if e4m3:
        pkv.pkv_attention_varlen_e4m3(
            d["q"], d["k_cache"], d["v_cache"], out, d["qsl"], d["seq_lens"], d["block_table"],
            meta["max_query_len"], meta["max_seq_len"], w.softmax_scale, w.k_scale, w.v_scale,
            causal=w.causal if causal is None else causal, num_splits=num_splits,
            workspace=workspace, lse_out=lse, error_flag=flag, window=getattr(w, "window", 0))
        return out, lse, flag
    pkv.pkv_attention_varlen(d["q"], d["k_cache"], d["v_cache"], out, d["qsl"], d["seq_lens"],
                             d["block_table"], meta["max_query_len"], meta["max_seq_len"],
                             w.softmax_scale, causal=w.causal if causal is None else causal,
                             num_splits=num_splits, workspace=workspace, lse_out=lse,
                             error_flag=flag, window=getattr(w, "window", 0))
    return out, lse, flag


def errors(out: torch.Tensor, ref: np.ndarray, tokens=None):
    got = out.float().cpu().double().numpy()
    if tokens is not None:
        got, ref = got[tokens], ref[tokens]
    e = np.abs(got - ref)
    return float(e.max()), float(e.mean())
