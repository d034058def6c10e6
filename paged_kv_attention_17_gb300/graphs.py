"""CUDA-graph capture ladder for decode steps.

"Model execution", section "torch.compile and CUDA graphs": a graph records the
GPU work of a step for a fixed token count and replays it with one launch; the
runner captures a ladder of sizes and pads each step up to the next captured
size, and steps above the largest size run without a graph.  "Inside the
engine: kernels, CUDA graphs and the life of a request", section on CUDA
graphs: capture needs fixed shapes and fixed addresses, so the engine pads,
buckets and keeps a static memory pool.

``DecodeGraphRunner`` records, per capture size b (and per host staging slot),
one graph holding a whole decode step on static buffers:

1. the step's packed inputs (q, new K/V, metadata) from pinned host memory
   into the device,
2.-3. ``pkv_write_attention_varlen``: the new tokens' K/V stored by the decode
   kernel itself, then attention (one query token per request),

(``pkv_write_attention_varlen_e4m3`` over an 8-bit E4M3 cache),
4. the output rows back to pinned host memory.

How step 1 and 4 are done (``inputs``):

* ``"stage"`` (default): ``pkv_stage_inputs``, one library kernel, reads the
  pinned staging over the host link in one burst into a device buffer and
  releases the attention kernels at once, so their set-up overlaps the
  transfer; the kernels write the output rows into pinned host memory.
* ``"mapped"``: no copy at all; the attention kernels read the pinned
  staging in place, each CTA paying host-link round trips for its metadata,
  table entries and q rows.
* ``"memcpy"``: copy nodes (copy engine) before and after the kernels; each
  costs a few microseconds and breaks the kernels' dependent-launch chain.

A step of B <= b requests is padded with requests of no token and no context
(query_start_loc repeats B, seq_len 0, slot -1): both calls treat them as
no-ops.  Two staging slots let the host fill one step while the previous one
runs.  All arithmetic stays in the library's kernels; this module only lays
out buffers, records and replays.
"""

from __future__ import annotations

import bisect
import ctypes
from dataclasses import dataclass

import torch

from . import _binding as B

_ALIGN = 256


def capture_ladder(top: int = 512) -> list[int]:
    """Capture sizes: 1, 2, 4, then every 8 up to 248, then every 16 up to
    ``top`` (the ladder the "Model execution" page describes)."""
    sizes = [1, 2, 4]
    sizes += list(range(8, min(top, 248) + 1, 8))
    sizes += list(range(256, top + 1, 16))
    return [s for s in sizes if s <= top]


def bucket(n: int, sizes: list[int]) -> int | None:
    """Smallest captured size >= n, or None when n exceeds the ladder."""
    k = bisect.bisect_left(sizes, n)
    return sizes[k] if k < len(sizes) else None


@dataclass(frozen=True)
class InputLayout:
    """Byte offsets of one size-b step's packed inputs (each field 256-byte
    aligned): q [b, hq, D], k_new and v_new [b, hkv, D] in the cache dtype,
    slot_mapping int64 [b], query_start_loc int32 [b + 1], seq_lens int32 [b],
    block_table int32 [b, max_blocks]."""
    b: int
    offsets: dict
    nbytes: int

    @staticmethod
    def of(b, hq, hkv, d, esize, max_blocks):
        sizes = {"q": b * hq * d * esize, "k_new": b * hkv * d * esize,
                 "v_new": b * hkv * d * esize, "slot_mapping": b * 8,
                 "query_start_loc": (b + 1) * 4, "seq_lens": b * 4,
                 "block_table": b * max_blocks * 4}
        off, offsets = 0, {}
        for name, n in sizes.items():
            offsets[name] = (off, n)
            off = (off + n + _ALIGN - 1) // _ALIGN * _ALIGN
        return InputLayout(b, offsets, off)


def fill_padding(qsl, slots, seq_lens, block_table, n_real: int, b: int) -> None:
    """Decode metadata of a size-b step whose first n_real requests are real:
    request r < n_real has token r; the rest have no token, no context and no
    slot."""
    qsl[: n_real + 1] = torch.arange(n_real + 1, dtype=qsl.dtype)
    qsl[n_real + 1: b + 1] = n_real
    slots[n_real:b] = -1
    seq_lens[n_real:b] = 0
    block_table[n_real:b] = 0


class Step:
    """One staged step: n real requests in captured size b, staging slot
    ``slot``.  Its input views (q, k_new, v_new, slot_mapping, seq_lens,
    block_table: rows 0..n-1 of the pinned staging) are made on first use."""

    __slots__ = ("n", "b", "slot", "_hv")

    def __init__(self, n, b, slot, hv):
        self.n, self.b, self.slot, self._hv = n, b, slot, hv

    def __getattr__(self, name):
        if name in ("q", "k_new", "v_new", "slot_mapping", "seq_lens", "block_table"):
            return self._hv[name][:self.n]
        raise AttributeError(name)


class DecodeGraphRunner:
    """Decode steps (one new token per request) replayed from a ladder of
    captured CUDA graphs over one paged cache.

    k_cache, v_cache: device [num_blocks, 16, hkv, D] (bf16 or fp32, or uint8
    E4M3 codes with ``kv_scales`` = (k_scale, v_scale) and bf16 q / new K/V /
    out), used in place.  max_seq_len bounds every request's context (it sizes the split
    count at capture).  The output of a step stays valid in the returned host
    tensor until its staging slot is reused (``slots`` steps later).
    inputs: "stage" (default), "mapped" or "memcpy" - how the packed inputs
    reach the kernels and the output rows reach the host (module docstring).
    """

    INPUT_PATHS = ("stage", "mapped", "memcpy")

    def __init__(self, k_cache, v_cache, num_q_heads, softmax_scale, max_blocks_per_seq,
                 max_seq_len, max_batch=64, sizes=None, slots=2, inputs="stage",
                 kv_scales=None):
        if inputs not in self.INPUT_PATHS:
            raise ValueError(f"inputs must be one of {self.INPUT_PATHS}")
        self.inputs = inputs
        self.k_cache, self.v_cache = k_cache, v_cache
        self.device = k_cache.device
        self.e4m3 = k_cache.dtype == torch.uint8
        if self.e4m3 and kv_scales is None:
            raise ValueError("an E4M3 (uint8) cache needs kv_scales=(k_scale, v_scale)")
        self.kv_scales = tuple(float(x) for x in kv_scales) if self.e4m3 else None
        self.dtype = torch.bfloat16 if self.e4m3 else k_cache.dtype   # q / new K/V / out
        _, bs, self.hkv, self.d = k_cache.shape
        if bs != 16:
            raise ValueError("block size must be 16")
        self.hq = int(num_q_heads)
        self.scale = float(softmax_scale)
        self.max_blocks = int(max_blocks_per_seq)
        self.max_seq_len = int(max_seq_len)
        ladder = sizes if sizes is not None else capture_ladder(max(int(max_batch), 1))
        self.sizes = sorted({int(s) for s in ladder if 1 <= int(s) <= max_batch})
        if not self.sizes or self.sizes[-1] < max_batch:
            self.sizes.append(int(max_batch))
        esize = torch.empty((), dtype=self.dtype).element_size()
        self.layouts = {b: InputLayout.of(b, self.hq, self.hkv, self.d, esize, self.max_blocks)
                        for b in self.sizes}
        top = self.layouts[self.sizes[-1]].nbytes
        dev = self.device
        self.dev_in = torch.zeros(top, dtype=torch.uint8, device=dev)
        self.host_in = [torch.zeros(top, dtype=torch.uint8).pin_memory() for _ in range(slots)]
        bmax = self.sizes[-1]
        self.out = torch.zeros(bmax, self.hq, self.d, dtype=self.dtype, device=dev)
        self.host_out = [torch.zeros(bmax, self.hq, self.d, dtype=self.dtype).pin_memory()
                         for _ in range(slots)]
        self.flag = torch.zeros(1, dtype=torch.int32, device=dev)
        self.host_flag = [torch.zeros(1, dtype=torch.int32).pin_memory() for _ in range(slots)]
        self.splits = {b: B.pkv_num_splits(b, 1, self.max_seq_len, self.hq, self.hkv, self.d,
                                           dev.index) for b in self.sizes}
        ws = max(B.pkv_workspace_bytes(b, self.hq, self.d, self.splits[b]) for b in self.sizes)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.events = [torch.cuda.Event() for _ in range(slots)]
        self.used = [False] * slots
        self.next_slot = 0
        self.graphs = {}
        self.host_views = {(b, k): self._views(self.host_in[k], b)
                           for b in self.sizes for k in range(slots)}
        self.padded_for = {}                 # (b, slot) -> real-request count its padding is set for
        self._capture()

    # -- views over a packed buffer -------------------------------------------------
    def _views(self, buf, b):
        lay = self.layouts[b]
        shapes = {"q": ((b, self.hq, self.d), self.dtype),
                  "k_new": ((b, self.hkv, self.d), self.dtype),
                  "v_new": ((b, self.hkv, self.d), self.dtype),
                  "slot_mapping": ((b,), torch.int64),
                  "query_start_loc": ((b + 1,), torch.int32),
                  "seq_lens": ((b,), torch.int32),
                  "block_table": ((b, self.max_blocks), torch.int32)}
        out = {}
        for name, (shape, dt) in shapes.items():
            off, n = lay.offsets[name]
            out[name] = buf[off:off + n].view(dt).view(shape)
        return out

    def _record(self, b, slot):
        lay = self.layouts[b]
        if self.inputs == "mapped":
            # the kernels read the pinned staging and write the pinned output
            # rows in place (host memory mapped into the device's address space)
            v = self._views(self.host_in[slot], b)
            out = self.host_out[slot][:b]
        elif self.inputs == "stage":
            B.pkv_stage_inputs(self.dev_in[:lay.nbytes], self.host_in[slot][:lay.nbytes])
            v = self._views(self.dev_in, b)
            out = self.host_out[slot][:b]
        else:
            v = self._views(self.dev_in, b)
            out = self.out[:b]
            self.flag.zero_()
            self.dev_in[:lay.nbytes].copy_(self.host_in[slot][:lay.nbytes], non_blocking=True)
        if self.e4m3:
            ks, vs = self.kv_scales
            B.pkv_write_attention_varlen_e4m3(v["k_new"], v["v_new"], v["slot_mapping"], v["q"],
                                              self.k_cache, self.v_cache, out,
                                              v["query_start_loc"], v["seq_lens"],
                                              v["block_table"], 1, self.max_seq_len, self.scale,
                                              ks, vs, causal=True, num_splits=self.splits[b],
                                              workspace=self.workspace, error_flag=self.flag)
        else:
            # one token per request: the write rides in the decode kernel
            B.pkv_write_attention_varlen(v["k_new"], v["v_new"], v["slot_mapping"], v["q"],
                                         self.k_cache, self.v_cache, out, v["query_start_loc"],
                                         v["seq_lens"], v["block_table"], 1, self.max_seq_len,
                                         self.scale, causal=True, num_splits=self.splits[b],
                                         workspace=self.workspace, error_flag=self.flag)
        if self.inputs == "memcpy":
            self.host_out[slot][:b].copy_(self.out[:b], non_blocking=True)
            self.host_flag[slot].copy_(self.flag, non_blocking=True)

    def _capture(self):
        stream = torch.cuda.Stream(device=self.device)
        stream.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(stream):
            for b in self.sizes:
                for slot in range(len(self.host_in)):
                    hv = self._views(self.host_in[slot], b)
                    fill_padding(hv["query_start_loc"], hv["slot_mapping"], hv["seq_lens"],
                                 hv["block_table"], 0, b)         # all padding: a no-op step
                    self._record(b, slot)                        # eager once (kernel set-up)
                    stream.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        self._record(b, slot)
                    self.graphs[(b, slot)] = g
        torch.cuda.current_stream(self.device).wait_stream(stream)
        torch.cuda.synchronize(self.device)

    # -- stepping -------------------------------------------------------------------
    def begin(self, n: int) -> Step:
        """Stage a step of n decode requests: returns host views of its
        inputs (rows 0..n-1 to fill; padding rows are already set)."""
        b = bucket(n, self.sizes)
        if b is None or n < 1:
            raise ValueError(f"step of {n} requests is outside the captured ladder "
                             f"(1..{self.sizes[-1]})")
        slot = self.next_slot
        self.next_slot = (slot + 1) % len(self.host_in)
        if self.used[slot]:
            self.events[slot].synchronize()          # its previous replay is done with it
        hv = self.host_views[(b, slot)]
        if self.padded_for.get((b, slot)) != n:
            fill_padding(hv["query_start_loc"], hv["slot_mapping"], hv["seq_lens"],
                         hv["block_table"], n, b)
            self.padded_for[(b, slot)] = n
        return Step(n, b, slot, hv)

    def pack(self, n, q, k_new, v_new, slot_mapping, seq_lens, block_table):
        # (contiguous CPU tensor: ``stage`` copies its bytes as they are)
        """The packed host bytes of a step of n requests (padding included),
        for ``stage``: build once, stage every time the same inputs recur."""
        b = bucket(n, self.sizes)
        if b is None:
            raise ValueError(f"step of {n} requests is outside the captured ladder")
        buf = torch.zeros(self.layouts[b].nbytes, dtype=torch.uint8)
        v = self._views(buf, b)
        v["q"][:n].copy_(q)
        v["k_new"][:n].copy_(k_new)
        v["v_new"][:n].copy_(v_new)
        v["slot_mapping"][:n].copy_(slot_mapping)
        v["seq_lens"][:n].copy_(seq_lens)
        v["block_table"][:n, :block_table.shape[1]].copy_(block_table)
        fill_padding(v["query_start_loc"], v["slot_mapping"], v["seq_lens"], v["block_table"],
                     n, b)
        return buf

    def stage(self, step: Step, packed: torch.Tensor) -> None:
        """Copy packed bytes (from ``pack``, same n) into the step's staging
        (a plain host memory copy)."""
        ctypes.memmove(self.host_in[step.slot].data_ptr(), packed.data_ptr(), packed.numel())
        self.padded_for[(step.b, step.slot)] = step.n

    def launch(self, step: Step) -> None:
        """Replay the step's graph on the current stream (asynchronous)."""
        self.graphs[(step.b, step.slot)].replay()
        self.events[step.slot].record()
        self.used[step.slot] = True

    def result(self, step: Step):
        """Wait for the step; returns (output rows [n, hq, D] in pinned host
        memory, device error flag value).  Unless inputs is "memcpy" the flag is
        not reset per step: it holds every error since the runner was made."""
        self.events[step.slot].synchronize()
        if self.inputs != "memcpy":
            return self.host_out[step.slot][:step.n], int(self.flag.item())
        return self.host_out[step.slot][:step.n], int(self.host_flag[step.slot][0])
